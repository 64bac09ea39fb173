"""The probes used by tests/test_gpu_kap_bound.py (tensor-core logits, hardware exp2) compile for sm_103a (no GPU
needed), so that a GPU run of that test fails only on its numbers."""
import ctypes

from tests import test_gpu_kap_bound as kb


def test_logit_probe_compiles_and_exports():
    lib = ctypes.CDLL(kb.build_probe())
    assert hasattr(lib, "umma_logits_probe")


def test_ex2_probe_compiles_and_exports():
    lib = ctypes.CDLL(kb.build_ex2_probe())
    assert hasattr(lib, "ex2_error_probe")

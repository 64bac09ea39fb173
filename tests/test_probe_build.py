"""The tensor-core logit probe used by tests/test_gpu_kap_bound.py compiles for sm_103a (no GPU
needed), so that a GPU run of that test fails only on its numbers."""
import ctypes

from tests import test_gpu_kap_bound as kb


def test_logit_probe_compiles_and_exports():
    lib = ctypes.CDLL(kb.build_probe())
    assert hasattr(lib, "umma_logits_probe")

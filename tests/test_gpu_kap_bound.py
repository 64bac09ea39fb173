"""The accumulation-error bound behind the KAP's exact selections, measured on the tensor cores.

The KAP ranks blocks on fp32 logits from tcgen05 (CoSA Sec. 4.2, Eqs. (9)-(13)) and certifies every
decision with |fp32 logit - exact| <= kappa * scale * ||q|| * ||k||, kappa = 2^-18 (the model: bf16
products are exact in fp32; groups of at most 16 products aligned to the group's largest term and
truncated, then added to a truncating fp32 accumulator, lose at most 48 * 2^-24 of sum |q_i k_i|).
If the hardware summed less accurately than that, a near-tie could be certified the wrong way round
and a mask would differ silently.  This test runs the tensor-core path the KAP logits kernel uses
(tests/probes/umma_logits_probe.cu: same TMA boxes, swizzle, descriptors and instruction) on
adversarial rows and compares every fp32 logit with the exact float64 dot product:

    worst |err| / (||q|| ||k||)       <= kappa / 2    (half the certified bound: margin for luck)
    worst |err| / sum_i |q_i k_i|     <= 48 * 2^-24   (the accumulation model itself)

The block scores (Eqs. (9)-(11)) take each exp(bm - M_r) with the hardware base-2 exponential
(ex2.approx.ftz.f32) and bound its relative error by EX2_REL; a second probe
(tests/probes/ex2_error_probe.cu) measures that instruction's largest relative error over every fp32
input whose result is a normal number (2^-126 .. 2^0.05), against the float64 exp2:

    worst relative error of ex2.approx <= EX2_REL / 2
"""
import ctypes
import os
import shutil
import subprocess

import numpy as np
import pytest
import torch

import synth
from tests import gpu_helpers as gh

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PROBE_SRC = os.path.join(ROOT, "tests", "probes", "umma_logits_probe.cu")
PROBE_LIB = os.path.join(ROOT, "tests", "probes", "_build", "umma_logits_probe.so")
KAPPA = 2.0 ** -18
MODEL = 48 * 2.0 ** -24
EX2_REL = 2.0 ** -21              # kEx2Rel in kap.cu
EX2_SRC = os.path.join(ROOT, "tests", "probes", "ex2_error_probe.cu")
EX2_LIB = os.path.join(ROOT, "tests", "probes", "_build", "ex2_error_probe.so")
ROWS = 384                        # 3 x 3 tiles of 128 x 128 per case


def build_probe(src: str = PROBE_SRC, lib: str = PROBE_LIB) -> str:
    srcs = [src, os.path.join(ROOT, "block_sparse_long_gb300", "csrc", "ptx.cuh")]
    if os.path.exists(lib) and all(os.path.getmtime(s) <= os.path.getmtime(lib) for s in srcs):
        return lib
    os.makedirs(os.path.dirname(lib), exist_ok=True)
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    cmd = [nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O2", "-std=c++17", "-Xcompiler", "-fPIC",
           "-shared", "-cudart", "static", "-I", os.path.join(ROOT, "block_sparse_long_gb300", "csrc"),
           src, "-o", lib + ".tmp"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stdout + r.stderr
    os.replace(lib + ".tmp", lib)
    return lib


def build_ex2_probe() -> str:
    return build_probe(EX2_SRC, EX2_LIB)


def _bf16(x):
    return synth.bf16_bits_to_f32(synth.f32_to_bf16_bits(np.asarray(x, np.float32))).astype(np.float64)


def adversarial(kind: str, d: int, seed: int):
    """(Q, K) float64 arrays of bf16 values, ROWS x d each."""
    g = np.random.default_rng(seed)
    n = ROWS
    if kind == "normal":
        q, k = g.standard_normal((n, d)), g.standard_normal((n, d))
    elif kind == "student_t3":
        q, k = g.standard_t(3, (n, d)), g.standard_t(3, (n, d))
    elif kind == "magnitudes_2^+-12":
        q = g.standard_normal((n, d)) * 2.0 ** g.uniform(-12, 12, (n, d))
        k = g.standard_normal((n, d)) * 2.0 ** g.uniform(-12, 12, (n, d))
    elif kind == "one_large_many_small":
        q, k = g.standard_normal((n, d)) * 2.0 ** -6, g.standard_normal((n, d)) * 2.0 ** -6
        j = g.integers(0, d, n)
        q[np.arange(n), j] = 2.0 ** 10 * np.sign(g.standard_normal(n))
        k[np.arange(n), g.integers(0, d, n)] = 2.0 ** 10
        k[:n // 2, j[:n // 2]] = 2.0 ** 10          # half the rows share the large coordinate
    elif kind == "cancelling":
        # exact dots near zero from large terms: q = (x, x), k = (y, -y) up to small noise
        h = d // 2
        x, y = g.standard_normal((n, h)) * 64, g.standard_normal((n, h)) * 64
        q = np.concatenate([x, x + g.standard_normal((n, h)) * 2.0 ** -3], axis=1)
        k = np.concatenate([y, -y], axis=1)
    else:
        raise ValueError(kind)
    return _bf16(q), _bf16(k)


KINDS = ["normal", "student_t3", "magnitudes_2^+-12", "one_large_many_small", "cancelling"]


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("kind", KINDS)
def test_tensor_core_logit_error_within_kappa(kind, d):
    lib = ctypes.CDLL(build_probe())
    lib.umma_logits_probe.restype = ctypes.c_int
    lib.umma_logits_probe.argtypes = [ctypes.c_void_p] * 3 + [ctypes.c_int] * 3 + [ctypes.c_void_p] * 2
    Q, K = adversarial(kind, d, seed=1000 + d + KINDS.index(kind))
    dev = torch.device("cuda")
    qt = torch.from_numpy(Q.astype(np.float32)).to(dev).to(torch.bfloat16).contiguous()
    kt = torch.from_numpy(K.astype(np.float32)).to(dev).to(torch.bfloat16).contiguous()
    # the conversion is exact: the values are already bf16
    assert np.array_equal(qt.float().cpu().numpy().astype(np.float64), Q)
    out = torch.full((ROWS, ROWS), float("nan"), dtype=torch.float32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    rc = lib.umma_logits_probe(qt.data_ptr(), kt.data_ptr(), out.data_ptr(), ROWS, ROWS, d, status.data_ptr(),
                               torch.cuda.current_stream().cuda_stream)
    assert rc == 0, rc
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    got = out.cpu().numpy().astype(np.float64)
    assert np.isfinite(got).all()
    exact = Q @ K.T                              # bf16 products are exact in float64; 2^-53 summation
    err = np.abs(got - exact)
    nq, nk = np.linalg.norm(Q, axis=1), np.linalg.norm(K, axis=1)
    r_norm = float((err / np.maximum(nq[:, None] * nk[None, :], 1e-300)).max())
    r_abs = float((err / np.maximum(np.abs(Q) @ np.abs(K).T, 1e-300)).max())
    gh.record("kappa", "tensor-core logits", case=f"{kind} d={d}", logits=int(err.size), r_norm=r_norm, r_abs=r_abs)
    assert r_norm <= KAPPA / 2, (kind, d, r_norm / 2.0 ** -24)
    assert r_abs <= MODEL, (kind, d, r_abs / 2.0 ** -24)


def test_ex2_approx_error_within_kap_assumption():
    """Every fp32 input of ex2.approx.ftz.f32 with a normal result: the exponents the block scores
    take lie in [-126, 0] up to their error bound (block maxima never exceed the row maximum by more)."""
    lib = ctypes.CDLL(build_ex2_probe())
    lib.ex2_error_probe.restype = ctypes.c_int
    lib.ex2_error_probe.argtypes = [ctypes.c_uint32, ctypes.c_uint32, ctypes.c_void_p, ctypes.c_void_p]
    dev = torch.device("cuda")
    worst, arg = 0.0, 0.0
    # [-126, -0] and [+0, 0.05]
    for lo, hi in ((0x80000000, 0xC2FC0000), (0x00000000, 0x3D4CCCCD)):
        out = torch.zeros(2, dtype=torch.int64, device=dev)
        rc = lib.ex2_error_probe(lo, hi, out.data_ptr(), torch.cuda.current_stream().cuda_stream)
        assert rc == 0, rc
        torch.cuda.synchronize()
        o = out.cpu().numpy()
        rel = float(o[:1].view(np.float64)[0])
        if rel > worst:
            worst, arg = rel, float(np.array([o[1]], np.uint32).view(np.float32)[0])
    gh.record("ex2", "tensor-core logits", inputs=int(0xC2FC0000 - 0x80000000 + 0x3D4CCCCD + 2), rel=worst, arg=arg)
    assert 0.0 < worst <= EX2_REL / 2, (worst / 2.0 ** -24, arg)

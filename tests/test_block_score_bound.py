"""The per-term error bound of the KAP block scores, checked against exact values.

`kap_block_scores_kernel` takes each term of s_ij = sum_r exp(bm[r, j] * scale - M_r) in base 2,
x = 2^u with u = fmaf(bm, scale log2 e, -M_r log2 e) in fp32 and the hardware exponential, and bounds
|x - exact| by x * t, t = fmaf(C, min(|u|, 1024), fmaf(B, ||k||max, A)) with A covering the
exponential's relative error and the rounding of M_r log2 e, B the tensor-core logit error (kappa *
scale * ||q|| per unit key norm) and C the rounding of u.  The certification of the mask order and
cut trusts that bound, so it is checked here on the same fp32 arithmetic (numpy float32, fused
multiply-adds taken exactly in float64 and rounded once), with the fp32 block maximum placed at the
edge of the logit error the kernel assumes and the exponential's error at the edge of its assumed
2^-21, against exp(L - M) in float64 for the exact block-maximum logit L and the float64 row maximum M.
Dropping the exponential's share from A breaks the bound, so the check has teeth.  The kernel's
expm1f branch (large norms or row maxima) is checked the same way."""
import numpy as np

F = np.float32
SCALE = 1.0 / np.sqrt(128.0)
KAPPA = F(1.0 / 262144.0)          # the kernel's kKappa
EX2_REL = F(8.0 / 16777216.0)      # kEx2Rel, 2^-21
GROW = F(1.0 + 1.0 / 524288.0)     # kGrow
RND = F(8.5e-8)                    # kRnd
RND_M = F(1.7e-7)                  # kRndM


def f32(x):
    return np.asarray(x, dtype=np.float64).astype(np.float32)


def cases(n, seed):
    """Norm bounds of q and of the key block, exact block-maximum logits L (|L / scale| <= ||q|| ||k||),
    row maxima M >= L (scaled logits), and the fp32 block maximum bm at 90-100 % of the assumed logit
    error from L / scale."""
    rng = np.random.default_rng(seed)
    qn = f32(np.exp(rng.uniform(np.log(0.01), np.log(30.0), n)))
    kn = f32(np.exp(rng.uniform(np.log(0.01), np.log(30.0), n)))
    err_raw = KAPPA.astype(np.float64) * qn * kn             # |fp32 dot - exact dot| <= kappa ||q|| ||k||
    dot = rng.uniform(-1.0, 1.0, n) * qn * kn                 # |q . k| <= ||q|| ||k||
    L = dot * SCALE
    M = L + np.where(rng.random(n) < 0.1, 0.0, rng.uniform(0.0, 60.0, n))
    bm = f32(dot + rng.choice([-1.0, 1.0], n) * rng.uniform(0.9, 1.0, n) * err_raw)
    ok = np.abs(bm.astype(np.float64) - dot) <= err_raw       # the rounding to fp32 is part of the error
    return M[ok], L[ok], qn[ok], kn[ok], bm[ok], rng


def ex2_errors(rng, n):
    """Relative errors of the exponential near the edge of its assumed 2^-21, leaving room for the
    rounding of its float32 result (at most 2^-24 relative)."""
    return rng.choice([-1.0, 1.0], n) * (rng.uniform(0.85, 0.87, n) * float(EX2_REL))


def kernel_term(M, qn, kn, bm, eps, with_ex2_share=True):
    """x and its bound x * t as the kernel computes them (eps: the exponential's relative error)."""
    sl2 = f32(SCALE * 1.4426950408889634)
    ml2 = f32(f32(M) * F(1.44269504))
    dl = f32(f32(f32(KAPPA * F(SCALE)) * qn) * F(1.001))
    a = f32(GROW * f32((EX2_REL if with_ex2_share else F(0.0)) + f32(RND_M * np.abs(ml2))))
    b = f32(f32(GROW * F(1.02)) * dl)
    c = f32(GROW * RND)
    u = f32(bm.astype(np.float64) * sl2.astype(np.float64) - ml2.astype(np.float64))
    # the instruction's result, a float32 within eps of 2^u (its stated error includes its own rounding)
    x = f32(np.exp2(u.astype(np.float64)) * (1.0 + eps))
    assert np.all(np.abs(x.astype(np.float64) / np.exp2(u.astype(np.float64)) - 1.0) <= float(EX2_REL))
    inner = f32(b.astype(np.float64) * kn.astype(np.float64) + a.astype(np.float64))
    t = f32(c.astype(np.float64) * np.minimum(np.abs(u), F(1024.0)).astype(np.float64) + inner.astype(np.float64))
    return x, f32(x.astype(np.float64) * t.astype(np.float64)), u


def test_block_score_term_bound_holds():
    M, L, qn, kn, bm, rng = cases(400_000, 7)
    eps = ex2_errors(rng, M.size)
    x, bound, u = kernel_term(M, qn, kn, bm, eps)
    exact = np.exp(L - M)
    live = u >= -120.0          # below that the instruction flushes to 0 and the 2^-125 term covers it
    assert live.sum() > 0.9 * M.size
    assert dl_fast_path(qn, kn)
    err = np.abs(x.astype(np.float64) - exact)
    assert np.all(err[live] <= bound[live].astype(np.float64))


def dl_fast_path(qn, kn):
    """The generated cases lie on the kernel's fast path (its expm1f branch starts at dl ||k|| > 0.013)."""
    dl = (KAPPA.astype(np.float64) * SCALE * qn * 1.001) * kn
    return bool(np.all(dl <= 0.013))


def test_bound_without_the_exponential_share_breaks():
    M, L, qn, kn, bm, rng = cases(400_000, 8)
    eps = ex2_errors(rng, M.size)
    x, bound, u = kernel_term(M, qn, kn, bm, eps, with_ex2_share=False)
    exact = np.exp(L - M)
    live = u >= -120.0
    err = np.abs(x.astype(np.float64) - exact)
    assert np.any(err[live] > bound[live].astype(np.float64))


def test_block_score_term_bound_holds_on_the_expm1_branch():
    """Large norms (dl ||k|| > 0.013): the kernel bounds the relative error of each term by
    expm1(ln 2 D) * 1.01 + 2^-21 * 1.01 with D the exponent's error bound, scaled by 1 + 2^-19."""
    rng = np.random.default_rng(9)
    n = 200_000
    qn = f32(np.exp(rng.uniform(np.log(200.0), np.log(2000.0), n)))
    kn = f32(np.exp(rng.uniform(np.log(200.0), np.log(2000.0), n)))
    err_raw = KAPPA.astype(np.float64) * qn * kn
    dot = rng.uniform(-1.0, 1.0, n) * qn * kn
    L = dot * SCALE
    M = L + np.where(rng.random(n) < 0.1, 0.0, rng.uniform(0.0, 60.0, n))
    bm = f32(dot + rng.choice([-1.0, 1.0], n) * rng.uniform(0.9, 1.0, n) * err_raw)
    keep = np.abs(bm.astype(np.float64) - dot) <= err_raw
    M, L, qn, kn, bm = M[keep], L[keep], qn[keep], kn[keep], bm[keep]
    eps = ex2_errors(rng, M.size)
    sl2 = f32(SCALE * 1.4426950408889634)
    ml2 = f32(f32(M) * F(1.44269504))
    dl = f32(f32(f32(KAPPA * F(SCALE)) * qn) * F(1.001))
    b = f32(f32(GROW * F(1.02)) * dl)
    u = f32(bm.astype(np.float64) * sl2.astype(np.float64) - ml2.astype(np.float64))
    x = f32(np.exp2(u.astype(np.float64)) * (1.0 + eps))
    slow = (dl.astype(np.float64) * kn > 0.013) | (np.abs(ml2) > 1e5)
    d = f32(f32(f32(F(1.4426950408889634) * b) / f32(GROW * F(1.02))) * kn) + \
        f32(F(1.2e-7) * f32(f32(F(2.0) * np.abs(ml2)) + np.minimum(np.abs(u), F(1.0e30))))
    d = f32(d)
    rel = f32(f32(np.expm1(f32(F(0.6931472) * d)) * F(1.01)) + f32(EX2_REL * F(1.01)))
    bound = f32(x.astype(np.float64) * f32(GROW * rel).astype(np.float64))
    exact = np.exp(L - M)
    live = slow & (u >= -120.0)
    assert live.sum() > 0.5 * M.size
    err = np.abs(x.astype(np.float64) - exact)
    assert np.all(err[live] <= bound[live].astype(np.float64))

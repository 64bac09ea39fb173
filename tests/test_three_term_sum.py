"""The three-term fp32 sum the KAP kernels use where the method needs float64 accuracy: a row's exact
maximum logit (`kap_exact_kernel`) and the repaired positions' exact block maxima (the select
kernels).  The products of two bf16 values are exact in fp32; their sum is carried as hi + lo + c,
every addition taken through Knuth's two-sum into (hi, lo) and the pair's own rounding errors
gathered in c, then read out as (double(hi) + double(lo)) + double(c).

Here the same arithmetic runs in numpy float32 (IEEE single, round to nearest, no extended
precision), with the lane splits the kernels use: one lane over all d products (the bulk repair),
four lanes of d / 4 (the warp-select repair), eight of d / 8 (the exact-row kernel) and 32 of d / 32
(the block-select repair), the lanes' triples combined by xor butterflies, on
vectors whose exact sums are taken with rationals.  The property the kernels rely on: the result is
within about one float64 rounding of the exact sum, |result - S| <= 2^-52 |S| + 2^-100 sum |x|, on
inputs where a float64 running sum is not (factors across 2^-12 .. 2^12, with cancellation).  A pair
without the third term fails the same bound, so the test tells the two apart."""
from fractions import Fraction

import numpy as np
import pytest

F = np.float32


def two_sum(a, b):
    s = F(a + b)
    bb = F(s - a)
    e = F(F(a - F(s - bb)) + F(b - bb))
    return s, e


def add1(t, y, third=True):
    hi, lo, c = t
    s, e = two_sum(hi, y)
    u, eu = two_sum(e, lo)
    hi, lo = two_sum(s, u)
    return hi, lo, (F(c + eu) if third else c)


def add3(t, o, third=True):
    hi, lo, c = t
    yh, yl, yc = o
    s, e = two_sum(hi, yh)
    u, eu = two_sum(e, lo)
    u2, eu2 = two_sum(u, yl)
    hi, lo = two_sum(s, u2)
    return hi, lo, (F(F(c + yc) + F(eu + eu2)) if third else c)


def lane_split_sum(prod, lanes, third=True):
    """Each lane sums its contiguous d / lanes products; lanes then combine by xor butterflies."""
    per = len(prod) // lanes
    acc = []
    for ln in range(lanes):
        t = (F(0), F(0), F(0))
        for y in prod[ln * per:(ln + 1) * per]:
            t = add1(t, y, third)
        acc.append(t)
    o = 1
    while o < lanes:
        acc = [add3(acc[ln], acc[ln ^ o], third) for ln in range(lanes)]
        o <<= 1
    hi, lo, c = acc[0]
    return (float(hi) + float(lo)) + float(c)


def to_bf16(x):
    """Round float32 values to bf16 (nearest even), returned as float32."""
    b = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    b = (b + 0x7FFF + ((b >> 16) & 1)) & 0xFFFF0000
    return b.astype(np.uint32).view(np.float32)


def vectors(kind, n, d, rng):
    if kind == "normal":
        q, k = rng.standard_normal((n, d)), rng.standard_normal((n, d))
    elif kind == "student_t":
        q, k = rng.standard_t(3, (n, d)), rng.standard_t(3, (n, d))
    elif kind == "magnitudes":
        # factors spread over 2^-12 .. 2^12 with random signs (products over 2^-24 .. 2^24: more bits
        # than a double holds, and heavy cancellation)
        q = rng.choice([-1.0, 1.0], (n, d)) * np.exp2(rng.uniform(-12, 12, (n, d)))
        k = rng.choice([-1.0, 1.0], (n, d)) * np.exp2(rng.uniform(-12, 12, (n, d)))
    elif kind == "cancel":
        # a large pair that cancels exactly plus many small terms
        q = rng.standard_normal((n, d)) * 2.0 ** -10
        k = rng.standard_normal((n, d))
        q[:, 0], k[:, 0] = 2.0 ** 11, 1.5
        q[:, 1], k[:, 1] = -(2.0 ** 11), 1.5
    else:
        raise ValueError(kind)
    return to_bf16(q.astype(np.float32)), to_bf16(k.astype(np.float32))


def errors(q, k, lanes, third=True):
    out = []
    for qv, kv in zip(q, k):
        prod = [F(a * b) for a, b in zip(qv, kv)]
        exact = sum(Fraction(float(p)) for p in prod)
        # the products are exact in fp32
        assert all(Fraction(float(p)) == Fraction(float(a)) * Fraction(float(b)) for p, a, b in zip(prod, qv, kv))
        mag = sum(abs(Fraction(float(p))) for p in prod)
        got = lane_split_sum(prod, lanes, third)
        run = 0.0
        for p in prod:
            run += float(p)
        bound = Fraction(2) ** -52 * abs(exact) + Fraction(2) ** -100 * mag
        out.append((abs(Fraction(got) - exact), abs(Fraction(run) - exact), bound))
    return out


@pytest.mark.parametrize("d,lanes", [(128, 1), (128, 4), (128, 8), (128, 32), (64, 4)])
@pytest.mark.parametrize("kind", ["normal", "student_t", "magnitudes", "cancel"])
def test_three_term_sum_is_float64_accurate(kind, d, lanes):
    rng = np.random.default_rng(11 + d + lanes + len(kind))
    q, k = vectors(kind, 60, d, rng)
    for err3, _, bound in errors(q, k, lanes):
        assert err3 <= bound


def test_the_bound_separates_the_sums():
    """On the cancellation inputs a float64 running sum and a two-term pair both break the bound the
    three-term sum keeps, so the check above has teeth."""
    rng = np.random.default_rng(5)
    q, k = vectors("magnitudes", 200, 128, rng)
    res3 = errors(q, k, 4)
    res2 = errors(q, k, 4, third=False)
    assert all(e3 <= b for e3, _, b in res3)
    assert any(ef > b for _, ef, b in res3), "float64 running sum never broke the bound"
    assert any(e2 > b for e2, _, b in res2), "the pair without its third term never broke the bound"

"""Pins for the float64 oracle, written as functions of the oracle module.

Each check ties the oracle to something other than itself: the worked example the
PageWeaver notes print, a textbook routine the method reduces to (dense causal
attention when every block is selected and skipping is off), closed forms of
hand-built cases, invariants that the equations imply, and brute force on tiny
inputs.  ``tests/test_oracle_pins.py`` runs them on the oracle;
``tests/test_oracle_mutations.py`` runs them on copies of the oracle with planted
mistakes and expects each mistake to be caught.
"""
from __future__ import annotations

import json
import math
import os

import numpy as np

import synth

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


# --------------------------------------------------------------------------- #
# helpers (independent of the oracle)
# --------------------------------------------------------------------------- #
def f64(bits):
    return synth.bf16_bits_to_f32(bits).astype(np.float64)


def bits(x):
    return synth.f32_to_bf16_bits(np.asarray(x, dtype=np.float32))


def tiny_spec(**kw):
    base = dict(name="tiny", lengths=(300, 173), num_q_heads=4, num_kv_heads=2, head_dim=16,
                block_size=32, page_size=16, stride=4, budget_ppm=400_000, stage2_budget_ppm=0,
                seed=11, shuffle_pages=True, salient_pages=3)
    base.update(kw)
    return synth.WorkloadSpec(**base)


def logical_kv(w, b, kv_head):
    """Tokens of request b in logical order, gathered with numpy fancy indexing."""
    L = w.lengths[b]
    P = w.spec.page_size
    t = np.arange(L)
    phys = w.page_table[b, t // P]
    return f64(w.k_cache[phys, t % P, kv_head, :]), f64(w.v_cache[phys, t % P, kv_head, :])


def params(orc, spec, budget_ppm=None, delta=-1.0):
    return orc.Params(spec.block_size, spec.page_size, spec.stride,
                      spec.budget_ppm if budget_ppm is None else budget_ppm,
                      1.0 / math.sqrt(spec.head_dim), float(delta))


def hand_problem(k_vals, v_vals, q_rows, L):
    """d = 1, b = P = s = 1 style arrays for hand-built cases (values exact in bf16)."""
    q = bits(np.asarray(q_rows, dtype=np.float32).reshape(L, 1, 1))
    k = bits(np.asarray(k_vals, dtype=np.float32).reshape(L, 1, 1, 1))
    v = bits(np.asarray(v_vals, dtype=np.float32).reshape(L, 1, 1, 1))
    return q, k, v


# --------------------------------------------------------------------------- #
# token-set semantics (PageWeaver Sec. 2.1)
# --------------------------------------------------------------------------- #
def check_token_set_worked_example(orc):
    g = json.load(open(os.path.join(GOLDEN, "pageweaver_token_set.json")))
    assert orc.token_set(g["S"], g["P"], g["L"], g["c"]) == g["A"]
    # duplicates count once, invalid IDs add nothing, empty support is empty
    assert orc.token_set([0, 2, 2, 0], 4, 11, 9) == g["A"]
    assert orc.token_set([0, 2, -1, 7, 100], 4, 11, 9) == g["A"]
    assert orc.token_set([], 4, 11, 9) == []
    assert orc.token_set([1], 4, 11, 3) == []            # page 1 starts after c


# --------------------------------------------------------------------------- #
# OSK reduces to dense causal attention (budget 100 %, skip off)
# --------------------------------------------------------------------------- #
def check_dense_reduction(orc):
    import torch
    spec = tiny_spec(budget_ppm=1_000_000)
    w = synth.make_workload(spec)
    prm = params(orc, spec, delta=-1.0)
    b = spec.block_size
    B = spec.num_reqs
    nqb_max = -(-spec.max_seqlen // b)
    mask = np.full((B, spec.num_q_heads, nqb_max, nqb_max), -1, np.int32)
    mask_len = np.zeros((B, spec.num_q_heads, nqb_max), np.int32)
    rng = np.random.default_rng(3)
    for bi in range(B):
        for h in range(spec.num_q_heads):
            for i in range(-(-w.lengths[bi] // b)):
                mask[bi, h, i, :i + 1] = rng.permutation(i + 1)
                mask_len[bi, h, i] = i + 1
    res = orc.osk_all(w.q, w.k_cache, w.v_cache, w.page_table, w.cu_seqlens, spec.num_q_heads,
                      spec.num_kv_heads, prm, mask, mask_len)
    G = spec.num_q_heads // spec.num_kv_heads
    for bi in range(B):
        L = w.lengths[bi]
        for h in range(spec.num_q_heads):
            K, V = logical_kv(w, bi, h // G)
            Q = f64(w.q[w.cu_seqlens[bi]:w.cu_seqlens[bi + 1], h, :])
            ref = torch.nn.functional.scaled_dot_product_attention(
                torch.from_numpy(Q)[None, None], torch.from_numpy(K)[None, None],
                torch.from_numpy(V)[None, None], is_causal=True, scale=prm.sm_scale)[0, 0].numpy()
            for i in range(-(-L // b)):
                out = res[(bi, h, i)].out
                np.testing.assert_allclose(out, ref[i * b:min(L, (i + 1) * b)], rtol=0, atol=1e-12)
                assert (res[(bi, h, i)].flags == orc.COMPUTED).all()


# --------------------------------------------------------------------------- #
# Property 2: visiting order does not change O (skip off)
# --------------------------------------------------------------------------- #
def check_order_invariance(orc):
    spec = tiny_spec(lengths=(480,), seed=5)
    w = synth.make_workload(spec)
    prm = params(orc, spec, delta=-1.0)
    rng = np.random.default_rng(9)
    G = spec.num_q_heads // spec.num_kv_heads
    Q = f64(w.q[:, 1, :])
    from oracle import cosa_oracle as base   # resolve keys with the unmutated reader
    K, ex = base.request_keys(w.k_cache, w.page_table[0], 480, spec.page_size, 1 // G)
    V, _ = base.request_keys(w.v_cache, w.page_table[0], 480, spec.page_size, 1 // G)
    for i in (3, 9, 14):
        sel = rng.choice(i + 1, size=max(2, (i + 1) // 2), replace=False)
        outs = []
        for _ in range(3):
            row = rng.permutation(sel)
            outs.append(orc.osk_qblock(Q, K, V, ex, i, row, len(row), prm).out)
        for o in outs[1:]:
            np.testing.assert_allclose(o, outs[0], rtol=0, atol=1e-12)


# --------------------------------------------------------------------------- #
# PageWeaver Eq. (2) on the selected token set; invalid pages, IDs and repeats
# --------------------------------------------------------------------------- #
def check_direct_definition(orc):
    import torch
    spec = tiny_spec(lengths=(333,), seed=21)
    w = synth.make_workload(spec)
    # two pages of the request disappear from the table (one negative, one out of range)
    w.page_table[0, 3] = -1
    w.page_table[0, 9] = spec.num_pages + 5
    prm = params(orc, spec, delta=-1.0)
    b, P = spec.block_size, spec.page_size
    L = 333
    t = np.arange(L)
    page = t // P
    exists = (w.page_table[0, page] >= 0) & (w.page_table[0, page] < spec.num_pages)
    phys = np.clip(w.page_table[0, page], 0, spec.num_pages - 1)
    h, kvh = 2, 2 // (spec.num_q_heads // spec.num_kv_heads)
    K = f64(w.k_cache[phys, t % P, kvh, :])
    V = f64(w.v_cache[phys, t % P, kvh, :])
    Q = f64(w.q[:, h, :])
    from oracle import cosa_oracle as base
    Ko, ex = base.request_keys(w.k_cache, w.page_table[0], L, P, kvh)
    Vo, _ = base.request_keys(w.v_cache, w.page_table[0], L, P, kvh)
    i = 10                                   # last block is ragged: 333 = 10 * 32 + 13
    row = [4, -3, 10, 4, 11, 0, 7, 99, 2, 10]
    res = orc.osk_qblock(Q, Ko, Vo, ex, i, row, len(row), prm)
    assert list(res.flags) == [0, 2, 0, 2, 2, 0, 0, 2, 0, 2]
    valid_blocks = [4, 10, 0, 7, 2]
    for r in range(res.out.shape[0]):
        pos = i * b + r
        toks = [tt for tt in range(L) if (tt // b) in valid_blocks and tt <= pos and exists[tt]]
        z = torch.from_numpy(K[toks] @ Q[pos]) * prm.sm_scale
        ref = (torch.softmax(z, 0).numpy()[:, None] * V[toks]).sum(0)
        np.testing.assert_allclose(res.out[r], ref, rtol=0, atol=1e-12)
        np.testing.assert_allclose(res.out[r], orc.direct_output(Q[pos], K, V, toks, prm.sm_scale), atol=1e-12)
    # duplicates / invalid IDs add no mass: bit-identical to the cleaned row
    clean = orc.osk_qblock(Q, Ko, Vo, ex, i, valid_blocks, len(valid_blocks), prm)
    assert np.array_equal(clean.out, res.out)
    # a block after the query block (j > i) is not a causal candidate: ignored, not visited
    mid = orc.osk_qblock(Q, Ko, Vo, ex, 5, [2, 7, 5, 6], 4, prm)
    assert list(mid.flags) == [0, 2, 0, 2]
    # empty support gives zero
    empty = orc.osk_qblock(Q, Ko, Vo, ex, i, [-1, 12, 11, -5], 4, prm)
    assert np.array_equal(empty.out, np.zeros_like(empty.out))
    assert (empty.flags == orc.IGNORED).all()


# --------------------------------------------------------------------------- #
# skip rule (Eq. 5, Algorithm A (the skip test)): hand-built cases with closed forms
# --------------------------------------------------------------------------- #
def _skip_case(orc, delta, order):
    # one row (position 7), b = P = s = 1, d = 1, scale 1: logit of token t is k_t
    k = [1, 0, 0, 4, 0, 3, 0, 5]
    v = [10, 0, 0, 20, 0, 30, 0, 40]
    q, kc, vc = hand_problem(k, v, [1.0] * 8, 8)
    prm = orc.Params(1, 1, 1, 1_000_000, 1.0, float(delta))
    K = f64(kc[:, 0, 0, :])
    V = f64(vc[:, 0, 0, :])
    Q = f64(q[:, 0, :])
    return orc.osk_qblock(Q, K, V, np.ones(8, bool), 7, order, len(order), prm)


def check_skip_hand_cases(orc):
    e = math.exp
    # HRM-first order, delta = 1 -> tau = ln(1/8): block 0 (logit 1, 4 below the max 5) is skipped
    r = _skip_case(orc, 1.0, [7, 3, 0, 5])
    assert list(r.flags) == [0, 0, 1, 0]
    tau = math.log(1 / 8)
    np.testing.assert_allclose(r.margins, [0 - tau, -1 - tau, -4 - tau, -2 - tau], atol=1e-12)
    want = (e(5) * 40 + e(4) * 20 + e(3) * 30) / (e(5) + e(4) + e(3))
    np.testing.assert_allclose(r.out[0, 0], want, rtol=1e-13)
    # ascending order with the same delta: the running max rises late, nothing is skipped
    r = _skip_case(orc, 1.0, [0, 3, 5, 7])
    assert list(r.flags) == [0, 0, 0, 0]
    # skip off (delta = -1): every block computed
    r = _skip_case(orc, -1.0, [7, 3, 0, 5])
    assert list(r.flags) == [0, 0, 0, 0]
    want = (e(5) * 40 + e(4) * 20 + e(1) * 10 + e(3) * 30) / (e(5) + e(4) + e(1) + e(3))
    np.testing.assert_allclose(r.out[0, 0], want, rtol=1e-13)
    # delta = N: tau = 0, only blocks strictly below the running max are skipped
    r = _skip_case(orc, 8.0, [7, 3, 0, 5])
    assert list(r.flags) == [0, 1, 1, 1]
    np.testing.assert_allclose(r.out[0, 0], 40.0, rtol=1e-13)
    # delta > N: tau > 0, even the first visit is skipped and O = 0 (empty support)
    r = _skip_case(orc, 9.0, [7, 3, 0, 5])
    assert list(r.flags) == [1, 1, 1, 1]
    assert r.out[0, 0] == 0.0


def check_skip_bucket_case(orc):
    # two query rows (positions 4, 5) with opposite queries; b = P = 2, s = 1, d = 1, scale 1.
    # block 1 is negligible for row 4 but holds row 5's maximum, so row 5 vetoes its skip (Eq. 5 AND).
    k = [3, 0, -3, 0, 0, 0]
    v = [1, 2, 3, 4, 5, 6]
    q, kc, vc = hand_problem(k, v, [0, 0, 0, 0, 1, -1], 6)
    kc = kc.reshape(3, 2, 1, 1)
    vc = vc.reshape(3, 2, 1, 1)
    prm = orc.Params(2, 2, 1, 1_000_000, 1.0, 1.0)       # tau = ln(1/6)
    from oracle import cosa_oracle as base
    K, ex = base.request_keys(kc, np.arange(3), 6, 2, 0)
    V, _ = base.request_keys(vc, np.arange(3), 6, 2, 0)
    Q = f64(q[:, 0, :])
    r = orc.osk_qblock(Q, K, V, ex, 2, [0, 1, 2], 3, prm)
    assert list(r.flags) == [0, 0, 1]
    np.testing.assert_allclose(r.margins, [0 - math.log(1 / 6), 0 - math.log(1 / 6), -3 - math.log(1 / 6)],
                               atol=1e-12)
    e = math.exp
    w4 = np.array([e(3), e(0), e(-3), e(0)])
    w5 = np.array([e(-3), e(0), e(3), e(0)])
    vv = np.array([1, 2, 3, 4.0])
    np.testing.assert_allclose(r.out[:, 0], [w4 @ vv / w4.sum(), w5 @ vv / w5.sum()], rtol=1e-13)


def check_skip_invariants(orc):
    spec = tiny_spec(lengths=(640,), seed=33, budget_ppm=600_000)
    w = synth.make_workload(spec)
    prm0 = params(orc, spec, delta=-1.0)
    kmax = 20
    mask, ml, _ = orc.kap_mask(w.q, w.k_cache, w.page_table, w.cu_seqlens, spec.num_q_heads,
                               spec.num_kv_heads, prm0, kmax)
    prm = params(orc, spec, delta=60.0)                   # tau = ln(60/640)
    res = orc.osk_all(w.q, w.k_cache, w.v_cache, w.page_table, w.cu_seqlens, spec.num_q_heads,
                      spec.num_kv_heads, prm, mask, ml)
    n_skip = 0
    for key, r in res.items():
        tested = r.flags != orc.IGNORED
        first = np.nonzero(tested)[0][0]
        assert r.flags[first] == orc.COMPUTED                 # first visit is never skipped (delta < L)
        assert ((r.margins[tested] < 0) == (r.flags[tested] == orc.SKIPPED)).all()
        n_skip += int((r.flags == orc.SKIPPED).sum())
        # replaying this oracle's own decisions reproduces the same output bit for bit
        b, h, i = key
        again = orc.osk_all(w.q, w.k_cache, w.v_cache, w.page_table, w.cu_seqlens, spec.num_q_heads,
                            spec.num_kv_heads, prm, mask, ml, items=[key], force={key: r.flags})[key]
        assert np.array_equal(again.out, r.out)
    assert n_skip > 0


# --------------------------------------------------------------------------- #
# KAP (Eqs. 8-14)
# --------------------------------------------------------------------------- #
def check_stage1_count(orc):
    assert orc.stage1_count(100_000, 10) == 1                # 0.1 * 10 = 1 exactly
    assert orc.stage1_count(100_000, 11) == 2
    assert orc.stage1_count(250_000, 3) == 1
    assert orc.stage1_count(200_000, 64) == 13               # ceil(12.8)
    assert orc.stage1_count(1_000_000, 37) == 37
    assert orc.stage1_count(1, 5) == 1


def _kap_hand(orc, k_vals):
    # d = 1, scale 1, b = P = 2, s = 1: query block 2 holds rows 4 and 5 with q = 1
    q, kc, vc = hand_problem(k_vals, [0] * 6, [1.0] * 6, 6)
    kc = kc.reshape(3, 2, 1, 1)
    prm = orc.Params(2, 2, 1, 1_000_000, 1.0, -1.0)
    from oracle import cosa_oracle as base
    K, ex = base.request_keys(kc, np.arange(3), 6, 2, 0)
    Q = f64(q[:, 0, :])
    return orc.kap_request_head(Q, K, ex, prm, [2])[2]


def check_kap_hand_cases(orc):
    e = math.exp
    # HRM blocks 0 and 2 (row 4 peaks in block 0, row 5 in block 2); block 1 outscores block 2
    # but the HRM group goes first (Eq. 13).
    row = _kap_hand(orc, [4, 0, 3.75, 0, 0, 4.5])
    np.testing.assert_allclose(row.scores, [1 + e(-0.5), e(-0.25) + e(-0.75), e(-4) + 1], rtol=1e-13)
    assert list(row.hrm) == [True, False, True]
    assert list(row.order) == [0, 2, 1]
    # one HRM block, rest sorted by score
    row = _kap_hand(orc, [2, 0, 1, 3, 0, 1])
    np.testing.assert_allclose(row.scores, [2 * e(-1), 2.0, e(-3) + e(-2)], rtol=1e-13)
    assert list(row.hrm) == [False, True, False]
    assert list(row.order) == [1, 0, 2]
    # exact tie between blocks 0 and 2: ascending block index
    row = _kap_hand(orc, [1, 0, 3, 0, 1, 0])
    assert row.scores[0] == row.scores[2]
    assert list(row.order) == [1, 0, 2]


def _kap_brute(Qs, pos, Ks, kex, b, n_blocks, scale):
    """Literal per-entry loops over Eqs. (8)-(12) with math.exp."""
    R = len(pos)
    pbar = np.zeros((R, n_blocks))
    for r in range(R):
        vis = [c for c in range(len(pos)) if pos[c] <= pos[r] and kex[c]]
        if not vis:
            continue
        lg = {c: float(np.dot(Qs[r], Ks[c])) * scale for c in vis}
        mx = max(lg.values())
        Z = sum(math.exp(x - mx) for x in lg.values())
        S = {c: math.exp(x - mx) / Z for c, x in lg.items()}
        Pm = [max([S[c] for c in vis if pos[c] // b == j], default=0.0) for j in range(n_blocks)]
        pm = max(Pm)
        pbar[r] = [p / pm for p in Pm]
    return pbar


def check_kap_brute_force(orc):
    spec = tiny_spec(lengths=(200,), head_dim=8, block_size=16, page_size=8, stride=4, seed=44)
    w = synth.make_workload(spec)
    w.page_table[0, 5] = -1                                  # one page of keys does not exist
    prm = params(orc, spec, budget_ppm=500_000)
    from oracle import cosa_oracle as base
    for h in (0, 3):
        kvh = h // (spec.num_q_heads // spec.num_kv_heads)
        K, ex = base.request_keys(w.k_cache, w.page_table[0], 200, spec.page_size, kvh)
        Q = f64(w.q[:, h, :])
        pos = np.arange(0, 200, spec.stride)
        got = orc.kap_request_head(Q, K, ex, prm)
        for i, row in got.items():
            ridx = np.nonzero(pos // spec.block_size == i)[0]
            pb = _kap_brute(Q[pos], pos, K[pos], ex[pos], spec.block_size, i + 1, prm.sm_scale)[ridx]
            np.testing.assert_allclose(row.pbar, pb, rtol=0, atol=1e-13)
            s = pb.sum(axis=0)
            np.testing.assert_allclose(row.scores, s, rtol=1e-13, atol=1e-15)
            hrm = (pb == 1.0).any(axis=0)
            assert np.array_equal(row.hrm, hrm)
            keys = sorted(range(i + 1), key=lambda j: (not hrm[j], -s[j], j))
            assert list(row.order) == keys


def check_kap_invariants(orc):
    spec = tiny_spec(lengths=(512,), seed=55)
    w = synth.make_workload(spec)
    prm = params(orc, spec)
    G = spec.num_q_heads // spec.num_kv_heads
    from oracle import cosa_oracle as base
    kb = spec.block_size // spec.stride
    for h in range(spec.num_q_heads):
        K, ex = base.request_keys(w.k_cache, w.page_table[0], 512, spec.page_size, h // G)
        Q = f64(w.q[:, h, :])
        for i, row in orc.kap_request_head(Q, K, ex, prm).items():
            assert row.pbar.shape == (kb, i + 1)
            assert (row.pbar >= 0).all() and (row.pbar <= 1).all()
            assert ((row.pbar == 1.0).sum(axis=1) >= 1).all()      # each row's own maximum
            nh = int(row.hrm.sum())
            assert 1 <= nh <= kb
            assert sorted(row.order.tolist()) == list(range(i + 1))
            assert row.hrm[row.order[:nh]].all() and not row.hrm[row.order[nh:]].any()
            for grp in (row.order[:nh], row.order[nh:]):
                sc = row.scores[grp]
                assert (np.diff(sc) <= 0).all()
            assert row.K == orc.stage1_count(prm.budget_ppm, i + 1)
            # direct form of Eqs. (9)-(10): Pbar = exp(blockmax - rowmax) on the logits
            pos = np.arange(0, 512, spec.stride)
            rp = pos[pos // spec.block_size == i]
            lg = (Q[rp] @ K[pos].T) * prm.sm_scale
            lg = np.where((pos[None, :] <= rp[:, None]) & ex[pos][None, :], lg, -np.inf)
            bm = np.stack([lg[:, (pos // spec.block_size) == j].max(axis=1) for j in range(i + 1)], 1)
            np.testing.assert_allclose(row.pbar, np.exp(bm - bm.max(axis=1, keepdims=True)), rtol=1e-12, atol=0)
            assert np.array_equal(row.hrm, (bm == bm.max(axis=1, keepdims=True)).any(axis=0))


def check_kap_mask_layout(orc):
    spec = tiny_spec(seed=66)
    w = synth.make_workload(spec)
    prm = params(orc, spec)
    kmax = 7
    mask, ml, rows = orc.kap_mask(w.q, w.k_cache, w.page_table, w.cu_seqlens, spec.num_q_heads,
                                  spec.num_kv_heads, prm, kmax)
    for (b, h, i), row in rows.items():
        assert ml[b, h, i] == row.K
        assert list(mask[b, h, i, :row.K]) == list(row.order[:row.K])
        assert (mask[b, h, i, row.K:] == -1).all()
    nqb1 = -(-spec.lengths[1] // spec.block_size)
    assert (ml[1, :, nqb1:] == 0).all() and (mask[1, :, nqb1:] == -1).all()


def check_top_p_count(orc):
    e = math.exp

    def hand(k_vals, ppm):
        q, kc, _ = hand_problem(k_vals, [0] * 6, [1.0] * 6, 6)
        kc = kc.reshape(3, 2, 1, 1)
        prm = orc.Params(2, 2, 1, ppm, 1.0, -1.0, top_p=True)
        from oracle import cosa_oracle as base
        K, ex = base.request_keys(kc, np.arange(3), 6, 2, 0)
        return orc.kap_request_head(f64(q[:, 0, :]), K, ex, prm, [2])[2]

    # scores [2/e, 2, e^-3 + e^-2], rho = [1, 0, 2], total T = 2.92088...
    T = 2 * e(-1) + 2 + e(-3) + e(-2)
    for ppm, want in ((500_000, 1), (900_000, 2), (950_000, 3), (1_000_000, 3), (1, 1)):
        assert hand([2, 0, 1, 3, 0, 1], ppm).K == want, (ppm, want)
    assert 2 < 0.9 * T <= 2 + 2 * e(-1) < 0.95 * T            # the closed form behind 2 and 3
    # HRM first: scores [1 + e^-0.5, e^-0.25 + e^-0.75, e^-4 + 1], rho = [0, 2, 1].  At p = 0.7 the
    # prefix {0, 2} holds 2.62 < 0.7 T = 2.71, so K = 3 (a score-ordered prefix {0, 1} would stop at 2)
    row = hand([4, 0, 3.75, 0, 0, 4.5], 700_000)
    assert list(row.order) == [0, 2, 1] and row.K == 3
    assert hand([4, 0, 3.75, 0, 0, 4.5], 600_000).K == 2
    # seeded batch: K_i is the shortest rho_i prefix reaching p T (plain loop), and grows with p
    spec = tiny_spec(seed=68)
    w = synth.make_workload(spec)
    prev = None
    for ppm in (300_000, 800_000, 950_000):
        prm = orc.Params(spec.block_size, spec.page_size, spec.stride, ppm, 1.0 / math.sqrt(spec.head_dim),
                         -1.0, top_p=True)
        _, ml, rows = orc.kap_mask(w.q, w.k_cache, w.page_table, w.cu_seqlens, spec.num_q_heads,
                                   spec.num_kv_heads, prm, 64)
        for key, r in rows.items():
            tot = 0.0
            for j in range(len(r.scores)):
                tot += r.scores[r.order[j]]
            run, k = 0.0, 0
            while True:
                run += r.scores[r.order[k]]
                k += 1
                if run >= ppm / 1e6 * tot:
                    break
            assert r.K == k == ml[key], (key, r.K, k)
        if prev is not None:
            assert (ml >= prev).all()
        prev = ml


def check_query_union(orc):
    g = json.load(open(os.path.join(GOLDEN, "pageweaver_union.json")))
    U, M = orc.query_union(g["S"])
    assert U == g["U"]
    assert M.tolist() == [[1, 1, 1, 0], [1, 1, 0, 1]]        # q0 skips page 9, q2 skips page 7
    assert orc.reuse_rate([g["S"]]) == g["rho_Q"]
    assert orc.reuse_rate([[[3, 3, 5]], [[5]]]) == 1.0         # singletons: no reuse; repeats count once
    # ordered sharing: one common order loads |U| blocks; disjoint sets load sum |S_i|; reversed orders
    # of the same set force a load per head and block except where both wait for the same one
    assert orc.ordered_shared_loads([[1, 4, 7], [1, 4, 7]]) == 3
    assert orc.ordered_shared_loads([[1, 2], [3, 4]]) == 4
    assert orc.ordered_shared_loads([[1, 4, 7], [1, 4, 9]]) == 4
    assert orc.ordered_shared_loads([[1, 2, 3], [3, 2, 1]]) == 5  # 1|3, then 2 for both, then 3|1
    assert orc.ordered_shared_loads([[5, 5, 2], [2]]) == 3     # repeats count once; greedy takes 2 first (5, 2 would do)
    rng = np.random.default_rng(4)
    for _ in range(50):
        G = [list(rng.choice(20, size=int(rng.integers(0, 8)), replace=False)) for _ in range(4)]
        n = orc.ordered_shared_loads(G)
        assert len(orc.query_union(G)[0]) <= n <= sum(len(S) for S in G)


def check_union_traversal(orc):
    # by hand: heads wait for 5 and 3 -> the lower ID (3) serves head 1 alone; then both wait for 5;
    # then 3 for head 0; then both wait for 7
    assert orc.union_traversal([[5, 3, 7], [3, 5, 7]]) == [(3, (1,)), (5, (0, 1)), (3, (0,)), (7, (0, 1))]
    assert orc.union_traversal([[1, 2], [3, 4]]) == [(1, (0,)), (2, (0,)), (3, (1,)), (4, (1,))]
    assert orc.union_traversal([[4, 4, 9], [], [9]]) == [(4, (0,)), (9, (0, 2))]      # repeats once
    assert orc.union_traversal([[2, 8], [8, 2], [8]]) == [(8, (1, 2)), (2, (0, 1)), (8, (0,))]  # most heads first
    assert orc.union_traversal([[], []]) == []
    rng = np.random.default_rng(5)
    for _ in range(100):
        H = int(rng.integers(1, 5))
        G = [list(rng.integers(0, 12, size=int(rng.integers(0, 9)))) for _ in range(H)]
        loads = orc.union_traversal(G)
        assert len(loads) == orc.ordered_shared_loads(G)
        pos = [0] * H
        seqs = [list(dict.fromkeys(int(x) for x in o)) for o in G]
        for blk, members in loads:
            assert members and list(members) == sorted(set(members))
            # exactly the heads whose next pending block this is, and as many as any candidate has
            nxt = [q[p] if p < len(q) else None for p, q in zip(pos, seqs)]
            assert [h for h in range(H) if nxt[h] == blk] == list(members)
            counts = {b: nxt.count(b) for b in nxt if b is not None}
            assert len(members) == max(counts.values())
            assert blk == min(b for b, c in counts.items() if c == len(members))
            for h in members:
                pos[h] += 1
        # every head saw its own order, in order, once
        assert pos == [len(q) for q in seqs]
        for h in range(H):
            assert [b for b, m in loads if h in m] == seqs[h]


def check_kept_visits(orc):
    # row of query block 3 (4 blocks exist): -1 and 5 are invalid, the second 2 repeats the first
    assert orc.kept_visits([2, -1, 2, 0, 5, 1, 3], 7, 3, 4) == [(0, 2), (3, 0), (5, 1), (6, 3)]
    assert orc.kept_visits([2, -1, 2, 0, 5, 1, 3], 5, 3, 4) == [(0, 2), (3, 0)]   # entries past n unread
    assert orc.kept_visits([0, 1, 2], 3, 2, 2) == [(0, 0), (1, 1)]               # block 2 does not exist
    # the same entries as osk_qblock visits (those it does not flag IGNORED)
    rng = np.random.default_rng(6)
    for _ in range(40):
        i, nblk = int(rng.integers(0, 6)), int(rng.integers(1, 7))
        row = rng.integers(-2, 8, size=9)
        n = int(rng.integers(0, 10))
        L, d = 4 * nblk, 4
        Q = rng.standard_normal((L, d))
        r = orc.osk_qblock(Q, Q, Q, np.ones(L, bool), min(i, nblk - 1), row, min(n, 9),
                           orc.Params(4, 4, 1, 1_000_000, 0.5, -1.0))
        kept = orc.kept_visits(row, min(n, 9), min(i, nblk - 1), nblk)
        assert [k for k, _ in kept] == [k for k in range(min(n, 9)) if r.flags[k] != orc.IGNORED]


# --------------------------------------------------------------------------- #
# ablation modes: ascending-order visiting (no remap) and binary-mask visiting
# --------------------------------------------------------------------------- #
def check_ascending_mask(orc):
    # hand case of _kap_hand: rho_2 = [1, 0, 2]; K_2 = ceil(0.6 * 3) = 2 keeps {1, 0}, written as [0, 1]
    q, kc, _ = hand_problem([2, 0, 1, 3, 0, 1], [0] * 6, [1.0] * 6, 6)
    kc = kc.reshape(3, 2, 1, 1)
    prm = orc.Params(2, 2, 1, 600_000, 1.0, -1.0)
    cu = np.array([0, 6], np.int32)
    pt = np.arange(3, dtype=np.int32)[None, :]
    m, ml, _ = orc.kap_mask(q, kc, pt, cu, 1, 1, prm, 3)
    assert list(m[0, 0, 2]) == [1, 0, -1] and ml[0, 0, 2] == 2
    m, ml, _ = orc.kap_mask(q, kc, pt, cu, 1, 1, prm, 3, ascending=True)
    assert list(m[0, 0, 2]) == [0, 1, -1] and ml[0, 0, 2] == 2
    # on a seeded workload: same lengths, same sets, strictly ascending rows, -1 tails
    spec = tiny_spec(seed=67)
    w = synth.make_workload(spec)
    prm = params(orc, spec)
    args = (w.q, w.k_cache, w.page_table, w.cu_seqlens, spec.num_q_heads, spec.num_kv_heads, prm, 9)
    m0, l0, _ = orc.kap_mask(*args)
    m1, l1, _ = orc.kap_mask(*args, ascending=True)
    assert np.array_equal(l0, l1)
    for idx in np.ndindex(l0.shape):
        n = int(l0[idx])
        row = m1[idx]
        assert sorted(m0[idx][:n].tolist()) == row[:n].tolist()
        assert (np.diff(row[:n]) > 0).all() and (row[n:] == -1).all()


def check_binary_mask_visiting(orc):
    e = math.exp
    # Eq. (3) from an ID list: invalid, future and repeated IDs select nothing
    ids = np.full((1, 1, 4, 5), -1, np.int32)
    ids[0, 0, 3] = [2, 0, -1, 5, 2]
    ids[0, 0, 1] = [1, 0, 0, 1, 0]
    m01, l01 = orc.binary_mask(ids, np.array([[[0, 2, 0, 5]]], np.int32), 6)
    assert m01[0, 0, 3].tolist() == [1, 0, 1, 0, 0, 0] and m01[0, 0, 1].tolist() == [1, 1, 0, 0, 0, 0]
    assert m01[0, 0, 0].tolist() == [0] * 6 and m01[0, 0, 2].tolist() == [0] * 6
    assert l01[0, 0].tolist() == [0, 2, 0, 4]
    # the hand case of _skip_case, walked in ascending order under the binary mask {0, 3, 5, 7}
    k = [1, 0, 0, 4, 0, 3, 0, 5]
    v = [10, 0, 0, 20, 0, 30, 0, 40]
    q, kc, vc = hand_problem(k, v, [1.0] * 8, 8)
    K = f64(kc[:, 0, 0, :])
    V = f64(vc[:, 0, 0, :])
    Q = f64(q[:, 0, :])
    row = [1, 0, 0, 1, 0, 1, 0, 1]
    # delta = 1 (tau = ln(1/8)): ascending visiting skips nothing
    r = orc.osk_qblock_binary(Q, K, V, np.ones(8, bool), 7, row, 8, orc.Params(1, 1, 1, 1_000_000, 1.0, 1.0))
    assert list(r.flags) == [0, 2, 2, 0, 2, 0, 2, 0]
    want = (e(1) * 10 + e(4) * 20 + e(3) * 30 + e(5) * 40) / (e(1) + e(4) + e(3) + e(5))
    np.testing.assert_allclose(r.out[0, 0], want, rtol=1e-13)
    # delta = N (tau = 0): block 5 (logit 3) comes after block 3 (logit 4) and is skipped
    r = orc.osk_qblock_binary(Q, K, V, np.ones(8, bool), 7, row, 8, orc.Params(1, 1, 1, 1_000_000, 1.0, 8.0))
    assert list(r.flags) == [0, 2, 2, 0, 2, 1, 2, 0]
    np.testing.assert_allclose(r.margins[[0, 3, 5, 7]], [0.0, 0.0, -1.0, 0.0], atol=1e-12)
    want = (e(1) * 10 + e(4) * 20 + e(5) * 40) / (e(1) + e(4) + e(5))
    np.testing.assert_allclose(r.out[0, 0], want, rtol=1e-13)
    # a walk shorter than the candidates: blocks past it are not visited
    r = orc.osk_qblock_binary(Q, K, V, np.ones(8, bool), 7, row, 4, orc.Params(1, 1, 1, 1_000_000, 1.0, -1.0))
    assert list(r.flags) == [0, 2, 2, 0]
    np.testing.assert_allclose(r.out[0, 0], (e(1) * 10 + e(4) * 20) / (e(1) + e(4)), rtol=1e-13)
    # every block selected and skipping off: dense causal attention
    import torch
    spec = tiny_spec(lengths=(200,), seed=12)
    w = synth.make_workload(spec)
    prm = params(orc, spec, delta=-1.0)
    b = spec.block_size
    nqb = -(-200 // b)
    ones = np.ones((1, spec.num_q_heads, nqb, nqb), np.int32)
    lens = np.broadcast_to(np.arange(1, nqb + 1, dtype=np.int32), (1, spec.num_q_heads, nqb)).copy()
    res = orc.osk_all(w.q, w.k_cache, w.v_cache, w.page_table, w.cu_seqlens, spec.num_q_heads,
                      spec.num_kv_heads, prm, ones, lens, items=[(0, 3, i) for i in range(nqb)], binary=True)
    Kd, Vd = logical_kv(w, 0, 3 // (spec.num_q_heads // spec.num_kv_heads))
    Qd = f64(w.q[:, 3, :])
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(Qd)[None, None], torch.from_numpy(Kd)[None, None],
        torch.from_numpy(Vd)[None, None], is_causal=True, scale=prm.sm_scale)[0, 0].numpy()
    for i in range(nqb):
        np.testing.assert_allclose(res[(0, 3, i)].out, ref[i * b:min(200, (i + 1) * b)], rtol=0, atol=1e-12)
        assert (res[(0, 3, i)].flags == orc.COMPUTED).all()


ALL_CHECKS = [
    check_token_set_worked_example, check_dense_reduction, check_order_invariance,
    check_direct_definition, check_skip_hand_cases, check_skip_bucket_case, check_skip_invariants,
    check_stage1_count, check_kap_hand_cases, check_kap_brute_force, check_kap_invariants,
    check_kap_mask_layout, check_ascending_mask, check_binary_mask_visiting, check_top_p_count,
    check_query_union, check_union_traversal, check_kept_visits,
]

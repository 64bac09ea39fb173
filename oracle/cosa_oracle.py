"""Float64 CPU oracle for CoSA sparse prefill: the Kernel-Aware Proxy (KAP) and the
Ordered-Skipping Kernel (OSK).

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` may import or run this module.  It shares no code
with the CUDA path: it decodes the bf16 inputs itself, resolves pages through the
page table itself, and computes every step in float64 with numpy.

Sources (paper "CoSA: Accelerating Long-Context Inference via Proxy-Kernel
Co-Designed Sparse Attention", arXiv 2607.25291v1, and the PageWeaver notes):

  * KAP block ranking, Sec. 4.2, Eqs. (8)-(12); flag-grouped sort, Eq. (13);
    computation-order mask, Eq. (14); Algorithm A (proxy stage) (causal candidates).
  * OSK, Sec. 4.3 and Algorithm A (ordered-skipping stage): ordered visits through the page
    table, running row max (Eqs. (1)-(2)), the skip rule of Eq. (5) tested against
    the updated running max, online-softmax rescaling.
  * Per-query output semantics, PageWeaver Sec. 2.1 Eqs. (1)-(2): the token set
    A_i = {t : floor(t/P) in S_i, 0 <= t < L_i, t <= c_i}; invalid IDs add no
    interaction, duplicate pages count once, empty support gives zero.

Readings taken where the pages are silent:
  * stride sampling keeps positions 0, s, 2s, ...; causality on the sampled grid is c <= r;
  * the softmax of Eq. (8) runs over the causal, valid sampled keys of the row;
    a row with no valid key contributes nothing;
  * ties in Eq. (13) are broken by ascending block index, inside each group;
  * candidates of query block i are the blocks j <= i (Algorithm A (causal candidates));
  * the stage-1 budget is a fraction: K_i = ceil(budget_ppm * J_i / 1e6), J_i = i + 1;
    with top-p, K_i is the shortest prefix of rho_i whose scores reach p of the row's total;
  * the skip threshold uses the request's own length: ln(delta / L); delta <= 0
    disables the skip (paper App. D.1: delta = -1 is the stage-1-only endpoint);
  * a row with no visible key in a visited block votes "skip" for that block;
  * mask entries < 0, > i, >= ceil(L/b), and repeats of an earlier entry are
    ignored (counted once, at the first occurrence, even if that one was skipped);
  * a token whose page-table entry is outside [0, num_pages) does not exist.
"""
from __future__ import annotations

import math
from dataclasses import dataclass
from typing import List, Optional, Sequence, Tuple

import numpy as np

COMPUTED, SKIPPED, IGNORED = 0, 1, 2


# --------------------------------------------------------------------------- #
# inputs
# --------------------------------------------------------------------------- #
def decode_bf16(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) -> float64, exactly."""
    return (np.asarray(bits).astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


@dataclass
class Params:
    block_size: int           # b
    page_size: int            # P
    stride: int               # s
    budget_ppm: int           # stage-1 fraction in parts per million
    sm_scale: float           # 1/sqrt(d)
    skip_delta: float         # Delta; <= 0 disables the in-kernel skip
    top_p: bool = False       # budget_ppm holds the top-p threshold p instead of the fraction


def request_keys(cache_bits: np.ndarray, page_table_row: np.ndarray, L: int, P: int, kv_head: int):
    """Tokens 0..L-1 of one request and kv head, resolved through the page table.

    Returns (X [L, d] float64, exists [L] bool).  Tokens on a page whose table entry is
    outside [0, num_pages) do not exist (their rows are zero and ``exists`` is False).
    """
    num_pages = cache_bits.shape[0]
    d = cache_bits.shape[-1]
    X = np.zeros((L, d), dtype=np.float64)
    exists = np.zeros(L, dtype=bool)
    for p in range(-(-L // P)):
        phys = int(page_table_row[p])
        lo, hi = p * P, min(L, (p + 1) * P)
        if 0 <= phys < num_pages:
            X[lo:hi] = decode_bf16(cache_bits[phys, : hi - lo, kv_head, :])
            exists[lo:hi] = True
    return X, exists


def request_queries(q_bits: np.ndarray, cu_seqlens: np.ndarray, b: int, h: int) -> np.ndarray:
    return decode_bf16(q_bits[int(cu_seqlens[b]):int(cu_seqlens[b + 1]), h, :])


# --------------------------------------------------------------------------- #
# PageWeaver Sec. 2.1, Eq. (1): the token set of one query
# --------------------------------------------------------------------------- #
def token_set(pages: Sequence[int], P: int, L: int, c: int) -> List[int]:
    """A = {t : floor(t/P) in S, 0 <= t < L, t <= c}, ascending.  Duplicates in S count once."""
    S = set(int(p) for p in pages)
    return [t for t in range(0, L) if (t // P) in S and t <= c]


def direct_output(q: np.ndarray, K: np.ndarray, V: np.ndarray, tokens: Sequence[int], sm_scale: float):
    """PageWeaver Eq. (2): o = sum_{t in A} exp(q.k_t * scale) v_t / sum_{t in A} exp(q.k_t * scale).

    Empty A gives the zero vector.
    """
    if len(tokens) == 0:
        return np.zeros(V.shape[1])
    idx = np.asarray(tokens)
    z = (K[idx] @ q) * sm_scale
    w = np.exp(z - z.max())
    return (w[:, None] * V[idx]).sum(axis=0) / w.sum()


# --------------------------------------------------------------------------- #
# KAP: Eqs. (8)-(14), Algorithm A (proxy stage)
# --------------------------------------------------------------------------- #
@dataclass
class KapRow:
    scores: np.ndarray        # s_ij for j = 0..i (Eq. 11)
    hrm: np.ndarray           # h_ij for j = 0..i (Eq. 12), bool
    order: np.ndarray         # rho_i (Eq. 13) over the i+1 causal candidates
    K: int                    # K_i
    pbar: np.ndarray          # Pbar rows of this query block, [rows, i+1]


def stage1_count(budget_ppm: int, J: int) -> int:
    """K_i = ceil(B * J_i) for a fractional budget B = budget_ppm / 1e6 (Eq. 14 text), in [1, J]."""
    return max(1, min(J, -(-budget_ppm * J // 1_000_000)))


def stage1_count_top_p(scores: np.ndarray, order: np.ndarray, p_ppm: int) -> int:
    """Top-p stage-1 length (Sec. 4.2 "Top-p selection", Sec. 5.1, App. D.1): the shortest prefix of
    rho_i whose scores s_ij reach p = p_ppm / 1e6 of the total over the causal candidates, summed in
    rho_i order; at least 1."""
    csum = np.cumsum(scores[order])                 # sequential, in visiting order
    thr = (p_ppm / 1e6) * csum[-1]
    return int(np.argmax(csum >= thr)) + 1


def kap_sampled(Q: np.ndarray, K: np.ndarray, exists: np.ndarray, s: int):
    """Stride downsampling (Sec. 4.2): sampled query rows and keys at positions 0, s, 2s, ..."""
    pos = np.arange(0, Q.shape[0], s)
    return pos, Q[pos], K[pos], exists[pos]


def kap_pbar_rows(Qs_rows: np.ndarray, rows_pos: np.ndarray, Ks: np.ndarray, ks_exists: np.ndarray,
                  keys_pos: np.ndarray, b: int, n_blocks: int, sm_scale: float) -> np.ndarray:
    """Pbar[r, j] for the given sampled rows (Eqs. (8)-(10)).

    Eq. (8): S_hat = Softmax(CausalMask(Q~ K~^T / sqrt(d))) over the row's causal, existing keys.
    Eq. (9): P[r, j] = max over the sampled keys of block j of S_hat[r, c].
    Eq. (10): Pbar[r, j] = P[r, j] / max_j' P[r, j'].
    """
    logits = (Qs_rows @ Ks.T) * sm_scale                                   # [rows, R]
    visible = (keys_pos[None, :] <= rows_pos[:, None]) & ks_exists[None, :]
    logits = np.where(visible, logits, -np.inf)
    row_max = logits.max(axis=1, keepdims=True)
    has_any = np.isfinite(row_max[:, 0])
    e = np.where(visible, np.exp(logits - np.where(has_any[:, None], row_max, 0.0)), 0.0)
    Z = e.sum(axis=1, keepdims=True)
    S_hat = np.where(has_any[:, None], e / np.where(Z > 0, Z, 1.0), 0.0)   # Eq. (8)
    # sampled keys are in position order, so the keys of block j are one contiguous run
    blk = keys_pos // b
    starts = np.searchsorted(blk, np.arange(n_blocks), side="left")
    ends = np.searchsorted(blk, np.arange(n_blocks), side="right")
    Pm = np.zeros((Qs_rows.shape[0], n_blocks))
    for j in range(n_blocks):                                              # Eq. (9)
        if ends[j] > starts[j]:
            Pm[:, j] = S_hat[:, starts[j]:ends[j]].max(axis=1)
    pmax = Pm.max(axis=1, keepdims=True)
    return np.where(pmax > 0, Pm / np.where(pmax > 0, pmax, 1.0), 0.0)     # Eq. (10)


def flag_grouped_order(scores: np.ndarray, hrm: np.ndarray) -> np.ndarray:
    """Eq. (13): descending argsort of the HRM group, then of the rest; ties by ascending index."""
    idx = np.arange(scores.shape[0])
    H = idx[hrm]
    R = idx[~hrm]
    H = H[np.lexsort((H, -scores[H]))]
    R = R[np.lexsort((R, -scores[R]))]
    return np.concatenate([H, R]).astype(np.int64)


def kap_request_head(Q: np.ndarray, K: np.ndarray, exists: np.ndarray, prm: Params,
                     qblocks: Optional[Sequence[int]] = None) -> dict:
    """KAP for one request and one q head.  Returns {i: KapRow} for the requested query blocks."""
    L = Q.shape[0]
    b, s = prm.block_size, prm.stride
    nqb = -(-L // b)
    pos, Qs, Ks, ks_exists = kap_sampled(Q, K, exists, s)
    rows_blk = pos // b
    out = {}
    for i in (range(nqb) if qblocks is None else qblocks):
        r_idx = np.nonzero(rows_blk == i)[0]
        J = i + 1
        pbar = kap_pbar_rows(Qs[r_idx], pos[r_idx], Ks, ks_exists, pos, b, J, prm.sm_scale)
        scores = np.zeros(J)
        for r in range(pbar.shape[0]):                                      # Eq. (11), r ascending
            scores = scores + pbar[r]
        hrm = (pbar == 1.0).any(axis=0) if pbar.shape[0] else np.zeros(J, dtype=bool)   # Eq. (12)
        order = flag_grouped_order(scores, hrm)                             # Eq. (13)
        K = stage1_count_top_p(scores, order, prm.budget_ppm) if prm.top_p else stage1_count(prm.budget_ppm, J)
        out[i] = KapRow(scores=scores, hrm=hrm, order=order, K=K, pbar=pbar)
    return out


def kap_mask(q_bits, k_bits, page_table, cu_seqlens, num_q_heads, num_kv_heads, prm: Params, kmax: int,
             heads: Optional[Sequence[int]] = None, qblocks: Optional[dict] = None, ascending: bool = False):
    """Eq. (14) for every (request, head, query block): returns (mask, mask_len, rows).

    mask [B, Hq, nqb_max, kmax] int32 (-1 padded), mask_len [B, Hq, nqb_max] int32,
    rows {(b, h, i): KapRow}.  ``qblocks`` may restrict the work to {(b, h): [i, ...]}; rows
    not computed keep mask_len 0.  ``ascending`` writes the same K_i blocks in ascending block
    order: visiting without KV page remapping, the "w/o remap" arm of Sec. 5.4 (Fig. 6) and
    App. D.4 (Fig. C).
    """
    B = len(cu_seqlens) - 1
    G = num_q_heads // num_kv_heads
    lens = np.diff(cu_seqlens)
    nqb_max = int(max(-(-int(L) // prm.block_size) for L in lens))
    mask = np.full((B, num_q_heads, nqb_max, kmax), -1, dtype=np.int32)
    mask_len = np.zeros((B, num_q_heads, nqb_max), dtype=np.int32)
    rows = {}
    for bi in range(B):
        L = int(lens[bi])
        for h in (range(num_q_heads) if heads is None else heads):
            sel = None if qblocks is None else qblocks.get((bi, h))
            if qblocks is not None and not sel:
                continue
            Q = request_queries(q_bits, cu_seqlens, bi, h)
            K, ex = request_keys(k_bits, page_table[bi], L, prm.page_size, h // G)
            for i, row in kap_request_head(Q, K, ex, prm, sel).items():
                if row.K > kmax:
                    raise ValueError("mask pitch too small")
                sel = row.order[:row.K]
                mask[bi, h, i, :row.K] = np.sort(sel) if ascending else sel
                mask_len[bi, h, i] = row.K
                rows[(bi, h, i)] = row
    return mask, mask_len, rows


# --------------------------------------------------------------------------- #
# OSK: Algorithm A (ordered-skipping stage) with the PageWeaver token-set semantics
# --------------------------------------------------------------------------- #
@dataclass
class OskResult:
    out: np.ndarray           # [rows, d] float64 (rows of the query block that exist, t < L)
    flags: np.ndarray         # per mask entry k < n: COMPUTED / SKIPPED / IGNORED
    margins: np.ndarray       # per mask entry: max_r(m_loc - m) - ln(delta/L); NaN if not tested
    row_max: np.ndarray       # final running max per row
    row_sum: np.ndarray       # final l per row


def osk_qblock(Q: np.ndarray, K: np.ndarray, V: np.ndarray, exists: np.ndarray, i: int,
               mask_row: Sequence[int], n: int, prm: Params,
               force: Optional[Sequence[int]] = None) -> OskResult:
    """Ordered-skipping sparse attention for query block i of one request and head.

    Q [L, d], K/V [L, d], exists [L]: the request's tokens (PageWeaver semantics: a token
    exists if its page does).  ``mask_row[:n]`` are the block IDs in visiting order.
    ``force`` (optional, per entry) replaces this oracle's skip decision by a given one
    (COMPUTED or SKIPPED) for entries it tests; the margin it reports is still its own.
    """
    L = Q.shape[0]
    b = prm.block_size
    nblk = -(-L // b)
    r0, r1 = i * b, min(L, (i + 1) * b)
    rows_pos = np.arange(r0, r1)
    Qi = Q[r0:r1]
    nr = r1 - r0
    m = np.full(nr, -np.inf)
    l = np.zeros(nr)
    O = np.zeros((nr, V.shape[1]))
    use_skip = prm.skip_delta > 0
    tau = math.log(prm.skip_delta / L) if use_skip else 0.0
    flags = np.full(n, IGNORED, dtype=np.int8)
    margins = np.full(n, np.nan)
    seen = set()
    for k in range(n):
        j = int(mask_row[k])
        if j < 0 or j > i or j >= nblk or j in seen:                       # invalid or repeated ID
            continue
        seen.add(j)
        c0, c1 = j * b, min(L, (j + 1) * b)                                 # "load pages via remap"
        keys_pos = np.arange(c0, c1)
        vis = (keys_pos[None, :] <= rows_pos[:, None]) & exists[c0:c1][None, :]
        S = (Qi @ K[c0:c1].T) * prm.sm_scale                                # S_ij = Q_i K_j^T / sqrt(d)
        S = np.where(vis, S, -np.inf)
        m_loc = S.max(axis=1)                                               # rowmax (Eq. 1)
        m_prev = m.copy()
        m = np.maximum(m, m_loc)                                            # Eq. (2), before the test
        if use_skip:
            has = np.isfinite(m_loc)
            diff = np.where(has, m_loc - np.where(has, m, 0.0), -np.inf)
            worst = diff.max()
            margins[k] = worst - tau
            skip = worst < tau                                              # Eq. (5)
            if force is not None:
                skip = int(force[k]) == SKIPPED
            if skip:
                flags[k] = SKIPPED
                continue
        fin = np.isfinite(m)
        m_ref = np.where(fin, m, 0.0)
        Pt = np.where(vis, np.exp(S - m_ref[:, None]), 0.0)                 # P~ = exp(S - m)
        alpha = np.where(np.isfinite(m_prev), np.exp(np.where(np.isfinite(m_prev), m_prev, 0.0) - m_ref), 0.0)
        l = alpha * l + Pt.sum(axis=1)
        O = alpha[:, None] * O + Pt @ V[c0:c1]
        flags[k] = COMPUTED
    out = np.where(l[:, None] > 0, O / np.where(l > 0, l, 1.0)[:, None], 0.0)
    return OskResult(out=out, flags=flags, margins=margins, row_max=m, row_sum=l)


def binary_mask(mask: np.ndarray, mask_len: np.ndarray, nqb_max: int) -> Tuple[np.ndarray, np.ndarray]:
    """The binary block mask M_01 of Eq. (3) (Sec. 3.2) holding the same selection as an ID-list
    mask: M01[b, h, i, j] = 1 iff block j is among the first mask_len[b, h, i] entries of row i
    and 0 <= j <= i (entries outside the causal candidates select nothing).  Returns (M01, lengths)
    with length i + 1 (every causal candidate) for rows that hold entries, else 0."""
    B, H, nqb, _ = mask.shape
    m01 = np.zeros((B, H, nqb, nqb_max), dtype=np.int32)
    len01 = np.where(mask_len > 0, np.arange(nqb, dtype=np.int32)[None, None, :] + 1, 0).astype(np.int32)
    for b in range(B):
        for h in range(H):
            for i in range(nqb):
                for k in range(int(mask_len[b, h, i])):
                    j = int(mask[b, h, i, k])
                    if 0 <= j <= i:
                        m01[b, h, i, j] = 1
    return m01, len01


def osk_qblock_binary(Q: np.ndarray, K: np.ndarray, V: np.ndarray, exists: np.ndarray, i: int,
                      m01_row: Sequence[int], n: int, prm: Params,
                      force: Optional[Sequence[int]] = None) -> OskResult:
    """Query block i driven by a binary block mask (Eq. (3)) with logical skipping, as BSA kernels
    do (Sec. 3.2, Sec. 4.3): the loop runs over blocks j = 0 .. min(n, i + 1) - 1 in ascending order
    and works on those with m01_row[j] != 0.  Flags and margins are indexed by j; unselected and
    unwalked entries are IGNORED.  ``force`` is indexed by j as well."""
    walk = min(n, i + 1)
    sel = [j for j in range(walk) if int(m01_row[j]) != 0]
    f = None if force is None else [force[j] for j in sel]
    r = osk_qblock(Q, K, V, exists, i, sel, len(sel), prm, f)
    flags = np.full(n, IGNORED, dtype=np.int8)
    margins = np.full(n, np.nan)
    for x, j in enumerate(sel):
        flags[j] = r.flags[x]
        margins[j] = r.margins[x]
    return OskResult(out=r.out, flags=flags, margins=margins, row_max=r.row_max, row_sum=r.row_sum)


def osk_all(q_bits, k_bits, v_bits, page_table, cu_seqlens, num_q_heads, num_kv_heads, prm: Params,
            mask, mask_len, items: Optional[Sequence[Tuple[int, int, int]]] = None, force=None,
            binary: bool = False):
    """OSK over (request, head, query block) items (all if ``items`` is None).

    Returns {(b, h, i): OskResult}.  ``force`` maps items to per-entry forced decisions.
    ``binary``: the mask rows are binary block masks (see osk_qblock_binary).
    """
    B = len(cu_seqlens) - 1
    G = num_q_heads // num_kv_heads
    lens = np.diff(cu_seqlens)
    if items is None:
        items = [(b, h, i) for b in range(B) for h in range(num_q_heads)
                 for i in range(-(-int(lens[b]) // prm.block_size))]
    by_req_head = {}
    for (b, h, i) in items:
        by_req_head.setdefault((b, h), []).append(i)
    res = {}
    for (b, h), blocks in by_req_head.items():
        L = int(lens[b])
        Q = request_queries(q_bits, cu_seqlens, b, h)
        K, ex = request_keys(k_bits, page_table[b], L, prm.page_size, h // G)
        V, _ = request_keys(v_bits, page_table[b], L, prm.page_size, h // G)
        for i in blocks:
            n = int(mask_len[b, h, i])
            f = None if force is None else force.get((b, h, i))
            run = osk_qblock_binary if binary else osk_qblock
            res[(b, h, i)] = run(Q, K, V, ex, i, mask[b, h, i], n, prm, f)
    return res


def query_union(sets: Sequence[Sequence[int]]) -> Tuple[List[int], np.ndarray]:
    """PageWeaver Sec. 2.2: the group's shared traversal U_G (ascending) and the membership mask
    M[i, p] = 1 if the p-th page of U_G is in S_i."""
    U = sorted(set(int(x) for S in sets for x in S))
    M = np.array([[1 if u in set(int(x) for x in S) else 0 for u in U] for S in sets], dtype=np.int8)
    return U, M


def reuse_rate(groups: Sequence[Sequence[Sequence[int]]]) -> float:
    """PageWeaver's logical page reuse rate rho_Q = sum_i |S_i| / sum_G |U_G| over groups of sets
    (duplicates within a set count once)."""
    num = sum(len(set(int(x) for x in S)) for G in groups for S in G)
    den = sum(len(query_union(G)[0]) for G in groups)
    return num / den if den else 0.0


def kept_visits(mask_row: Sequence[int], n: int, i: int, nblk: int) -> List[Tuple[int, int]]:
    """The blocks Algorithm A visits for query block i from the mask entries 0..n-1, as (k, j) pairs
    in mask order: entries with 0 <= j <= i and j < nblk, each block at its first occurrence (the
    entries osk_qblock does not flag IGNORED)."""
    seen = set()
    out = []
    for k in range(n):
        j = int(mask_row[k])
        if not (0 <= j <= i and j < nblk) or j in seen:
            continue
        seen.add(j)
        out.append((k, j))
    return out


def union_traversal(orders: Sequence[Sequence[int]]) -> List[Tuple[int, Tuple[int, ...]]]:
    """One K stream for a group of heads that each keep their own visiting order: PageWeaver Sec. 2.2
    (a shared traversal of the group's pages with a membership mask per head) applied to CoSA's ordered
    visits (Sec. 4.3).  Returns the loads in order as (block, members): the heads (indices into
    ``orders``) whose next pending block it is; each of them moves past it.  Greedy: load the block that
    is next for the most heads, ties to the lowest block ID.  Repeats inside an order count once (first
    occurrence).  Each head's blocks, read off the loads it is a member of, are its own order."""
    seqs = [list(dict.fromkeys(int(x) for x in o)) for o in orders]   # first occurrence of each ID
    pos = [0] * len(seqs)
    loads = []
    while any(p < len(q) for p, q in zip(pos, seqs)):
        cand = {}
        for p, q in zip(pos, seqs):
            if p < len(q):
                cand[q[p]] = cand.get(q[p], 0) + 1
        blk = min(cand, key=lambda b: (-cand[b], b))
        members = []
        for h, q in enumerate(seqs):
            if pos[h] < len(q) and q[pos[h]] == blk:
                members.append(h)
                pos[h] += 1
        loads.append((blk, tuple(members)))
    return loads


def ordered_shared_loads(orders: Sequence[Sequence[int]]) -> int:
    """Loads of union_traversal: an upper bound on the shortest common supersequence of the orders;
    equal to sum |S_i| when no two heads ever wait for the same block, and to |U_G| when all heads
    share one order."""
    return len(union_traversal(orders))

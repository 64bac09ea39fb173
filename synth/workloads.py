"""Seeded synthetic prefill workloads for CoSA sparse prefill.

This module only draws random numbers and lays them out; it holds none of the
method's arithmetic (no scores, no softmax, no selection).  Both the float64
oracle and the CUDA path are fed from here, so that the two see bit-identical
bf16 inputs.

Layouts (all row-major, little-endian):
  q           uint16 bf16 bits, [total_tokens, Hq, d]      packed requests (cu_seqlens)
  k_cache     uint16 bf16 bits, [num_pages, P, Hkv, d]     paged, physical order
  v_cache     uint16 bf16 bits, [num_pages, P, Hkv, d]
  page_table  int32, [num_reqs, max_pages]                 logical page -> physical page, -1 unused
  cu_seqlens  int32, [num_reqs + 1]

The structure of the keys follows the long-context workloads described for
CoSA (an attention sink on page 0, a local window of a few pages, and a set of
seeded "salient" pages per kv head whose keys are shifted toward the mean
query).  The magnitudes are this module's own choice; they are stated in the
table below and chosen so that the in-kernel skip rule has something to skip.
"""
from __future__ import annotations

import dataclasses
import math
import os
from concurrent.futures import ThreadPoolExecutor
from typing import Dict, List, Optional, Sequence

import numpy as np

__all__ = [
    "WorkloadSpec", "Workload", "WORKLOADS", "make_workload", "f32_to_bf16_bits",
    "bf16_bits_to_f32", "inject_mask_noise", "spec_for",
]


# --------------------------------------------------------------------------- #
# bf16 helpers (bit manipulation only)
# --------------------------------------------------------------------------- #
def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bf16 (round to nearest, ties to even); returns uint16 bits."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32)
    bias = ((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((u + bias) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bits to float32."""
    return (np.ascontiguousarray(b).astype(np.uint32) << np.uint32(16)).view(np.float32)


# --------------------------------------------------------------------------- #
# Workload specification
# --------------------------------------------------------------------------- #
@dataclasses.dataclass(frozen=True)
class WorkloadSpec:
    name: str
    lengths: Sequence[int]            # per-request token counts L_b
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int                   # logical block b (query and key)
    page_size: int                    # physical page P
    stride: int                       # KAP stride s
    budget_ppm: int                   # stage-1 fraction, parts per million
    stage2_budget_ppm: int            # realised-budget target the skip scale is calibrated to
    seed: int
    key_dist: str = "normal"          # "normal" or "student_t3"
    shuffle_pages: bool = False
    # structure (see module docstring); logit bumps are in nats after 1/sqrt(d)
    query_mean_norm: float = 8.0      # norm of the shared per-kv-group query direction
    sink_bump: float = 12.0           # mean logit bump of page-0 keys
    salient_pages: int = 16           # salient logical pages per kv head
    salient_bump: float = 6.0         # mean logit bump of salient keys
    local_pages: int = 4              # local window: keys less than this many pages behind
    local_bump: float = 6.0           # logit bump inside the local window
    iid_queries: bool = False         # iid Q, salient keys shifted by 4*sqrt(d) toward the mean Q
    tail_garbage_std: float = 100.0   # value std of cache slots past L (must never be read)
    mask_noise_frac: float = 0.0      # fraction of mask rows given duplicate / invalid IDs

    @property
    def num_reqs(self) -> int:
        return len(self.lengths)

    @property
    def total_tokens(self) -> int:
        return int(sum(self.lengths))

    @property
    def max_seqlen(self) -> int:
        return int(max(self.lengths))

    def pages_of(self, L: int) -> int:
        return -(-L // self.page_size)

    @property
    def max_pages(self) -> int:
        return max(self.pages_of(L) for L in self.lengths)

    @property
    def num_pages(self) -> int:
        return sum(self.pages_of(L) for L in self.lengths)

    def with_(self, **kw) -> "WorkloadSpec":
        return dataclasses.replace(self, **kw)


_GQA = dict(num_q_heads=32, num_kv_heads=8, head_dim=128, block_size=128, page_size=64, stride=16)

# The five workloads of the CoSA long-context study, shaped after Qwen3-8B attention
# (32 q heads / 8 kv heads, d = 128) at 2K-128K tokens.
WORKLOADS: Dict[str, WorkloadSpec] = {s.name: s for s in (
    WorkloadSpec(name="2k_d64_1head", lengths=(2048,), num_q_heads=1, num_kv_heads=1, head_dim=64,
                 block_size=64, page_size=64, stride=8, budget_ppm=250_000, stage2_budget_ppm=250_000,
                 seed=20261203, salient_pages=4, iid_queries=True),
    WorkloadSpec(name="8k_gqa", lengths=(8192,), budget_ppm=200_000, stage2_budget_ppm=100_000,
                 seed=20261204, **_GQA),
    WorkloadSpec(name="32k_gqa_shuffled", lengths=(32768,), budget_ppm=150_000, stage2_budget_ppm=50_000,
                 seed=20261205, shuffle_pages=True, **_GQA),
    WorkloadSpec(name="128k_gqa_student_t", lengths=(131072,), budget_ppm=100_000, stage2_budget_ppm=30_000,
                 seed=20261206, key_dist="student_t3", **_GQA),
    WorkloadSpec(name="ragged4_gqa_noisy_masks", lengths=(16384, 49152, 98304, 131072), budget_ppm=100_000,
                 stage2_budget_ppm=40_000, seed=20261207, shuffle_pages=True, mask_noise_frac=0.05, **_GQA),
    # the literal reading of "N(0,1) Q/K/V" for the GQA shapes: iid queries, the 16 salient pages per kv
    # head shifted by 4*sqrt(d) toward the unit mean query (no sink or window: with iid queries no key
    # direction raises every query's logit, and nothing ties a query to its neighbours)
    WorkloadSpec(name="32k_gqa_shuffled_iidq", lengths=(32768,), budget_ppm=150_000, stage2_budget_ppm=50_000,
                 seed=20261208, shuffle_pages=True, iid_queries=True, **_GQA),
)}


def spec_for(workload: str, **overrides) -> WorkloadSpec:
    """The named workload's spec, with fields (the name among them) replaced by ``overrides``."""
    s = WORKLOADS[workload]
    return s.with_(**overrides) if overrides else s


@dataclasses.dataclass
class Workload:
    spec: WorkloadSpec
    q: np.ndarray
    k_cache: np.ndarray
    v_cache: np.ndarray
    page_table: np.ndarray
    cu_seqlens: np.ndarray

    @property
    def lengths(self) -> List[int]:
        return [int(x) for x in np.diff(self.cu_seqlens)]


# --------------------------------------------------------------------------- #
# random draws
# --------------------------------------------------------------------------- #
def _threads() -> int:
    return max(1, min(16, os.cpu_count() or 1))


def _draw(seq: np.random.SeedSequence, n_rows: int, row_shape, dist: str, chunk_rows: int):
    """float32 draws of shape (n_rows, *row_shape), generated in parallel chunks.

    Chunk c uses child c of ``seq``; the result does not depend on the thread count.
    """
    row_elems = int(np.prod(row_shape))
    out = np.empty((n_rows, row_elems), dtype=np.float32)
    n_chunks = max(1, -(-n_rows // chunk_rows))
    children = seq.spawn(n_chunks)

    def work(c):
        lo, hi = c * chunk_rows, min(n_rows, (c + 1) * chunk_rows)
        g = np.random.Generator(np.random.PCG64(children[c]))
        if dist == "normal":
            g.standard_normal(out=out[lo:hi], dtype=np.float32)
        elif dist == "student_t3":
            # Student-t with 3 degrees of freedom, scaled to unit variance
            out[lo:hi] = (g.standard_t(3.0, size=(hi - lo, row_elems)) / math.sqrt(3.0)).astype(np.float32)
        else:
            raise ValueError(dist)

    with ThreadPoolExecutor(_threads()) as ex:
        list(ex.map(work, range(n_chunks)))
    return out.reshape((n_rows,) + tuple(row_shape))


def _unit_rows(g: np.random.Generator, n: int, d: int) -> np.ndarray:
    v = g.standard_normal((n, d))
    return (v / np.linalg.norm(v, axis=1, keepdims=True)).astype(np.float32)


# --------------------------------------------------------------------------- #
# workload construction
# --------------------------------------------------------------------------- #
def make_workload(spec: WorkloadSpec, *, with_values: bool = True) -> Workload:
    """Build the seeded workload described by ``spec``.  Deterministic in ``spec``."""
    B, Hq, Hkv, d, P = spec.num_reqs, spec.num_q_heads, spec.num_kv_heads, spec.head_dim, spec.page_size
    assert Hq % Hkv == 0
    G = Hq // Hkv
    root = np.random.SeedSequence(spec.seed)
    s_struct, s_q, s_k, s_v, s_tail, s_pages = root.spawn(6)
    gs = np.random.Generator(np.random.PCG64(s_struct))
    sqrt_d = math.sqrt(d)

    lengths = [int(L) for L in spec.lengths]
    cu = np.zeros(B + 1, dtype=np.int32)
    cu[1:] = np.cumsum(lengths)
    T = int(cu[-1])

    # shared query direction per kv group (u_g) and local-window directions
    u = _unit_rows(gs, Hkv, d)                                      # [Hkv, d]
    a_q = 0.0 if spec.iid_queries else spec.query_mean_norm

    # ---------------- Q ----------------
    qf = _draw(s_q, T, (Hq, d), "normal", chunk_rows=4096)          # [T, Hq, d] float32
    if a_q:
        qf += (a_q * u[np.arange(Hq) // G])[None, :, :]
    # local window: q(t) += a_loc * (w(seg) + w(seg-1)) / sqrt(2), k(t) += a_loc * w(seg);
    # segments of half the window, so keys in the current or previous segment get the bump
    seg_len = max(1, spec.local_pages * P // 2)
    a_loc = math.sqrt(spec.local_bump * sqrt_d * math.sqrt(2.0)) if (spec.local_bump and not spec.iid_queries) else 0.0
    local_dirs = []
    for b in range(B):
        n_seg = -(-lengths[b] // seg_len) + 1
        w = _unit_rows(gs, n_seg * Hkv, d).reshape(n_seg, Hkv, d)  # [seg, Hkv, d]
        local_dirs.append(w)
        if a_loc:
            t = np.arange(lengths[b])
            seg = t // seg_len
            wq = (w[seg] + w[np.maximum(seg - 1, 0)] * (seg >= 1)[:, None, None]) / math.sqrt(2.0)
            qf[cu[b]:cu[b + 1]] += a_loc * wq[:, np.arange(Hq) // G, :]

    q_bits = f32_to_bf16_bits(qf)
    qmean_dir = None
    if spec.iid_queries:
        # unit mean query of each kv group, from the bf16 queries themselves
        qd = bf16_bits_to_f32(q_bits).astype(np.float64)
        qmean_dir = np.zeros((Hkv, d), dtype=np.float32)
        for g in range(Hkv):
            m = qd[:, g * G:(g + 1) * G, :].reshape(-1, d).mean(axis=0)
            qmean_dir[g] = (m / np.linalg.norm(m)).astype(np.float32)
    del qf

    # ---------------- page table ----------------
    n_pages = [spec.pages_of(L) for L in lengths]
    num_pages = sum(n_pages)
    max_pages = max(n_pages)
    phys = np.arange(num_pages, dtype=np.int32)
    if spec.shuffle_pages:
        gp = np.random.Generator(np.random.PCG64(s_pages))
        phys = gp.permutation(num_pages).astype(np.int32)
    page_table = np.full((B, max_pages), -1, dtype=np.int32)
    off = 0
    for b in range(B):
        page_table[b, :n_pages[b]] = phys[off:off + n_pages[b]]
        off += n_pages[b]

    # ---------------- K / V ----------------
    k_cache = np.empty((num_pages, P, Hkv, d), dtype=np.uint16)
    v_cache = np.empty((num_pages, P, Hkv, d), dtype=np.uint16)
    k_children = s_k.spawn(B)
    v_children = s_v.spawn(B)
    t_children = s_tail.spawn(B)
    for b in range(B):
        L = lengths[b]
        npg = n_pages[b]
        Lp = npg * P
        kf = _draw(k_children[b], Lp, (Hkv, d), spec.key_dist, chunk_rows=8192)
        if spec.iid_queries:
            # keys of the salient pages shifted by 4*sqrt(d) toward the unit mean query
            sal = gs.choice(np.arange(1, npg), size=min(spec.salient_pages, npg - 1), replace=False)
            for g in range(Hkv):
                for p in sal:
                    kf[p * P:(p + 1) * P, g, :] += 4.0 * sqrt_d * qmean_dir[g]
        else:
            # attention sink: page 0 keys toward u_g
            gam_sink = spec.sink_bump * sqrt_d / a_q
            kf[0:P, :, :] += gam_sink * u[None, :, :]
            # salient pages per kv head
            gam_sal = spec.salient_bump * sqrt_d / a_q
            for g in range(Hkv):
                sal = gs.choice(np.arange(1, npg), size=min(spec.salient_pages, npg - 1), replace=False)
                for p in sal:
                    kf[p * P:(p + 1) * P, g, :] += gam_sal * u[g]
            # local window: k(t) += a_loc * w(seg(t))
            if a_loc:
                w = local_dirs[b]
                t = np.arange(Lp)
                kf += a_loc * w[t // seg_len]
        # slots past L hold garbage that the method must never read
        if Lp > L:
            gt = np.random.Generator(np.random.PCG64(t_children[b]))
            kf[L:] = (spec.tail_garbage_std * gt.standard_normal((Lp - L, Hkv, d))).astype(np.float32)
        kb = f32_to_bf16_bits(kf).reshape(npg, P, Hkv, d)
        del kf
        k_cache[page_table[b, :npg]] = kb
        del kb
        if with_values:
            vf = _draw(v_children[b], Lp, (Hkv, d), "normal", chunk_rows=8192)
            if Lp > L:
                gt = np.random.Generator(np.random.PCG64(t_children[b].spawn(1)[0]))
                vf[L:] = (spec.tail_garbage_std * gt.standard_normal((Lp - L, Hkv, d))).astype(np.float32)
            v_cache[page_table[b, :npg]] = f32_to_bf16_bits(vf).reshape(npg, P, Hkv, d)
            del vf
        else:
            v_cache[page_table[b, :npg]] = 0

    return Workload(spec=spec, q=q_bits, k_cache=k_cache, v_cache=v_cache,
                    page_table=page_table, cu_seqlens=cu)


# --------------------------------------------------------------------------- #
# mask noise (the ragged batch): duplicates and invalid IDs, injected after selection
# --------------------------------------------------------------------------- #
def inject_mask_noise(mask: np.ndarray, mask_len: np.ndarray, lengths: Sequence[int], block_size: int,
                      frac: float, seed: int, rows=None) -> tuple:
    """Return copies of (mask, mask_len) with duplicate and invalid block IDs spliced into
    a seeded ``frac`` of the rows.

    mask: int32 [B, H, nqb_max, Kmax] (-1 padded), mask_len: int32 [B, H, nqb_max].
    Each row (request b, head h, query block i < nqb_b) draws from its own generator, seeded by
    (seed, b, h, i), so a row's noise depends only on the row: it is selected with probability
    ``frac`` and then gets up to four extra entries inserted at random positions, each one of:
    a copy of an entry already in the row, -2, an ID >= ceil(L_b / b), or an ID > i.  Rows keep
    their pitch; inserted entries only use free slots past mask_len.  ``rows`` restricts the
    work to the given (b, h, i) triples (others are copied unchanged).
    """
    mask = mask.copy()
    mask_len = mask_len.copy()
    B, H, NQ, KM = mask.shape
    if rows is None:
        rows = [(b, h, i) for b in range(B) for h in range(H) for i in range(-(-int(lengths[b]) // block_size))]
    for (b, h, i) in rows:
        g = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, b, h, i])))
        if g.random() >= frac:
            continue
        nqb = -(-int(lengths[b]) // block_size)
        n = int(mask_len[b, h, i])
        room = KM - n
        if room <= 0:
            continue
        extra = []
        for _ in range(int(min(room, g.integers(1, 5)))):
            kind = int(g.integers(0, 4))
            if kind == 0 and n > 0:
                extra.append(int(mask[b, h, i, g.integers(0, n)]))
            elif kind == 1:
                extra.append(-2)
            elif kind == 2:
                extra.append(nqb + int(g.integers(0, 3)))
            else:
                extra.append(i + 1 + int(g.integers(0, 3)))
        row = list(mask[b, h, i, :n])
        for e in extra:
            row.insert(int(g.integers(0, len(row) + 1)), e)
        mask[b, h, i, :len(row)] = row
        mask_len[b, h, i] = len(row)
    return mask, mask_len

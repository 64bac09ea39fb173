"""Helpers shared by the GPU parity tests: device copies of seeded workloads, calls through
the C ABI, and comparisons against the float64 oracle."""
from __future__ import annotations

import math
import os
from dataclasses import dataclass
from typing import Dict, List, Optional, Tuple

import numpy as np
import torch

import synth
from block_sparse_long_gb300 import cosa as C
from oracle import cosa_oracle as orc

# tolerances of the output comparison (bf16 output, fp32 accumulation)
O_MAX_ABS = 2e-2
O_MEAN_ABS = 2e-3
# skip decisions: agreement rate, and the largest |margin| (nats) at which they may differ
SKIP_AGREE = 0.999
SKIP_MARGIN_TOL = 1e-3
# two oracle scores closer than this (relative) are a float64 tie: either order is valid
SCORE_TIE_RTOL = 1e-12

# The parity record: every comparison against the oracle appends an entry here, and the terminal
# summary of tests/conftest.py prints them grouped by workload (skip agreement with each
# disagreement's oracle margin, output errors, mask rows and accepted float64 ties).
PARITY_LOG: List[dict] = []


def _current_test() -> str:
    return os.environ.get("PYTEST_CURRENT_TEST", "").split(" ")[0]


def record(kind: str, workload: str, **fields) -> None:
    PARITY_LOG.append(dict(kind=kind, workload=workload, test=_current_test(), **fields))


def bf16_tensor(bits: np.ndarray, dev) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(dev).view(torch.bfloat16)


def i32_tensor(x: np.ndarray, dev) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.int32)).to(dev)


@dataclass
class DevWorkload:
    w: synth.Workload
    q: torch.Tensor
    k: torch.Tensor
    v: torch.Tensor
    pt: torch.Tensor
    cu: torch.Tensor


def to_device(w: synth.Workload, dev="cuda") -> DevWorkload:
    return DevWorkload(w, bf16_tensor(w.q, dev), bf16_tensor(w.k_cache, dev), bf16_tensor(w.v_cache, dev),
                       i32_tensor(w.page_table, dev), i32_tensor(w.cu_seqlens, dev))


def oracle_params(spec, delta: float, budget_ppm: Optional[int] = None) -> orc.Params:
    return orc.Params(spec.block_size, spec.page_size, spec.stride,
                      spec.budget_ppm if budget_ppm is None else budget_ppm, 1.0 / math.sqrt(spec.head_dim),
                      float(delta))


def cosa_params(dw: DevWorkload, *, delta: float, mask_pitch: int, budget_ppm: Optional[int] = None):
    sp = dw.w.spec
    return C.params_for(dw.q, dw.k, dw.pt, dw.cu, block_size=sp.block_size, max_seqlen=sp.max_seqlen,
                        stride=sp.stride, budget_ppm=sp.budget_ppm if budget_ppm is None else budget_ppm,
                        mask_pitch=mask_pitch, skip_delta=delta)


def binary_of(mask: np.ndarray, mask_len: np.ndarray) -> Tuple[np.ndarray, np.ndarray]:
    """Binary block masks (entry j = 1 iff block j is listed, 0 <= j <= i) of ID-list masks, with
    walk length i + 1 on rows that list something (vectorised form of the oracle's binary_mask)."""
    B, H, nqb, pitch = mask.shape
    i_idx = np.arange(nqb)[None, None, :, None]
    k_idx = np.arange(pitch)[None, None, None, :]
    ok = (k_idx < mask_len[..., None]) & (mask >= 0) & (mask <= i_idx)
    m01 = np.zeros((B, H, nqb, nqb + 1), dtype=np.int32)
    bb, hh, ii, kk = np.nonzero(ok)
    m01[bb, hh, ii, mask[bb, hh, ii, kk]] = 1
    len01 = np.where(mask_len > 0, np.arange(nqb, dtype=np.int32)[None, None, :] + 1, 0).astype(np.int32)
    return m01[..., :nqb], len01


def ascending_of(m01: np.ndarray, len01: np.ndarray) -> Tuple[np.ndarray, np.ndarray]:
    """ID lists of the selected blocks in ascending order (the visits a binary mask walk makes)."""
    B, H, nqb, _ = m01.shape
    ids = np.full((B, H, nqb, nqb), -1, dtype=np.int32)
    lens = np.zeros((B, H, nqb), dtype=np.int32)
    for b in range(B):
        for h in range(H):
            for i in range(nqb):
                sel = np.nonzero(m01[b, h, i, :len01[b, h, i]])[0]
                ids[b, h, i, :len(sel)] = sel
                lens[b, h, i] = len(sel)
    return ids, lens


def run_kap(dw: DevWorkload, p) -> Tuple[np.ndarray, np.ndarray]:
    status = torch.zeros(1, dtype=torch.int32, device=dw.q.device)
    mask, mask_len = C.cosa_proxy_select(p, dw.q, dw.cu, dw.k, dw.pt, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0, C.cosa_status_string(int(status.item()))
    return mask.cpu().numpy(), mask_len.cpu().numpy()


def run_osk(dw: DevWorkload, p, mask: np.ndarray, mask_len: np.ndarray) -> Tuple[np.ndarray, np.ndarray]:
    dev = dw.q.device
    m = i32_tensor(mask, dev)
    ml = i32_tensor(mask_len, dev)
    flags = torch.full(mask.shape, 255, dtype=torch.uint8, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    out = torch.full_like(dw.q, float("nan"))
    C.cosa_sparse_prefill(p, dw.q, dw.cu, dw.k, dw.v, dw.pt, m, ml, out=out, visit_flags=flags, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0, C.cosa_status_string(int(status.item()))
    return out.float().cpu().numpy(), flags.cpu().numpy()


def items_of(spec, heads=None, qblocks=None) -> List[Tuple[int, int, int]]:
    out = []
    for b, L in enumerate(spec.lengths):
        nqb = -(-L // spec.block_size)
        for h in (range(spec.num_q_heads) if heads is None else heads):
            for i in (range(nqb) if qblocks is None else [x for x in qblocks if x < nqb]):
                out.append((b, h, i))
    return out


@dataclass
class OskReport:
    n_items: int
    n_tested: int
    n_disagree: int
    max_disagree_margin: float
    max_abs: float
    mean_abs: float
    disagreements: list


def compare_osk(w: synth.Workload, prm: orc.Params, mask, mask_len, out_gpu, flags_gpu,
                items, binary: bool = False) -> OskReport:
    """Oracle vs GPU on the given items.  Skip decisions may differ only near a zero margin;
    the oracle is then replayed with the GPU's decisions so outputs compare like for like.
    ``binary``: the masks are binary block masks (COSA_FLAG_BINARY_MASK)."""
    sp = w.spec
    ref = orc.osk_all(w.q, w.k_cache, w.v_cache, w.page_table, w.cu_seqlens, sp.num_q_heads, sp.num_kv_heads,
                      prm, mask, mask_len, items=items, binary=binary)
    n_tested = 0
    dis = []
    force = {}
    for it, r in ref.items():
        b, h, i = it
        n = int(mask_len[b, h, i])
        g = flags_gpu[b, h, i, :n]
        assert ((g == orc.IGNORED) == (r.flags == orc.IGNORED)).all(), f"ignored entries differ at {it}"
        tested = r.flags != orc.IGNORED
        n_tested += int(tested.sum())
        bad = np.nonzero(tested & (g != r.flags))[0]
        for k in bad:
            dis.append((it, int(k), float(r.margins[k])))
        if len(bad):
            force[it] = g.astype(np.int8)
        # entries past mask_len are reported ignored
        assert (flags_gpu[b, h, i, n:] == orc.IGNORED).all()
    if force:
        ref.update(orc.osk_all(w.q, w.k_cache, w.v_cache, w.page_table, w.cu_seqlens, sp.num_q_heads,
                               sp.num_kv_heads, prm, mask, mask_len, items=list(force), force=force,
                               binary=binary))
    errs = []
    cu = w.cu_seqlens
    for (b, h, i), r in ref.items():
        t0 = int(cu[b]) + i * sp.block_size
        got = out_gpu[t0:t0 + r.out.shape[0], h, :]
        errs.append(np.abs(got - r.out).ravel())
    e = np.concatenate(errs) if errs else np.zeros(1)
    rep = OskReport(len(ref), n_tested, len(dis), max([abs(x[2]) for x in dis], default=0.0),
                    float(e.max()), float(e.mean()), dis)
    record("osk", sp.name, items=rep.n_items, tested=rep.n_tested, disagree=rep.n_disagree,
           disagreements=list(dis), max_abs=rep.max_abs, mean_abs=rep.mean_abs, binary=binary)
    return rep


def assert_osk_ok(rep: OskReport):
    assert np.isfinite(rep.max_abs)
    assert rep.max_abs <= O_MAX_ABS, rep
    assert rep.mean_abs <= O_MEAN_ABS, rep
    if rep.n_tested:
        assert 1.0 - rep.n_disagree / rep.n_tested >= SKIP_AGREE, rep
    assert rep.max_disagree_margin <= SKIP_MARGIN_TOL, rep


# top-p: the kernel certifies the cut (or takes it from exact scores); a length that differs from the
# oracle's is accepted only at a float64 tie: the oracle's prefix mass within this fraction of the total
# from p times the total
TOP_P_RTOL = 1e-12


def compare_masks_top_p(mask_gpu, len_gpu, rows: Dict, p_ppm: int, workload: str = "") -> Tuple[List, List]:
    """Top-p masks: the GPU row must be a prefix of the oracle's rho_i (float64 ties accepted as in
    compare_masks) whose length is the oracle's K_i, except at a float64 tie of the cut (oracle prefix
    mass within TOP_P_RTOL * total of p * total).  Returns (accepted cut differences, accepted ties)."""
    cuts, ties = [], []
    p = p_ppm / 1e6
    for key, row in rows.items():
        b, h, i = key
        kg, ko = int(len_gpu[b, h, i]), row.K
        assert 1 <= kg <= i + 1, (key, kg)
        if kg != ko:
            csum = np.cumsum(row.scores[row.order])
            T = csum[-1]
            for k in range(min(kg, ko), max(kg, ko)):
                assert abs(csum[k - 1] - p * T) <= TOP_P_RTOL * T, (key, kg, ko, k, csum[k - 1] / T)
            cuts.append((key, kg, ko))
        sub = type(row)(scores=row.scores, hrm=row.hrm, order=row.order, K=kg, pbar=row.pbar)
        ties += _compare_mask_rows(mask_gpu, len_gpu, {key: sub})
    record("top_p", workload, rows=len(rows), p_ppm=p_ppm, cuts=list(cuts), ties=len(ties))
    return cuts, ties


def compare_masks_rows(mask_gpu, len_gpu, rows: Dict, workload: str = "") -> List:
    """compare_masks restricted to the oracle's rows (no check of absent query blocks)."""
    return compare_masks(mask_gpu, len_gpu, rows, None, None, workload=workload)


def compare_masks(mask_gpu, len_gpu, rows: Dict, lengths, block_size, workload: str = "") -> List:
    """Bit-exact comparison of M_KAP rows; a difference is accepted only between blocks whose
    oracle keys (HRM flag, score) are equal within a float64 tie.  Returns accepted ties;
    raises on a real mismatch."""
    ties = _compare_mask_rows(mask_gpu, len_gpu, rows)
    # absent query blocks
    for b, L in enumerate(lengths or []):
        nqb = -(-L // block_size)
        assert (len_gpu[b, :, nqb:] == 0).all()
        assert (mask_gpu[b, :, nqb:, :] == -1).all()
    record("mask", workload, rows=len(rows), entries=int(sum(r.K for r in rows.values())), ties=list(ties))
    return ties


def _compare_mask_rows(mask_gpu, len_gpu, rows: Dict) -> List:
    ties = []
    for (b, h, i), row in rows.items():
        K = row.K
        assert int(len_gpu[b, h, i]) == K, ((b, h, i), int(len_gpu[b, h, i]), K)
        g = mask_gpu[b, h, i, :K]
        o = row.order[:K]
        if np.array_equal(g, o):
            assert (mask_gpu[b, h, i, K:] == -1).all()
            continue
        # accept only float64 ties: same multiset of keys position by position
        sc = row.scores
        for p in range(K):
            if g[p] == o[p]:
                continue
            a, c = int(g[p]), int(o[p])
            assert 0 <= a <= i, ((b, h, i), p, a)
            same_flag = bool(row.hrm[a]) == bool(row.hrm[c])
            tie = abs(sc[a] - sc[c]) <= SCORE_TIE_RTOL * max(abs(sc[a]), abs(sc[c]), 1e-300)
            assert same_flag and tie, f"mask mismatch at {(b, h, i)} pos {p}: gpu {a} ({sc[a]!r}, hrm {row.hrm[a]}) " \
                                      f"oracle {c} ({sc[c]!r}, hrm {row.hrm[c]})"
            ties.append(((b, h, i), p, a, c, float(sc[a]), float(sc[c])))
        assert len(set(g.tolist())) == K
        assert (mask_gpu[b, h, i, K:] == -1).all()
    return ties


# --------------------------------------------------------------------------- #
# the parity record, as printed after the test run
# --------------------------------------------------------------------------- #
def parity_summary_lines() -> List[str]:
    """One line per workload (masks, top-p cuts, skip decisions, outputs), the named workloads of
    synth.WORKLOADS last in registry order, each skip disagreement on its own line with its oracle
    margin, and the tensor-core error bound at the end."""
    by = {}
    for e in PARITY_LOG:
        by.setdefault(e["workload"] or "?", []).append(e)
    named = [n for n in synth.WORKLOADS if n in by]
    others = [n for n in by if n not in synth.WORKLOADS and n != "tensor-core logits"]
    lines = []
    small = [e for n in others for e in by[n]]
    if small:
        lines += _summary_of(f"small and edge cases ({len(others)} shapes)", small)
    for n in named:
        lines += _summary_of(n, by[n])
    kap = [e for e in by.get("tensor-core logits", []) if e["kind"] == "kappa"]
    ex2 = [e for e in by.get("tensor-core logits", []) if e["kind"] == "ex2"]
    if kap:
        wn = max(kap, key=lambda e: e["r_norm"])
        wa = max(kap, key=lambda e: e["r_abs"])
        lines.append(f"kappa bound: {len(kap)} cases, {sum(e['logits'] for e in kap)} tensor-core logits; worst "
                     f"|err|/(|q||k|) {wn['r_norm'] / 2.0 ** -24:.2f}*2^-24 ({wn['case']}; limit 32*2^-24), worst "
                     f"|err|/sum|q_i k_i| {wa['r_abs'] / 2.0 ** -24:.2f}*2^-24 ({wa['case']}; model 48*2^-24)")
    for e in ex2:
        lines.append(f"ex2.approx: {e['inputs']} fp32 inputs, worst relative error {e['rel'] / 2.0 ** -24:.2f}*2^-24 "
                     f"at x = {e['arg']!r} (block scores assume 8*2^-24)")
    return lines


def _summary_of(name: str, es: List[dict]) -> List[str]:
    parts, extra = [], []
    ms = [e for e in es if e["kind"] == "mask"]
    if ms:
        ties = sum(len(e["ties"]) for e in ms)
        parts.append(f"masks {sum(e['rows'] for e in ms)} rows / {sum(e['entries'] for e in ms)} entries exact "
                     f"({ties} float64 ties)")
    tp = [e for e in es if e["kind"] == "top_p"]
    if tp:
        cuts = [c for e in tp for c in e["cuts"]]
        parts.append(f"top-p {sum(e['rows'] for e in tp)} rows, {len(cuts)} cuts differ")
    os_ = [e for e in es if e["kind"] == "osk"]
    if os_:
        tested = sum(e["tested"] for e in os_)
        dis = [d for e in os_ for d in e["disagreements"]]
        agree = 100.0 * (1.0 - len(dis) / tested) if tested else 100.0
        parts.append(f"skip {tested} visits of {sum(e['items'] for e in os_)} items, {len(dis)} disagree "
                     f"({agree:.3f}% agree); O max-abs {max(e['max_abs'] for e in os_):.1e} mean-abs "
                     f"{max(e['mean_abs'] for e in os_):.1e}")
        extra = [f"    disagreement {name} item {it} entry {k}: oracle margin {m:+.3e} nats" for (it, k, m) in dis]
    return [f"{name}: " + "; ".join(parts)] + extra

"""The GQA page-union variant of the OSK (COSA_FLAG_GQA_UNION; PageWeaver notes Sec. 2.2 applied to
CoSA's ordered visits, Sec. 4.3): two query heads of a kv group share one stream of K tiles while each
keeps its own order, running maximum and skip vote.

Checked through the C ABI against
  * the default kernel on the same masks: outputs and visit decisions bit for bit (the per-head
    arithmetic is the same),
  * the oracle's union traversal: exactly the entries whose K tile the oracle's greedy merge loads
    once for both heads carry COSA_VISIT_SHARED_LOAD,
  * the float64 oracle (Algorithm A per head) on the outputs and skip decisions."""
import json
import os

import numpy as np
import pytest
import torch

import synth
from oracle import cosa_oracle as orc
from tests import gpu_helpers as gh
from tests.test_gpu_full import sampled_items

pytestmark = pytest.mark.gpu

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "delta_calibration.json")

SMALL = {
    # (q heads, kv heads): 2 pairs per group, an odd group (a head alone), one head per group
    "d128_P64_g4": dict(head_dim=128, page_size=64, heads=(8, 2), lengths=(1000, 300, 129, 1)),
    "d128_P32_g3": dict(head_dim=128, page_size=32, heads=(6, 2), lengths=(1100, 257)),
    "d64_P16_g2": dict(head_dim=64, page_size=16, heads=(4, 2), lengths=(1300, 200)),
    "d128_P128_g1": dict(head_dim=128, page_size=128, heads=(2, 2), lengths=(700, 128)),
}


def small_spec(name, seed):
    c = SMALL[name]
    return synth.WorkloadSpec(name=name, lengths=c["lengths"], num_q_heads=c["heads"][0],
                              num_kv_heads=c["heads"][1], head_dim=c["head_dim"], block_size=128,
                              page_size=c["page_size"], stride=16, budget_ppm=400_000, stage2_budget_ppm=0,
                              seed=seed, shuffle_pages=True, salient_pages=3)


def run_union(dw, p, mask, mask_len):
    p.flags |= gh.C.COSA_FLAG_GQA_UNION
    try:
        return gh.run_osk(dw, p, mask, mask_len)
    finally:
        p.flags &= ~gh.C.COSA_FLAG_GQA_UNION


def run_osk_bits(dw, p, mask, mask_len, union):
    """Output as raw bf16 bits (for a bitwise comparison) and the visit flags."""
    dev = dw.q.device
    m, ml = gh.i32_tensor(mask, dev), gh.i32_tensor(mask_len, dev)
    flags = torch.full(mask.shape, 255, dtype=torch.uint8, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    out = torch.full_like(dw.q, float("nan"))
    if union:
        p.flags |= gh.C.COSA_FLAG_GQA_UNION
    try:
        gh.C.cosa_sparse_prefill(p, dw.q, dw.cu, dw.k, dw.v, dw.pt, m, ml, out=out, visit_flags=flags,
                                 status=status)
        torch.cuda.synchronize()
    finally:
        p.flags &= ~gh.C.COSA_FLAG_GQA_UNION
    assert int(status.item()) == 0, gh.C.cosa_status_string(int(status.item()))
    return out.view(torch.int16).cpu().numpy(), flags.cpu().numpy()


def pairs_of(spec):
    """The head pairs the union kernel serves: heads 2x and 2x + 1 of each kv group (the group's last
    head alone when the group has an odd number of heads)."""
    G = spec.num_q_heads // spec.num_kv_heads
    out = []
    for kvh in range(spec.num_kv_heads):
        for pr in range((G + 1) // 2):
            h0 = kvh * G + 2 * pr
            out.append([h0] + ([h0 + 1] if 2 * pr + 1 < G else []))
    return out


def expected_shared(spec, mask, mask_len, rows=None):
    """COSA_VISIT_SHARED_LOAD per mask entry from the oracle: the kept visits of a pair's heads
    (Algorithm A's filter) merged by the oracle's union traversal; an entry is shared when its load
    serves both heads.  ``rows``: the (b, h, i) whose pairs are evaluated (all if None)."""
    G = spec.num_q_heads // spec.num_kv_heads
    shared = np.zeros(mask.shape, dtype=bool)
    want = None if rows is None else {(b, (h // G) * G + ((h % G) // 2) * 2, i) for (b, h, i) in rows}
    for b, L in enumerate(spec.lengths):
        nblk = -(-L // spec.block_size)
        for heads in pairs_of(spec):
            for i in range(nblk):
                if want is not None and (b, heads[0], i) not in want:
                    continue
                kept = [orc.kept_visits(mask[b, h, i], int(mask_len[b, h, i]), i, nblk) for h in heads]
                loads = orc.union_traversal([[j for _, j in kv] for kv in kept])
                cur = [0] * len(heads)
                for _, members in loads:
                    for x in members:
                        if len(members) > 1:
                            shared[b, heads[x], i, kept[x][cur[x]][0]] = True
                        cur[x] += 1
    return shared


def check_against_default(spec, dw, p, mask, ml, rows=None):
    """Union kernel vs the default kernel (bitwise) and vs the oracle's shared-load entries."""
    o_ref, f_ref = run_osk_bits(dw, p, mask, ml, union=False)
    o_uni, f_uni = run_osk_bits(dw, p, mask, ml, union=True)
    # entries of absent query blocks are never written (255 in both)
    assert np.array_equal(np.where(f_uni == 255, 255, f_uni & 3), f_ref), "visit decisions differ from the default kernel"
    assert np.array_equal(o_uni, o_ref), "outputs differ from the default kernel"
    sh = expected_shared(spec, mask, ml, rows)
    got = (f_uni != 255) & ((f_uni & gh.C.VISIT_SHARED_LOAD) != 0)
    if rows is None:
        assert np.array_equal(got, sh), "shared loads differ from the oracle's union traversal"
    else:
        for (b, h, i) in rows:
            assert np.array_equal(got[b, h, i], sh[b, h, i]), ((b, h, i), np.nonzero(got[b, h, i] != sh[b, h, i]))
    return f_uni, got


@pytest.mark.parametrize("name", sorted(SMALL))
@pytest.mark.parametrize("delta", [-1.0, 40.0])
def test_union_small_edge_cases(name, delta):
    sp = small_spec(name, seed=300 + len(name))
    w = synth.make_workload(sp)
    w.page_table[0, 1] = -1                   # missing pages
    w.page_table[0, 3] = sp.num_pages + 7
    prm = gh.oracle_params(sp, delta)
    pitch = gh.C.stage1_pitch(sp.budget_ppm, sp.max_seqlen, sp.block_size) + 6
    mask, ml, _ = orc.kap_mask(w.q, w.k_cache, w.page_table, w.cu_seqlens, sp.num_q_heads, sp.num_kv_heads,
                               prm, pitch)
    mask, ml = synth.inject_mask_noise(mask, ml, sp.lengths, sp.block_size, 0.3, 7)
    dw = gh.to_device(w)
    p = gh.cosa_params(dw, delta=delta, mask_pitch=pitch)
    f_uni, shared = check_against_default(sp, dw, p, mask, ml)
    if sp.num_q_heads > sp.num_kv_heads:
        assert shared.any()
    out, flags = run_union(dw, p, mask, ml)
    rep = gh.compare_osk(w, prm, mask, ml, out, flags & 3, gh.items_of(sp))
    gh.assert_osk_ok(rep)


def test_union_identical_and_disjoint_rows():
    """Both heads of a pair with the same row (every load shared), with disjoint rows (none shared), and
    with one head's row empty."""
    sp = small_spec("d128_P64_g4", seed=77)
    w = synth.make_workload(sp)
    nqb = -(-sp.max_seqlen // sp.block_size)
    pitch = nqb
    mask = np.full((sp.num_reqs, sp.num_q_heads, nqb, pitch), -1, np.int32)
    ml = np.zeros((sp.num_reqs, sp.num_q_heads, nqb), np.int32)
    rng = np.random.default_rng(3)
    for b, L in enumerate(sp.lengths):
        for i in range(-(-L // sp.block_size)):
            perm = rng.permutation(i + 1)
            mask[b, 0, i, :i + 1] = perm                       # heads 0 and 1: identical rows
            mask[b, 1, i, :i + 1] = perm
            ml[b, 0, i] = ml[b, 1, i] = i + 1
            even, odd = perm[perm % 2 == 0], perm[perm % 2 == 1]
            mask[b, 2, i, :len(even)] = even                    # heads 2 and 3: disjoint rows
            mask[b, 3, i, :len(odd)] = odd
            ml[b, 2, i], ml[b, 3, i] = len(even), len(odd)
            mask[b, 4, i, :i + 1] = perm                        # head 5: empty rows
            ml[b, 4, i] = i + 1
    dw = gh.to_device(w)
    for delta in (-1.0, 40.0):
        p = gh.cosa_params(dw, delta=delta, mask_pitch=pitch)
        _, shared = check_against_default(sp, dw, p, mask, ml)
        for b in range(sp.num_reqs):
            valid = np.arange(pitch)[None, :] < ml[b, 0][:, None]
            assert (shared[b, 0] == valid).all() and (shared[b, 1] == valid).all()
            assert not shared[b, 2:6].any()
        prm = gh.oracle_params(sp, delta)
        out, flags = run_union(dw, p, mask, ml)
        rep = gh.compare_osk(w, prm, mask, ml, out, flags & 3, gh.items_of(sp, heads=[0, 1, 2, 3, 4, 5]))
        gh.assert_osk_ok(rep)
        assert (out[:, 5, :] == 0).all()


@pytest.mark.parametrize("name,n_items,seed", [("32k_gqa_shuffled", 32, 13), ("128k_gqa_student_t", 32, 14),
                                               ("ragged4_gqa_noisy_masks", 32, 15)])
def test_union_full_size(name, n_items, seed):
    """At full size, in the bench's launch configuration: KAP masks from the GPU, the union kernel
    against the default kernel on every item (bitwise) and against the oracle on sampled items."""
    sp = synth.spec_for(name)
    delta = json.load(open(GOLDEN))["workloads"][name]["delta"]
    w = synth.make_workload(sp)
    prm = gh.oracle_params(sp, delta)
    pitch = gh.C.stage1_pitch(sp.budget_ppm, sp.max_seqlen, sp.block_size) + (4 if sp.mask_noise_frac else 0)
    dw = gh.to_device(w)
    p = gh.cosa_params(dw, delta=delta, mask_pitch=pitch)
    mask, ml = gh.run_kap(dw, p)
    if sp.mask_noise_frac:
        mask, ml = synth.inject_mask_noise(mask, ml, sp.lengths, sp.block_size, sp.mask_noise_frac, seed=sp.seed)
    items = sampled_items(sp, n_items, seed)
    _, shared = check_against_default(sp, dw, p, mask, ml, rows=items)
    assert shared.any()
    out, flags = run_union(dw, p, mask, ml)
    rep = gh.compare_osk(w, prm, mask, ml, out, flags & 3, items)
    gh.assert_osk_ok(rep)

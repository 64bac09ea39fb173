"""The two ablation switches on the GPU against the float64 oracle.

COSA_FLAG_ASCENDING_ORDER (cosa_proxy_select): the same K_i blocks as the computation-order mask
of Eq. (14), written in ascending block order, i.e. visiting without KV page remapping (CoSA
Sec. 5.4, Fig. 6; App. D.4, Fig. C).  COSA_FLAG_BINARY_MASK (cosa_sparse_prefill): the mask rows
are binary block masks M_01 (Eq. (3), Sec. 3.2) walked block by block in ascending order with
logical skipping, as BSA kernels do (App. D.3, Fig. B)."""
import json
import os

import numpy as np
import pytest

import synth
from oracle import cosa_oracle as orc
from tests import gpu_helpers as gh
from tests.test_gpu_osk import SMALL, small_spec

pytestmark = pytest.mark.gpu

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "delta_calibration.json")


def _kap_both(dw, ppm, pitch):
    p = gh.cosa_params(dw, delta=-1.0, mask_pitch=pitch, budget_ppm=ppm)
    m0, l0 = gh.run_kap(dw, p)
    p.flags = gh.C.COSA_FLAG_ASCENDING_ORDER
    m1, l1 = gh.run_kap(dw, p)
    return m0, l0, m1, l1


def _assert_sorted_copy(m0, l0, m1, l1):
    """Ascending rows hold exactly the computation-order rows' blocks, sorted, with -1 tails."""
    assert np.array_equal(l0, l1)
    pitch = m0.shape[-1]
    live = np.arange(pitch)[None, None, None, :] < l0[..., None]
    s0 = np.sort(np.where(live, m0, np.iinfo(np.int32).max), axis=-1)
    assert np.array_equal(np.where(live, s0, -1), m1)


@pytest.mark.parametrize("name", sorted(SMALL))
@pytest.mark.parametrize("ppm", [400_000, 1_000_000])
def test_kap_ascending_small(name, ppm):
    if SMALL[name]["block_size"] // SMALL[name]["stride"] not in (4, 8, 16):
        pytest.skip("stride ratio not supported")
    sp = small_spec(name, seed=400 + len(name))
    w = synth.make_workload(sp)
    dw = gh.to_device(w)
    pitch = gh.C.stage1_pitch(ppm, sp.max_seqlen, sp.block_size)
    m0, l0, m1, l1 = _kap_both(dw, ppm, pitch)
    _assert_sorted_copy(m0, l0, m1, l1)
    prm = gh.oracle_params(sp, -1.0, budget_ppm=ppm)
    mo, lo, rows = orc.kap_mask(w.q, w.k_cache, w.page_table, w.cu_seqlens, sp.num_q_heads, sp.num_kv_heads,
                                prm, pitch, ascending=True)
    ties = gh.compare_masks(m0, l0, rows, sp.lengths, sp.block_size, workload=sp.name)
    if not ties:
        assert np.array_equal(m1, mo) and np.array_equal(l1, lo)


def test_kap_ascending_32k_all_rows():
    """32K tokens, 32 heads: every row of the ascending mask is the sorted computation-order row."""
    sp = synth.spec_for("32k_gqa_shuffled")
    w = synth.make_workload(sp)
    dw = gh.to_device(w)
    pitch = gh.C.stage1_pitch(sp.budget_ppm, sp.max_seqlen, sp.block_size)
    _assert_sorted_copy(*_kap_both(dw, sp.budget_ppm, pitch))


@pytest.mark.parametrize("name", sorted(SMALL))
@pytest.mark.parametrize("delta", [-1.0, 40.0])
def test_osk_binary_small(name, delta):
    sp = small_spec(name, seed=500 + len(name))
    w = synth.make_workload(sp)
    w.page_table[0, 1] = -1
    prm = gh.oracle_params(sp, delta)
    pitch = gh.C.stage1_pitch(sp.budget_ppm, sp.max_seqlen, sp.block_size)
    mask, ml, _ = orc.kap_mask(w.q, w.k_cache, w.page_table, w.cu_seqlens, sp.num_q_heads, sp.num_kv_heads,
                               prm, pitch)
    m01, l01 = gh.binary_of(mask, ml)
    dw = gh.to_device(w)
    p = gh.cosa_params(dw, delta=delta, mask_pitch=m01.shape[-1])
    p.flags = gh.C.COSA_FLAG_BINARY_MASK
    out_b, flags_b = gh.run_osk(dw, p, m01, l01)
    rep = gh.compare_osk(w, prm, m01, l01, out_b, flags_b, gh.items_of(sp), binary=True)
    gh.assert_osk_ok(rep)
    # the same kernel on the ascending ID lists makes the same visits: identical bits
    ids, lens = gh.ascending_of(m01, l01)
    p2 = gh.cosa_params(dw, delta=delta, mask_pitch=ids.shape[-1])
    out_a, flags_a = gh.run_osk(dw, p2, ids, lens)
    assert np.array_equal(out_a, out_b)
    _assert_flags_map(flags_b, l01, flags_a, ids, lens)


def _assert_flags_map(flags_b, l01, flags_a, ids, lens):
    B, H, nqb = lens.shape
    for b in range(B):
        for h in range(H):
            for i in range(nqb):
                if l01[b, h, i] == 0:
                    continue          # query block absent from the request: not an item
                n = int(lens[b, h, i])
                sel = ids[b, h, i, :n]
                fb = flags_b[b, h, i]
                assert np.array_equal(fb[sel], flags_a[b, h, i, :n])
                rest = np.ones(fb.shape[0], bool)
                rest[sel] = False
                assert (fb[rest] == orc.IGNORED).all()


def test_osk_binary_32k_sampled():
    """32K tokens, 32 heads, calibrated Delta: binary-mask visiting against the oracle on sampled
    rows, and bit-identical to the ascending ID lists on every row."""
    from tests.test_gpu_full import sampled_items
    sp = synth.spec_for("32k_gqa_shuffled")
    delta = json.load(open(GOLDEN))["workloads"]["32k_gqa_shuffled"]["delta"]
    w = synth.make_workload(sp)
    dw = gh.to_device(w)
    pitch = gh.C.stage1_pitch(sp.budget_ppm, sp.max_seqlen, sp.block_size)
    p = gh.cosa_params(dw, delta=delta, mask_pitch=pitch)
    p.flags = gh.C.COSA_FLAG_ASCENDING_ORDER
    ids, lens = gh.run_kap(dw, p)
    m01, l01 = gh.binary_of(ids, lens)
    pb = gh.cosa_params(dw, delta=delta, mask_pitch=m01.shape[-1])
    pb.flags = gh.C.COSA_FLAG_BINARY_MASK
    out_b, flags_b = gh.run_osk(dw, pb, m01, l01)
    p.flags = 0
    out_a, flags_a = gh.run_osk(dw, p, ids, lens)
    assert np.array_equal(out_a, out_b)
    _assert_flags_map(flags_b, l01, flags_a, ids, lens)
    items = sampled_items(sp, 6, seed=77)
    rep = gh.compare_osk(w, gh.oracle_params(sp, delta), m01, l01, out_b, flags_b, items, binary=True)
    gh.assert_osk_ok(rep)

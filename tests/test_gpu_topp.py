"""Top-p stage-1 budget (COSA_FLAG_TOP_P) on the GPU against the float64 oracle: K_i is the shortest
prefix of rho_i (Eq. (13)) whose block scores (Eq. (11)) reach p of the row's total (CoSA Sec. 4.2,
Sec. 5.1 and App. D.1, p = 0.95).  The order is exact as for the fraction rule, and so is the cut: the
kernel certifies it from the scores' error bounds, or takes it from exact scores of every candidate when
the bounds straddle p times the total; a length may differ from the oracle's only at a float64 tie."""
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


def _run(w, ppm, delta=-1.0, items=None):
    sp = w.spec
    nqb = -(-sp.max_seqlen // sp.block_size)
    dw = gh.to_device(w)
    p = gh.cosa_params(dw, delta=delta, mask_pitch=nqb, budget_ppm=ppm)
    p.flags = gh.C.COSA_FLAG_TOP_P
    mask_g, len_g = gh.run_kap(dw, p)
    prm = gh.oracle_params(sp, delta, budget_ppm=ppm)
    prm.top_p = True
    by = None
    if items is not None:
        by = {}
        for (b, h, i) in items:
            by.setdefault((b, h), []).append(i)
    _, len_o, rows = orc.kap_mask(w.q, w.k_cache, w.page_table, w.cu_seqlens, sp.num_q_heads, sp.num_kv_heads,
                                  prm, nqb, qblocks=by)
    cuts, ties = gh.compare_masks_top_p(mask_g, len_g, rows, ppm, workload=sp.name)
    return dw, p, prm, mask_g, len_g, rows, cuts


@pytest.mark.parametrize("name", sorted(SMALL))
@pytest.mark.parametrize("ppm", [500_000, 950_000, 990_000])
def test_top_p_small(name, ppm):
    if SMALL[name]["block_size"] // SMALL[name]["stride"] not in (4, 8, 16):
        pytest.skip("stride ratio not supported")
    w = synth.make_workload(small_spec(name, seed=600 + len(name)))
    _, _, _, mask_g, len_g, rows, cuts = _run(w, ppm)
    assert len(cuts) <= max(1, len(rows) // 100), cuts    # float64 ties only
    sp = w.spec
    for b, L in enumerate(sp.lengths):
        nqb = -(-L // sp.block_size)
        assert (len_g[b, :, nqb:] == 0).all() and (mask_g[b, :, nqb:] == -1).all()


def test_top_p_full_pipeline_32k():
    """32K tokens, 32 heads, p = 0.95 and the workload's Delta: KAP + OSK through the C ABI, the oracle
    on sampled (head, query block) items."""
    from tests.test_gpu_full import sampled_items
    sp = synth.spec_for("32k_gqa_shuffled")
    delta = json.load(open(GOLDEN))["workloads"]["32k_gqa_shuffled"]["delta"]
    w = synth.make_workload(sp)
    items = sampled_items(sp, 24, seed=95)
    dw, p, prm, mask_g, len_g, rows, cuts = _run(w, 950_000, delta=delta, items=items)
    assert len(cuts) <= 1, cuts
    # realised stage-1 budget of the rule on this input, for the record
    nqb = mask_g.shape[2]
    frac = len_g.sum() / (sp.num_q_heads * nqb * (nqb + 1) / 2)
    assert 0.0 < frac <= 1.0
    out, flags = gh.run_osk(dw, p, mask_g, len_g)
    exact = [it for it in items if not any(c[0] == it for c in cuts)]
    mask_o = mask_g.copy()
    rep = gh.compare_osk(w, prm, mask_o, len_g, out, flags, exact)
    gh.assert_osk_ok(rep)
    print(f"top-p 0.95 on {sp.name}: realised stage-1 budget {frac:.3f}, cut differences {len(cuts)}")


@pytest.mark.parametrize("ppm", [500_000, 750_000])
def test_top_p_constant_keys_exact_path(ppm):
    """Every key equal: every block of a row scores the same (8 sampled rows, each at its maximum), so
    p times the total falls exactly on a prefix boundary whenever p J_i is an integer.  The fp32 bounds
    cannot settle such a cut; the kernel takes it from exact scores of every candidate, and any length
    that differs from the oracle's must be a float64 tie."""
    from tests.test_gpu_osk import small_spec as ss
    sp = ss("d128_b128_P64", seed=611)
    w = synth.make_workload(sp)
    w.k_cache[...] = w.k_cache[0, 0, 0, :]
    _, _, _, mask_g, len_g, rows, cuts = _run(w, ppm)
    for (b, h, i), r in rows.items():
        J = i + 1
        want = -(-ppm * J // 1_000_000)
        assert int(len_g[b, h, i]) in (max(1, want), want + 1), ((b, h, i), int(len_g[b, h, i]), want)

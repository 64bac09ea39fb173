"""KAP parity on the GPU: cosa_proxy_select through the C ABI against the float64 oracle
(CoSA Sec. 4.2, Eqs. (8)-(14)).  Masks must be bit-exact; a difference is accepted only
between two blocks whose oracle scores tie in float64."""
import math

import numpy as np
import pytest

import synth
from oracle import cosa_oracle as orc
from tests import gpu_helpers as gh
from tests.test_gpu_osk import SMALL, small_spec

pytestmark = pytest.mark.gpu


def _kap_check(w, budget_ppm=None, heads=None, missing_pages=False):
    sp = w.spec
    if missing_pages:
        w.page_table[0, 2] = -1
    ppm = sp.budget_ppm if budget_ppm is None else budget_ppm
    prm = gh.oracle_params(sp, -1.0, budget_ppm=ppm)
    pitch = gh.C.stage1_pitch(ppm, sp.max_seqlen, sp.block_size)
    dw = gh.to_device(w)
    mask_g, len_g = gh.run_kap(dw, gh.cosa_params(dw, delta=-1.0, mask_pitch=pitch, budget_ppm=ppm))
    _, _, rows = orc.kap_mask(w.q, w.k_cache, w.page_table, w.cu_seqlens, sp.num_q_heads, sp.num_kv_heads,
                              prm, pitch, heads=heads)
    ties = gh.compare_masks(mask_g, len_g, rows, sp.lengths, sp.block_size, workload=sp.name)
    return ties


@pytest.mark.parametrize("name", sorted(SMALL))
def test_kap_small(name):
    if SMALL[name]["block_size"] // SMALL[name]["stride"] not in (4, 8, 16):
        pytest.skip("stride ratio not supported")
    w = synth.make_workload(small_spec(name, seed=200 + len(name)))
    _kap_check(w, missing_pages=True)


@pytest.mark.parametrize("ppm", [1_000_000, 250_000, 1])
def test_kap_budgets(ppm):
    """Budget 100 % orders every causal block; budget 1 ppm keeps one block per row."""
    w = synth.make_workload(small_spec("d128_b128_P64", seed=300))
    _kap_check(w, budget_ppm=ppm)


def test_kap_2k_single_head():
    w = synth.make_workload(synth.spec_for("2k_d64_1head"))
    _kap_check(w)


def test_kap_8k_all_heads():
    w = synth.make_workload(synth.spec_for("8k_gqa"))
    ties = _kap_check(w)
    assert len(ties) < 5


def test_kap_constant_keys_ties():
    """Degenerate input: every key equal, so every block ties for every row's maximum."""
    sp = small_spec("d128_b128_P64", seed=301)
    w = synth.make_workload(sp)
    w.k_cache[...] = w.k_cache[0, 0, 0, :]
    _kap_check(w, budget_ppm=500_000)


def test_kap_long_rows_both_select_paths():
    """b = 64 over 70,000 tokens: query blocks up to 1,094, so rows with J_i <= 1024 and K_i <= 128
    are selected one warp per row and the others (J_i > 1024, or K_i > 128 at a 20 % budget) by the
    block-per-row kernel from its list.  Rows on both sides of each limit against the oracle."""
    sp = synth.WorkloadSpec(name="long_b64", lengths=(70000,), num_q_heads=2, num_kv_heads=1, head_dim=64,
                            block_size=64, page_size=32, stride=8, budget_ppm=200_000, stage2_budget_ppm=0,
                            seed=303, shuffle_pages=True, salient_pages=4)
    w = synth.make_workload(sp)
    prm = gh.oracle_params(sp, -1.0)
    pitch = gh.C.stage1_pitch(sp.budget_ppm, sp.max_seqlen, sp.block_size)
    dw = gh.to_device(w)
    mask_g, len_g = gh.run_kap(dw, gh.cosa_params(dw, delta=-1.0, mask_pitch=pitch))
    # K_i = ceil(0.2 (i + 1)) passes 128 at i = 640; J_i passes 1024 at i = 1024
    rows = [0, 5, 600, 639, 640, 641, 1000, 1022, 1023, 1024, 1025, 1093]
    by = {(0, h): rows for h in range(sp.num_q_heads)}
    _, _, orows = orc.kap_mask(w.q, w.k_cache, w.page_table, w.cu_seqlens, sp.num_q_heads, sp.num_kv_heads,
                               prm, pitch, qblocks=by)
    gh.compare_masks_rows(mask_g, len_g, orows, workload=sp.name)
    nqb = -(-70000 // 64)
    want = np.maximum(1, -(-200_000 * np.arange(1, nqb + 1) // 1_000_000))
    assert (len_g[0, :, :nqb] == want[None, :]).all()

"""OSK parity on the GPU: cosa_sparse_prefill through the C ABI against the float64 oracle,
with the oracle's own KAP masks as input (CoSA Sec. 4.3, Algorithm A (ordered-skipping stage); PageWeaver
Sec. 2.1 output semantics)."""
import json
import math
import os

import numpy as np
import pytest

import synth
from oracle import cosa_oracle as orc
from tests import gpu_helpers as gh

pytestmark = pytest.mark.gpu

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "delta_calibration.json")

SMALL = {
    # ragged tails, a request shorter than one block, single-token request, shuffled pages
    "d128_b128_P64": dict(head_dim=128, block_size=128, page_size=64, stride=16, lengths=(1000, 300, 129, 1)),
    "d64_b64_P64": dict(head_dim=64, block_size=64, page_size=64, stride=8, lengths=(777, 64, 63)),
    "d128_b64_P32": dict(head_dim=128, block_size=64, page_size=32, stride=8, lengths=(900, 65)),
    "d64_b128_P16": dict(head_dim=64, block_size=128, page_size=16, stride=16, lengths=(1300, 200)),
}


def small_spec(name, seed):
    c = SMALL[name]
    return synth.WorkloadSpec(name=name, lengths=c["lengths"], num_q_heads=4, num_kv_heads=2,
                              head_dim=c["head_dim"], block_size=c["block_size"], page_size=c["page_size"],
                              stride=c["stride"], budget_ppm=400_000, stage2_budget_ppm=0, seed=seed,
                              shuffle_pages=True, salient_pages=3)


def oracle_masks(w, prm, pitch, noise_seed=None, missing_pages=()):
    sp = w.spec
    mask, ml, rows = orc.kap_mask(w.q, w.k_cache, w.page_table, w.cu_seqlens, sp.num_q_heads,
                                  sp.num_kv_heads, prm, pitch)
    if noise_seed is not None:
        mask, ml = synth.inject_mask_noise(mask, ml, sp.lengths, sp.block_size, 0.3, noise_seed)
    return mask, ml, rows


@pytest.mark.parametrize("name", sorted(SMALL))
@pytest.mark.parametrize("delta", [-1.0, 40.0])
def test_osk_small_edge_cases(name, delta):
    sp = small_spec(name, seed=100 + len(name))
    w = synth.make_workload(sp)
    # two pages of the first request vanish from its page table
    w.page_table[0, 1] = -1
    w.page_table[0, 3] = sp.num_pages + 7
    prm = gh.oracle_params(sp, delta)
    pitch = gh.C.stage1_pitch(sp.budget_ppm, sp.max_seqlen, sp.block_size) + 6
    mask, ml, _ = oracle_masks(w, prm, pitch, noise_seed=5)
    dw = gh.to_device(w)
    p = gh.cosa_params(dw, delta=delta, mask_pitch=pitch)
    out, flags = gh.run_osk(dw, p, mask, ml)
    rep = gh.compare_osk(w, prm, mask, ml, out, flags, gh.items_of(sp))
    gh.assert_osk_ok(rep)
    if delta > 0:
        assert (flags == orc.SKIPPED).any()


@pytest.mark.parametrize("delta", [-1.0, 2000.0])
def test_osk_2k_single_head(delta):
    """1 head, d = 64, 2048 tokens, page/block 64, budget 25 %, skip off and on (Delta = 2000)."""
    sp = synth.spec_for("2k_d64_1head")
    w = synth.make_workload(sp)
    prm = gh.oracle_params(sp, delta)
    pitch = gh.C.stage1_pitch(sp.budget_ppm, sp.max_seqlen, sp.block_size)
    mask, ml, _ = oracle_masks(w, prm, pitch)
    dw = gh.to_device(w)
    out, flags = gh.run_osk(dw, gh.cosa_params(dw, delta=delta, mask_pitch=pitch), mask, ml)
    rep = gh.compare_osk(w, prm, mask, ml, out, flags, gh.items_of(sp))
    gh.assert_osk_ok(rep)


def test_osk_8k_sampled_heads():
    """GQA 32/8, d = 128, 8K tokens; GPU runs every item, the oracle checks three heads."""
    sp = synth.spec_for("8k_gqa")
    delta = json.load(open(GOLDEN))["workloads"]["8k_gqa"]["delta"]
    w = synth.make_workload(sp)
    prm = gh.oracle_params(sp, delta)
    pitch = gh.C.stage1_pitch(sp.budget_ppm, sp.max_seqlen, sp.block_size)
    heads = [0, 13, 31]
    mask, ml, _ = orc.kap_mask(w.q, w.k_cache, w.page_table, w.cu_seqlens, sp.num_q_heads, sp.num_kv_heads,
                               prm, pitch, heads=heads)
    dw = gh.to_device(w)
    out, flags = gh.run_osk(dw, gh.cosa_params(dw, delta=delta, mask_pitch=pitch), mask, ml)
    rep = gh.compare_osk(w, prm, mask, ml, out, flags, gh.items_of(sp, heads=heads))
    gh.assert_osk_ok(rep)
    assert (flags == orc.SKIPPED).any()


def test_osk_empty_and_all_invalid_rows():
    """Rows whose entries are all invalid give zero output; mask_len 0 visits nothing."""
    sp = small_spec("d128_b128_P64", seed=9)
    w = synth.make_workload(sp)
    prm = gh.oracle_params(sp, -1.0)
    nqb = -(-sp.max_seqlen // sp.block_size)
    pitch = 5
    mask = np.full((sp.num_reqs, sp.num_q_heads, nqb, pitch), -1, np.int32)
    ml = np.zeros((sp.num_reqs, sp.num_q_heads, nqb), np.int32)
    mask[0, 0, 3, :4] = [-7, 9, 100, -1]      # nothing valid for query block 3
    ml[0, 0, 3] = 4
    mask[0, 1, 2, :3] = [2, 2, 0]             # repeats count once
    ml[0, 1, 2] = 3
    dw = gh.to_device(w)
    out, flags = gh.run_osk(dw, gh.cosa_params(dw, delta=-1.0, mask_pitch=pitch), mask, ml)
    rep = gh.compare_osk(w, prm, mask, ml, out, flags, gh.items_of(sp))
    gh.assert_osk_ok(rep)
    t0 = 3 * sp.block_size
    assert (out[t0:t0 + sp.block_size, 0, :] == 0).all()
    assert list(flags[0, 1, 2, :3]) == [0, 2, 0]

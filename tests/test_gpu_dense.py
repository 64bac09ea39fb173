"""Dense endpoint of the OSK (every causal block, ascending order, skipping off: B1 = 100 %, Delta = -1,
the stage-1-only endpoint of CoSA App. D.1) against the float64 oracle's Algorithm A on the same masks,
every item compared, and against PyTorch's fp32 causal attention on the same GPU: with B1 = 100 % and
Delta <= 0, CoSA's Algorithm A reduces to exact causal softmax attention (CoSA Sec. 4.3; the oracle
pins the same reduction in float64)."""
import math

import numpy as np
import pytest
import torch

import synth
from tests import gpu_helpers as gh

pytestmark = pytest.mark.gpu


def dense_mask(lengths, block_size, num_q_heads, pitch):
    nqb = -(-max(lengths) // block_size)
    mask = np.full((len(lengths), num_q_heads, nqb, pitch), -1, np.int32)
    ml = np.zeros((len(lengths), num_q_heads, nqb), np.int32)
    for b, L in enumerate(lengths):
        for i in range(-(-L // block_size)):
            mask[b, :, i, :i + 1] = np.arange(i + 1, dtype=np.int32)
            ml[b, :, i] = i + 1
    return mask, ml


def paged_to_dense(w, dev):
    """Per request: K and V rows [L, Hkv, d] gathered through the page table (fp32)."""
    sp = w.spec
    out = []
    kc = torch.from_numpy(synth.bf16_bits_to_f32(w.k_cache)).to(dev)
    vc = torch.from_numpy(synth.bf16_bits_to_f32(w.v_cache)).to(dev)
    for b, L in enumerate(sp.lengths):
        pages = [int(p) for p in w.page_table[b, :-(-L // sp.page_size)]]
        k = torch.cat([kc[p] for p in pages])[:L]
        v = torch.cat([vc[p] for p in pages])[:L]
        out.append((k, v))
    return out


@pytest.mark.parametrize("block_size,page_size,head_dim", [(128, 64, 128), (64, 32, 64)])
def test_dense_endpoint_matches_torch_causal_attention(block_size, page_size, head_dim):
    sp = synth.WorkloadSpec(name=f"dense_b{block_size}_P{page_size}_d{head_dim}", lengths=(2048, 1500, 77), num_q_heads=4, num_kv_heads=2,
                            head_dim=head_dim, block_size=block_size, page_size=page_size,
                            stride=block_size // 8, budget_ppm=1_000_000, stage2_budget_ppm=0, seed=31,
                            shuffle_pages=True, salient_pages=3)
    w = synth.make_workload(sp)
    dw = gh.to_device(w)
    dev = dw.q.device
    nqb = -(-sp.max_seqlen // sp.block_size)
    mask, ml = dense_mask(sp.lengths, sp.block_size, sp.num_q_heads, nqb)
    p = gh.cosa_params(dw, delta=-1.0, mask_pitch=nqb)
    out, flags = gh.run_osk(dw, p, mask, ml)
    for b, L in enumerate(sp.lengths):
        n = -(-L // sp.block_size)
        assert (flags[b, :, :n, :][np.arange(nqb)[None, None, :] < ml[b, :, :n, None]] == 0).all()

    # the oracle's Algorithm A over the same dense masks, every (request, head, query block)
    prm = gh.oracle_params(sp, -1.0, budget_ppm=1_000_000)
    rep = gh.compare_osk(w, prm, mask, ml, out, flags, gh.items_of(sp))
    gh.assert_osk_ok(rep)
    assert rep.n_disagree == 0 and rep.n_items == sum(sp.num_q_heads * -(-L // sp.block_size) for L in sp.lengths)

    q = torch.from_numpy(synth.bf16_bits_to_f32(w.q)).to(dev)
    g = sp.num_q_heads // sp.num_kv_heads
    kv = paged_to_dense(w, dev)
    t0 = 0
    worst, total, count = 0.0, 0.0, 0
    for b, L in enumerate(sp.lengths):
        qb = q[t0:t0 + L].permute(1, 0, 2)                              # [Hq, L, d]
        k, v = kv[b]
        kb = k.permute(1, 0, 2).repeat_interleave(g, dim=0)            # [Hq, L, d]
        vb = v.permute(1, 0, 2).repeat_interleave(g, dim=0)
        ref = torch.nn.functional.scaled_dot_product_attention(qb, kb, vb, is_causal=True,
                                                               scale=1.0 / math.sqrt(head_dim))
        got = torch.from_numpy(out[t0:t0 + L]).to(dev).permute(1, 0, 2)
        d = (got - ref).abs()
        worst = max(worst, float(d.max()))
        total += float(d.sum())
        count += d.numel()
        t0 += L
    assert worst <= gh.O_MAX_ABS, worst
    assert total / count <= gh.O_MEAN_ABS, total / count

"""Host-side checks of the Python binding: every buffer passed to the C ABI must hold at least the
elements the parameters imply (the library cannot see tensor sizes).  Meta tensors stand in for
device memory, so this runs without a GPU."""
import pytest
import torch

import synth
from block_sparse_long_gb300 import cosa as C


def meta(shape, dtype):
    return torch.empty(shape, dtype=dtype, device="meta")


def buffers_for(spec, pitch):
    nqb = -(-spec.max_seqlen // spec.block_size)
    B, Hq = spec.num_reqs, spec.num_q_heads
    q = meta((spec.total_tokens, Hq, spec.head_dim), torch.bfloat16)
    k = meta((spec.num_pages, spec.page_size, spec.num_kv_heads, spec.head_dim), torch.bfloat16)
    pt = meta((B, max(spec.pages_of(L) for L in spec.lengths)), torch.int32)
    cu = meta((B + 1,), torch.int32)
    mask = meta((B, Hq, nqb, pitch), torch.int32)
    return dict(q=q, k_cache=k, v_cache=k, page_table=pt, cu_seqlens=cu, mask=mask,
                mask_len=meta((B, Hq, nqb), torch.int32), out=q, visit_flags=meta(mask.shape, torch.uint8),
                status=meta((1,), torch.int32))


def params(spec, bufs, pitch):
    return C.params_for(bufs["q"], bufs["k_cache"], bufs["page_table"], bufs["cu_seqlens"],
                        block_size=spec.block_size, max_seqlen=spec.max_seqlen, stride=spec.stride,
                        budget_ppm=spec.budget_ppm, mask_pitch=pitch, skip_delta=-1.0)


@pytest.mark.parametrize("name", sorted(synth.WORKLOADS))
@pytest.mark.parametrize("extra", [0, 4])
def test_buffers_shaped_like_the_callers_pass(name, extra):
    spec = synth.spec_for(name)
    pitch = C.stage1_pitch(spec.budget_ppm, spec.max_seqlen, spec.block_size) + extra
    bufs = buffers_for(spec, pitch)
    C.validate_buffers(params(spec, bufs, pitch), **bufs)
    # binary block masks: one entry per causal block, pitch = nqb_max
    nqb = -(-spec.max_seqlen // spec.block_size)
    bb = buffers_for(spec, nqb)
    C.validate_buffers(params(spec, bb, nqb), **bb)


@pytest.mark.parametrize("victim", ["q", "k_cache", "v_cache", "page_table", "cu_seqlens", "mask", "mask_len",
                                    "out", "visit_flags", "status"])
def test_undersized_buffer_is_refused(victim):
    spec = synth.WorkloadSpec(name="tiny", lengths=(300, 129), num_q_heads=4, num_kv_heads=2, head_dim=64,
                              block_size=64, page_size=32, stride=8, budget_ppm=400_000, stage2_budget_ppm=0,
                              seed=1)
    pitch = C.stage1_pitch(spec.budget_ppm, spec.max_seqlen, spec.block_size)
    bufs = buffers_for(spec, pitch)
    p = params(spec, bufs, pitch)
    t = bufs[victim]
    bufs[victim] = meta((t.numel() - 1,), t.dtype)
    with pytest.raises(ValueError, match=victim):
        C.validate_buffers(p, **bufs)


def test_required_sizes_by_hand():
    # 2 requests (300 and 129 tokens), 4 q heads, 2 kv heads, d = 64, b = 64, P = 32: nqb_max = 5
    p = C.make_params(num_reqs=2, num_q_heads=4, num_kv_heads=2, head_dim=64, block_size=64, page_size=32,
                      total_tokens=429, max_seqlen=300, num_pages=15, max_pages_per_req=10, mask_pitch=3)
    need = C.required_numel(p)
    assert need["q"] == need["out"] == 429 * 4 * 64
    assert need["k_cache"] == need["v_cache"] == 15 * 32 * 2 * 64
    assert need["cu_seqlens"] == 3 and need["page_table"] == 20
    assert need["mask"] == need["visit_flags"] == 2 * 4 * 5 * 3
    assert need["mask_len"] == 2 * 4 * 5 and need["status"] == 1

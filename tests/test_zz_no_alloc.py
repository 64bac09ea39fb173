"""cosa_proxy_select_static: the KAP entry point that allocates nothing.

It exists for callers that cannot allocate device memory (for example code inside a host
framework that owns every device allocation, or a serving loop that must not enter an
allocator while requests are in flight).  Its scratch is a fixed device array inside the
library.  This file checks, through the C ABI, that it produces exactly the mask of
cosa_proxy_select (which takes a workspace) on two calls in a row, and that a problem
larger than the fixed scratch is refused.  It is named so that pytest collects it last.
"""
import ctypes

import numpy as np
import pytest
import torch

import synth
from block_sparse_long_gb300 import cosa as C
from tests import gpu_helpers as gh

pytestmark = pytest.mark.gpu


def _specs():
    small = synth.WorkloadSpec(name="no_alloc_ragged", lengths=(1500, 300, 129), num_q_heads=4, num_kv_heads=2,
                               head_dim=128, block_size=128, page_size=64, stride=16, budget_ppm=300_000,
                               stage2_budget_ppm=0, seed=77, shuffle_pages=True, salient_pages=3)
    return [small, synth.spec_for("8k_gqa")]


@pytest.mark.parametrize("spec", _specs(), ids=lambda s: s.name)
def test_static_scratch_matches_workspace_entry_point(spec):
    from block_sparse_long_gb300 import build
    build.build()
    w = synth.make_workload(spec)
    dw = gh.to_device(w)
    pitch = C.stage1_pitch(spec.budget_ppm, spec.max_seqlen, spec.block_size)
    p = gh.cosa_params(dw, delta=-1.0, mask_pitch=pitch)
    assert C.cosa_proxy_workspace_size(p) <= C.STATIC_SCRATCH_BYTES
    ref_mask, ref_len = gh.run_kap(dw, p)                       # the workspace entry point
    nqb = -(-spec.max_seqlen // spec.block_size)
    for call in range(2):                                      # the array keeps the last call's contents
        mask = torch.full((spec.num_reqs, spec.num_q_heads, nqb, pitch), 12345 + call, dtype=torch.int32,
                          device="cuda")
        mask_len = torch.full((spec.num_reqs, spec.num_q_heads, nqb), -7, dtype=torch.int32, device="cuda")
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        C.cosa_proxy_select_static(p, dw.q, dw.cu, dw.k, dw.pt, mask, mask_len, status=status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0, C.cosa_status_string(int(status.item()))
        assert np.array_equal(mask.cpu().numpy(), ref_mask), f"mask differs on call {call}"
        assert np.array_equal(mask_len.cpu().numpy(), ref_len), f"mask_len differs on call {call}"


def test_static_scratch_refuses_oversized_problem():
    # the 128K-token GQA workload needs far more than the fixed scratch; refused on the host
    spec = synth.spec_for("128k_gqa_student_t")
    L = spec.max_seqlen
    p = C.make_params(num_reqs=1, num_q_heads=32, num_kv_heads=8, head_dim=128, block_size=128, page_size=64,
                      stride=16, total_tokens=L, max_seqlen=L, num_pages=L // 64, max_pages_per_req=L // 64,
                      mask_pitch=C.stage1_pitch(spec.budget_ppm, L, 128), budget_ppm=spec.budget_ppm)
    assert C.cosa_proxy_workspace_size(p) > C.STATIC_SCRATCH_BYTES
    t = torch.zeros(16, dtype=torch.int32, device="cuda")
    q = torch.zeros(16, dtype=torch.bfloat16, device="cuda")
    # the binding refuses buffers smaller than the parameters imply ...
    with pytest.raises(ValueError):
        C.cosa_proxy_select_static(p, q, t, q, t, t, t)
    # ... and the library refuses the problem itself, on the host, before it touches any buffer
    vp = ctypes.c_void_p
    rc = C.library().cosa_proxy_select_static(ctypes.byref(p), vp(q.data_ptr()), vp(t.data_ptr()), vp(q.data_ptr()),
                                              vp(t.data_ptr()), vp(t.data_ptr()), vp(t.data_ptr()), None,
                                              vp(torch.cuda.current_stream().cuda_stream))
    assert rc == C.COSA_ERR_WORKSPACE

"""Failure detection on the GPU without a fault: with COSA_FLAG_TEST_STALL the OSK's producer of
Q and K tiles issues nothing, so every bounded wait in the kernel runs out.  The call must end by
itself, report COSA_ERR_DEVICE_TIMEOUT through device_status, and leave the CUDA context usable
for a normal call right after."""
import time

import numpy as np
import pytest
import torch

import synth
from oracle import cosa_oracle as orc
from tests import gpu_helpers as gh

pytestmark = pytest.mark.gpu


def _small():
    sp = synth.WorkloadSpec(name="timeout", lengths=(700, 260), num_q_heads=4, num_kv_heads=2, head_dim=128,
                            block_size=128, page_size=64, stride=16, budget_ppm=500_000, stage2_budget_ppm=0,
                            seed=77, shuffle_pages=True, salient_pages=2)
    return sp, synth.make_workload(sp)


@pytest.mark.parametrize("union", [False, True])
def test_stalled_producer_times_out_and_context_survives(union):
    """Both OSK kernels: the default one and the GQA page-union one (COSA_FLAG_GQA_UNION)."""
    extra = gh.C.COSA_FLAG_GQA_UNION if union else 0
    sp, w = _small()
    prm = gh.oracle_params(sp, 40.0)
    pitch = gh.C.stage1_pitch(sp.budget_ppm, sp.max_seqlen, sp.block_size)
    mask, ml, _ = orc.kap_mask(w.q, w.k_cache, w.page_table, w.cu_seqlens, sp.num_q_heads, sp.num_kv_heads,
                               prm, pitch)
    dw = gh.to_device(w)
    dev = dw.q.device
    m = gh.i32_tensor(mask, dev)
    mlt = gh.i32_tensor(ml, dev)

    # stalled: every wait runs out (2 s budget), the kernel stops and reports it
    p = gh.cosa_params(dw, delta=40.0, mask_pitch=pitch)
    p.flags = gh.C.COSA_FLAG_TEST_STALL | extra
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    out = torch.zeros_like(dw.q)
    t0 = time.perf_counter()
    gh.C.cosa_sparse_prefill(p, dw.q, dw.cu, dw.k, dw.v, dw.pt, m, mlt, out=out, status=status)
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    assert int(status.item()) == gh.C.COSA_ERR_DEVICE_TIMEOUT, gh.C.cosa_status_string(int(status.item()))
    assert elapsed < 30.0, elapsed

    # the context is still good: the same call without the hook succeeds and matches the oracle
    p.flags = extra
    out2, flags2 = gh.run_osk(dw, p, mask, ml)
    rep = gh.compare_osk(w, prm, mask, ml, out2, flags2 & 3, gh.items_of(sp))
    gh.assert_osk_ok(rep)


def test_unknown_flag_is_rejected_before_launch():
    sp, w = _small()
    dw = gh.to_device(w)
    pitch = gh.C.stage1_pitch(sp.budget_ppm, sp.max_seqlen, sp.block_size)
    p = gh.cosa_params(dw, delta=40.0, mask_pitch=pitch)
    p.flags = 1 << 5
    mask = np.full((len(sp.lengths), sp.num_q_heads, -(-sp.max_seqlen // sp.block_size), pitch), -1, np.int32)
    ml = np.zeros(mask.shape[:3], np.int32)
    with pytest.raises(gh.C.CosaError):
        gh.C.cosa_sparse_prefill(p, dw.q, dw.cu, dw.k, dw.v, dw.pt, gh.i32_tensor(mask, dw.q.device),
                                 gh.i32_tensor(ml, dw.q.device))

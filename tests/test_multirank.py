"""The multi-rank host logic of bench.py on CPU: two gloo ranks, each timing one replica of the
workload, report the slowest rank's time and the whole job's throughput (weak scaling)."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, times, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w, r, local = bench.dist_env()
        assert (w, r, local) == (world, rank, rank)
        ms = bench.max_over_ranks(times[rank], w, torch.device("cpu"))
        dist.barrier()
        out[rank] = ms
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    world = 2
    times = [3.5, 7.25]
    out = mp.Manager().dict()
    mp.spawn(_rank, args=(world, _free_port(), times, out), nprocs=world, join=True)
    assert out[0] == out[1] == max(times)


def test_whole_job_throughput_counts_every_replica():
    # 9.07 TFLOP per replica step, 10 ms per step: 907 TFLOP/s on one rank, twice that on two
    assert bench.job_tflops(1, 9.07e12, 10.0) == pytest.approx(907.0)
    assert bench.job_tflops(2, 9.07e12, 10.0) == pytest.approx(1814.0)
    assert bench.max_over_ranks(4.0, 1, torch.device("cpu")) == 4.0


# --------------------------------------------------------------------------- #
# the kv-head split of one prefill over ranks (block_sparse_long_gb300/shard.py)
# --------------------------------------------------------------------------- #
def test_kv_head_ranges_cover_every_head_once():
    from block_sparse_long_gb300 import shard
    for hkv in (1, 2, 3, 7, 8, 16):
        for world in range(1, hkv + 1):
            ranges = shard.head_ranges(world, hkv)
            assert ranges[0][0] == 0 and ranges[-1][1] == hkv
            assert all(a[1] == b[0] for a, b in zip(ranges, ranges[1:]))       # contiguous, disjoint
            sizes = [b - a for a, b in ranges]
            assert min(sizes) >= 1 and max(sizes) - min(sizes) <= 1
    with pytest.raises(ValueError):
        shard.kv_head_range(0, 9, 8)                                           # a rank without heads


def test_shard_keeps_the_query_to_kv_head_mapping():
    import numpy as np
    from block_sparse_long_gb300 import shard
    T, P, pages, hkv, g, d = 5, 4, 3, 8, 4, 6
    q = np.arange(T * hkv * g * d).reshape(T, hkv * g, d)
    k = np.arange(pages * P * hkv * d).reshape(pages, P, hkv, d)
    for world in (1, 2, 4, 8):
        for rank in range(world):
            kv0, kv1 = shard.kv_head_range(rank, world, hkv)
            qs, ks, vs = shard.shard_heads(q, k, k, kv0, kv1, g)
            assert qs.flags["C_CONTIGUOUS"] and ks.flags["C_CONTIGUOUS"]
            for lh in range(qs.shape[1]):
                h = kv0 * g + lh                                              # global query head
                assert np.array_equal(qs[:, lh], q[:, h])
                # local query head lh reads local kv head lh // g, which is global kv head h // g
                assert np.array_equal(ks[:, :, lh // g], k[:, :, h // g])


def test_sharded_oracle_equals_whole_problem():
    """Each (request, kv head) group is independent (CoSA Sec. 4.2-4.3): the oracle's masks and outputs
    on one rank's heads equal those heads' rows of the whole problem."""
    import math
    import numpy as np
    import synth
    from block_sparse_long_gb300 import shard
    from oracle import cosa_oracle as orc
    sp = synth.WorkloadSpec(name="shard", lengths=(300, 170), num_q_heads=8, num_kv_heads=4, head_dim=16,
                            block_size=32, page_size=16, stride=4, budget_ppm=400_000, stage2_budget_ppm=0,
                            seed=17, shuffle_pages=True, salient_pages=2)
    w = synth.make_workload(sp)
    prm = orc.Params(32, 16, 4, 400_000, 1.0 / math.sqrt(16), 40.0)
    mask, ml, _ = orc.kap_mask(w.q, w.k_cache, w.page_table, w.cu_seqlens, 8, 4, prm, 8)
    full = orc.osk_all(w.q, w.k_cache, w.v_cache, w.page_table, w.cu_seqlens, 8, 4, prm, mask, ml)
    kv0, kv1 = shard.kv_head_range(1, 2, 4)                                  # heads 2, 3 of 4
    qs, ks, vs = shard.shard_heads(w.q, w.k_cache, w.v_cache, kv0, kv1, 2)
    m1, l1, _ = orc.kap_mask(qs, ks, w.page_table, w.cu_seqlens, 4, 2, prm, 8)
    assert np.array_equal(m1, mask[:, 4:8]) and np.array_equal(l1, ml[:, 4:8])
    part = orc.osk_all(qs, ks, vs, w.page_table, w.cu_seqlens, 4, 2, prm, m1, l1)
    for (b, lh, i), r in part.items():
        ref = full[(b, lh + 4, i)]
        assert np.array_equal(r.out, ref.out) and np.array_equal(r.flags, ref.flags)


def _gather_rank(rank, world, port, hkv, g, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        from block_sparse_long_gb300 import shard
        T, d = 6, 3
        whole = torch.arange(T * hkv * g * d, dtype=torch.float32).reshape(T, hkv * g, d)
        kv0, kv1 = shard.kv_head_range(rank, world, hkv)
        h0, h1 = shard.q_head_range(kv0, kv1, g)
        got = shard.gather_heads(whole[:, h0:h1].contiguous(), world, hkv, g)
        out[rank] = bool(torch.equal(got, whole))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("hkv,g", [(8, 4), (3, 2)])
def test_two_gloo_ranks_gather_o_over_heads(hkv, g):
    """The gathered O of a head split (uneven when 3 kv heads go to 2 ranks) has the single-rank layout."""
    world = 2
    out = mp.Manager().dict()
    mp.spawn(_gather_rank, args=(world, _free_port(), hkv, g, out), nprocs=world, join=True)
    assert out[0] and out[1]


def _bench_shard_rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import synth
        sp = synth.WorkloadSpec(name="tiny", lengths=(100,), num_q_heads=8, num_kv_heads=4, head_dim=16,
                                block_size=32, page_size=16, stride=4, budget_ppm=400_000, stage2_budget_ppm=0, seed=3)
        w = synth.make_workload(sp)
        ws, (kv0, kv1) = bench.shard_workload(w, rank, world)
        flops = bench.kap_flops(ws.spec)
        out[rank] = (kv0, kv1, ws.spec.num_q_heads, bench.sum_over_ranks(flops, world, torch.device("cpu")),
                     bench.kap_flops(sp))
    finally:
        dist.destroy_process_group()


def test_bench_head_split_counts_the_whole_job_once():
    world = 2
    out = mp.Manager().dict()
    mp.spawn(_bench_shard_rank, args=(world, _free_port(), out), nprocs=world, join=True)
    assert (out[0][0], out[0][1], out[1][0], out[1][1]) == (0, 2, 2, 4)
    assert out[0][2] == out[1][2] == 4
    assert out[0][3] == out[1][3] == pytest.approx(out[0][4])                 # sum over ranks = whole job

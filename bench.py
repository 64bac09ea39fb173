"""Benchmark of CoSA sparse prefill (KAP + OSK) on one or more GB300s.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload 128k_gqa_student_t] [--impl cosa|reference]

One step is one pass of the whole hot path over the workload's batch:
cosa_proxy_select (KAP: sampled logits, block scores, HRM-first ordered mask) followed by
cosa_sparse_prefill (OSK: ordered visits through the page table, in-kernel skip, online
softmax).  Inputs are resident in HBM when the timed region starts; the end-to-end variant
(`e2e`) also copies the step's inputs from pinned host memory and reads the output back.

Work accounting (algorithmic FLOPs, the same for every implementation):
  OSK  2*b*b*d per visited block (Q K^T, diagonal blocks counted whole) plus 2*b*b*d per
       computed block (P V), b = block size, d = head dim;
  KAP  2*d per causal (sampled row, sampled key) pair.
Prints one JSON line (rank 0).

Other modes (one JSON line per measurement, not the bench line): --sweep (CoSA against the dense
endpoint of the same kernel, 4K to 128K tokens), --ablation remap|jump|topp|union (skip ratio
against Delta with and without page remapping, physical jumps against logical skipping of a binary
mask, the top-p stage-1 rule, GQA page reuse), --ablation union-kernel (the GQA page-union OSK against
the default OSK on the same masks), --clocks-log PATH (keep the raw clock samples).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import multiprocessing as mp
import os
import shutil
import statistics
import subprocess
import sys
import tempfile
import time

# BLAS threads pinned to one, so the oracle's core count is exactly the pool size
for _v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_v, "1")

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import synth  # noqa: E402

METRIC = "OSK sparse prefill ms and effective TFLOP/s at 128K; % bf16 tensor peak"
UNIT = "TFLOP/s"
L2_BYTES = 129 * 1024 * 1024
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# --------------------------------------------------------------------------- #
# workload and work accounting
# --------------------------------------------------------------------------- #
def delta_for(workload: str) -> float:
    cal = json.load(open(os.path.join(ROOT, "tests", "golden", "delta_calibration.json")))
    return float(cal["workloads"][workload]["delta"])


def kap_flops(spec) -> float:
    total = 0.0
    for L in spec.lengths:
        R = -(-L // spec.stride)
        total += spec.num_q_heads * 2.0 * spec.head_dim * R * (R + 1) / 2.0
    return total


def osk_flops_from_flags(spec, flags: np.ndarray) -> tuple:
    tile = 2.0 * spec.block_size * spec.block_size * spec.head_dim
    f = flags & 3          # the GQA page-union kernel adds a shared-load bit (4)
    visited = int((f != 2).sum())
    computed = int((f == 0).sum())
    return tile * (visited + computed), visited, computed


def dense_equiv_flops(spec) -> float:
    total = 0.0
    for L in spec.lengths:
        nqb = -(-L // spec.block_size)
        total += spec.num_q_heads * 4.0 * spec.block_size ** 2 * spec.head_dim * nqb * (nqb + 1) / 2.0
    return total


# --------------------------------------------------------------------------- #
# CPU baseline: the float64 oracle on a bounded sample (process pool, one item group per task)
# --------------------------------------------------------------------------- #
_W = None  # workload inherited by forked workers


def _oracle_group(args):
    b, h, qblocks, delta = args
    os.environ["OMP_NUM_THREADS"] = "1"
    from oracle import cosa_oracle as orc
    w = _W
    sp = w.spec
    G = sp.num_q_heads // sp.num_kv_heads
    t0 = time.perf_counter()
    prm = orc.Params(sp.block_size, sp.page_size, sp.stride, sp.budget_ppm, 1.0 / math.sqrt(sp.head_dim), delta)
    L = sp.lengths[b]
    Q = orc.request_queries(w.q, w.cu_seqlens, b, h)
    K, ex = orc.request_keys(w.k_cache, w.page_table[b], L, sp.page_size, h // G)
    V, _ = orc.request_keys(w.v_cache, w.page_table[b], L, sp.page_size, h // G)
    rows = orc.kap_request_head(Q, K, ex, prm, qblocks)
    tile = 2.0 * sp.block_size ** 2 * sp.head_dim
    flops = 0.0
    for i, row in rows.items():
        r = orc.osk_qblock(Q, K, V, ex, i, row.order[:row.K], row.K, prm)
        flops += tile * (int((r.flags != orc.IGNORED).sum()) + int((r.flags == orc.COMPUTED).sum()))
        nrows = len(range(i * sp.block_size, min(L, (i + 1) * sp.block_size), sp.stride))
        first = i * sp.block_size // sp.stride
        flops += 2.0 * sp.head_dim * sum(first + k + 1 for k in range(nrows))
    return flops, time.perf_counter() - t0


def sample_groups(spec, n_groups: int, per_group: int, delta: float, seed: int = 99):
    rng = np.random.default_rng(seed)
    groups = []
    b = int(np.argmax(spec.lengths))
    nqb = -(-spec.lengths[b] // spec.block_size)
    heads = rng.choice(spec.num_q_heads, size=min(n_groups, spec.num_q_heads), replace=False)
    for gi, h in enumerate(heads):
        # stratified over the query-block axis, the last block always included
        qs = sorted({int(nqb - 1 - gi % 2)} | {int(x) for x in rng.integers(0, nqb, per_group - 1)})
        groups.append((b, int(h), qs, delta))
    return groups


def cpu_oracle_run(w, groups, cores: int):
    global _W
    _W = w
    ctx = mp.get_context("fork")          # forked before this process touches CUDA
    t0 = time.perf_counter()
    with ctx.Pool(cores) as pool:
        res = pool.map(_oracle_group, groups)
    wall = time.perf_counter() - t0
    flops = sum(r[0] for r in res)
    cpu_s = sum(r[1] for r in res)
    return flops, wall, cpu_s


# --------------------------------------------------------------------------- #
# clocks during the timed region
# --------------------------------------------------------------------------- #
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, bus_id: str, keep: str = None):
        self.bus_id = bus_id
        self.keep = keep            # optional path that receives the raw samples
        self.proc = None
        fd, self.path = tempfile.mkstemp(prefix="cosa_clocks_", suffix=".csv")
        os.close(fd)

    def __enter__(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", self.bus_id, f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "50"], stdout=self.f,
                                         stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
            return self
        # the timed region starts only once the sampler is writing, so that it is covered throughout
        t0 = time.perf_counter()
        while time.perf_counter() - t0 < 1.5 and self.proc.poll() is None:
            self.f.flush()
            if os.path.getsize(self.path) > 0:
                break
            time.sleep(0.02)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.f.close()

    def summary(self):
        if self.proc is None or not os.path.exists(self.path):
            if os.path.exists(self.path):
                os.remove(self.path)
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"]}
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if self.keep:
            shutil.copyfile(self.path, self.keep)
        os.remove(self.path)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# --------------------------------------------------------------------------- #
# helpers
# --------------------------------------------------------------------------- #
def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        d = json.load(open(path))
        return d, "measured"
    return FALLBACK_PEAKS, "fallback"


def kernel_sha() -> str:
    h = hashlib.sha256()
    for f in ("osk.cu", "osk_kernel.cuh", "ptx.cuh"):
        h.update(open(os.path.join(ROOT, "block_sparse_long_gb300", "csrc", f), "rb").read())
    return h.hexdigest()[:16]


def traffic_per_launch(workload: str):
    """DRAM bytes per OSK launch from the committed ncu summary, if it is for this kernel source."""
    path = os.path.join(ROOT, "profiles", "osk_traffic.json")
    if not os.path.exists(path):
        return None
    d = json.load(open(path))
    if d.get("kernel_sha") != kernel_sha() or d.get("workload") != workload:
        return None
    return d.get("dram_bytes_per_launch")


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(ms: float, world: int, device) -> float:
    """The slowest rank's time (the job ends with it); the value itself on one rank."""
    if world <= 1:
        return ms
    import torch
    import torch.distributed as dist
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tflops(world: int, flops_per_rank_step: float, ms_per_step: float) -> float:
    """Whole-job throughput when every rank runs one replica of the step (weak scaling)."""
    return world * flops_per_rank_step / (ms_per_step * 1e-3) / 1e12


def sum_over_ranks(x: float, world: int, device) -> float:
    """The sum of a per-rank figure over the ranks (the work of the whole job); the value itself on one rank."""
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def shard_workload(w, rank: int, world: int, kv_range=None):
    """The kv heads of ``rank`` (and their query heads) of workload ``w``, as a workload of their own
    (contiguous host arrays; the page table and request lengths are shared).  ``kv_range`` (kv0, kv1)
    names the kv heads directly instead."""
    from block_sparse_long_gb300 import shard
    sp = w.spec
    G = sp.num_q_heads // sp.num_kv_heads
    kv0, kv1 = kv_range if kv_range is not None else shard.kv_head_range(rank, world, sp.num_kv_heads)
    if not 0 <= kv0 < kv1 <= sp.num_kv_heads:
        raise ValueError(f"kv heads [{kv0}, {kv1}) of {sp.num_kv_heads}")
    q, k, v = shard.shard_heads(w.q, w.k_cache, w.v_cache, kv0, kv1, G)
    spec = sp.with_(num_q_heads=(kv1 - kv0) * G, num_kv_heads=kv1 - kv0)
    return synth.Workload(spec=spec, q=q, k_cache=k, v_cache=v, page_table=w.page_table, cu_seqlens=w.cu_seqlens), \
        (kv0, kv1)


# --------------------------------------------------------------------------- #
# reference arm: the oracle, as it stands, on the host cores
# --------------------------------------------------------------------------- #
def run_reference(args, spec, workload_name, delta):
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    cores = os.cpu_count() or 1
    w = synth.make_workload(spec)
    groups = sample_groups(spec, n_groups=cores, per_group=10, delta=delta)
    sample = (f"{sum(len(g[2]) for g in groups)} (head, query block) items of the {workload_name} workload, "
              f"{len(groups)} heads x up to 10 blocks stratified over the block axis, KAP + OSK each")
    for _ in range(args.warmup):
        cpu_oracle_run(w, groups, cores)
    walls, flops = [], 0.0
    for _ in range(args.steps):
        f, wall, _ = cpu_oracle_run(w, groups, cores)
        walls.append(wall)
        flops = f
    ms = 1e3 * sum(walls) / len(walls)
    value = flops / (ms * 1e-3) / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": workload_name, "skip_delta": delta, "sample": sample},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


# --------------------------------------------------------------------------- #
# CUDA arm
# --------------------------------------------------------------------------- #
def run_cosa(args, spec, workload_name, delta):
    world, rank, local = dist_env()
    w = synth.make_workload(spec)
    if args.kv_slice:
        # a slice of the workload at full length: kv heads [a, b) and their query heads (for profiling)
        a_, b_ = (int(x) for x in args.kv_slice.split(":"))
        w, _ = shard_workload(w, 0, 1, kv_range=(a_, b_))
        spec = w.spec
        workload_name = f"{workload_name} kv heads [{a_}, {b_})"
    w_full = w
    by_heads = world > 1 and args.shard == "heads"
    # CPU baseline first: the oracle pool is forked before this process touches CUDA
    cpu = None
    if rank == 0 and world >= 1 and not args.no_cpu_baseline:
        cores = os.cpu_count() or 1
        groups = sample_groups(spec, n_groups=cores, per_group=40, delta=delta)
        f, wall, cpu_s = cpu_oracle_run(w, groups, cores)
        cpu = {"value": f / wall / 1e12, "unit": UNIT, "cores": cores, "kind": "oracle",
               "sample": f"{sum(len(g[2]) for g in groups)} (head, query block) items of the {workload_name} "
                         f"workload ({len(groups)} heads x up to 40 blocks, KAP + OSK each), {wall:.1f} s wall, "
                         f"{cpu_s:.1f} s CPU"}

    import torch
    from block_sparse_long_gb300 import cosa as C

    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    kv_range = (0, spec.num_kv_heads)
    if by_heads:
        # this rank's kv heads and their query heads: the step computes only those (strong scaling)
        w, kv_range = shard_workload(w_full, rank, world)
        spec = w.spec
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream()

    def bf(x):
        return torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).to(dev).view(torch.bfloat16)

    q, k, v = bf(w.q), bf(w.k_cache), bf(w.v_cache)
    pt = torch.from_numpy(w.page_table).to(dev)
    cu = torch.from_numpy(w.cu_seqlens).to(dev)
    pitch = C.stage1_pitch(spec.budget_ppm, spec.max_seqlen, spec.block_size)
    p = C.params_for(q, k, pt, cu, block_size=spec.block_size, max_seqlen=spec.max_seqlen, stride=spec.stride,
                     budget_ppm=spec.budget_ppm, mask_pitch=pitch, skip_delta=delta,
                     flags=C.COSA_FLAG_GQA_UNION if args.gqa_union else 0)
    nqb = -(-spec.max_seqlen // spec.block_size)
    mask = torch.empty((spec.num_reqs, spec.num_q_heads, nqb, pitch), dtype=torch.int32, device=dev)
    mask_len = torch.empty((spec.num_reqs, spec.num_q_heads, nqb), dtype=torch.int32, device=dev)
    ws = torch.empty(C.cosa_proxy_workspace_size(p), dtype=torch.uint8, device=dev)
    out = torch.empty_like(q)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    # entries of absent query blocks (shorter requests) are not written: IGNORED marks them
    flags = torch.full((spec.num_reqs, spec.num_q_heads, nqb, pitch), 2, dtype=torch.uint8, device=dev)

    def kap():
        C.cosa_proxy_select(p, q, cu, k, pt, mask=mask, mask_len=mask_len, workspace=ws, status=status)

    def osk(record=False):
        C.cosa_sparse_prefill(p, q, cu, k, v, pt, mask, mask_len, out=out, visit_flags=flags if record else None,
                              status=status)

    # one untimed pass with visit recording: the work of a step (deterministic)
    kap()
    osk(record=True)
    torch.cuda.synchronize()
    if int(status.item()) != 0:
        raise RuntimeError(C.cosa_status_string(int(status.item())))
    fl = flags.cpu().numpy()
    ofl, visited, computed = osk_flops_from_flags(spec, fl)
    kfl = kap_flops(spec)
    step_flops = ofl + kfl
    causal = sum(spec.num_q_heads * (-(-L // spec.block_size)) * (-(-L // spec.block_size) + 1) / 2
                 for L in spec.lengths)

    for _ in range(args.warmup):
        kap()
        osk()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True),
           torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    bus = torch.cuda.get_device_properties(dev)
    bus_id = f"{getattr(bus, 'pci_domain_id', 0):08X}:{getattr(bus, 'pci_bus_id', 0):02X}:" \
             f"{getattr(bus, 'pci_device_id', 0):02X}.0"
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(bus_id, keep=args.clocks_log) as clk:
        start.record(stream)
        for s in range(args.steps):
            e0, e1, e2 = ev[s]
            e0.record(stream)
            kap()
            e1.record(stream)
            osk()
            e2.record(stream)
        stop.record(stream)
        torch.cuda.synchronize()
    total_ms = start.elapsed_time(stop)
    kap_ms = [ev[s][0].elapsed_time(ev[s][1]) for s in range(args.steps)]
    osk_ms = [ev[s][1].elapsed_time(ev[s][2]) for s in range(args.steps)]
    total_ms = max_over_ranks(total_ms, world, dev)
    if int(status.item()) != 0:
        raise RuntimeError(C.cosa_status_string(int(status.item())))
    ms_step = total_ms / args.steps
    job_flops = sum_over_ranks(step_flops, world, dev)      # the work of every rank's step
    value = job_flops / (ms_step * 1e-3) / 1e12

    # end to end through the public API with host buffers (pinned), copies inside the timed region.
    # Two sets of device inputs and outputs, pipelined across steps: step s's host-to-device copies
    # (one copy stream) and step s-1's device-to-host read (another) overlap the kernels in between.
    hq = torch.from_numpy(np.ascontiguousarray(w.q).view(np.int16)).pin_memory()
    hk = torch.from_numpy(np.ascontiguousarray(w.k_cache).view(np.int16)).pin_memory()
    hv = torch.from_numpy(np.ascontiguousarray(w.v_cache).view(np.int16)).pin_memory()
    hpt = torch.from_numpy(w.page_table).pin_memory()
    hcu = torch.from_numpy(w.cu_seqlens).pin_memory()
    hout = torch.empty(out.shape, dtype=torch.int16).pin_memory()
    houts = [hout, torch.empty_like(hout).pin_memory()]
    sets = [dict(q=q, k=k, v=v, pt=pt, cu=cu, out=out)]
    sets.append({name: torch.empty_like(t) for name, t in sets[0].items()})
    # each direction's copies split over args.copy_streams streams (contiguous chunks of every tensor)
    ncs = max(1, args.copy_streams)
    h2d_streams = [torch.cuda.Stream(device=dev) for _ in range(ncs)]
    d2h_streams = [torch.cuda.Stream(device=dev) for _ in range(ncs)]

    def chunk(t, k):
        flat = t.view(-1)
        return flat[flat.numel() * k // ncs: flat.numel() * (k + 1) // ncs]

    def e2e_steps(n, start_event=None):
        ev_done, ev_out = [None, None], [[], []]
        if start_event is not None:
            for cs in h2d_streams + d2h_streams:
                cs.wait_event(start_event)
        for s in range(n):
            x = s % 2
            b = sets[x]
            ev_in = []
            for k, cs in enumerate(h2d_streams):
                with torch.cuda.stream(cs):
                    if ev_done[x] is not None:
                        cs.wait_event(ev_done[x])           # step s - 2 has finished with this set
                    for name, src in (("q", hq), ("k", hk), ("v", hv)):
                        chunk(b[name].view(torch.int16), k).copy_(chunk(src, k), non_blocking=True)
                    if k == 0:
                        b["pt"].copy_(hpt, non_blocking=True)
                        b["cu"].copy_(hcu, non_blocking=True)
                    ev = torch.cuda.Event()
                    ev.record(cs)
                    ev_in.append(ev)
            for ev in ev_in:
                stream.wait_event(ev)
            for ev in ev_out[x]:
                stream.wait_event(ev)                       # step s - 2's output has been read
            C.cosa_proxy_select(p, b["q"], b["cu"], b["k"], b["pt"], mask=mask, mask_len=mask_len, workspace=ws,
                                status=status)
            C.cosa_sparse_prefill(p, b["q"], b["cu"], b["k"], b["v"], b["pt"], mask, mask_len, out=b["out"],
                                  status=status)
            ev_done[x] = torch.cuda.Event()
            ev_done[x].record(stream)
            ev_out[x] = []
            for k, cs in enumerate(d2h_streams):
                with torch.cuda.stream(cs):
                    cs.wait_event(ev_done[x])
                    chunk(houts[x], k).copy_(chunk(b["out"].view(torch.int16), k), non_blocking=True)
                    ev = torch.cuda.Event()
                    ev.record(cs)
                    ev_out[x].append(ev)
        # a step ends when its output is on the host
        for evs in ev_out:
            for ev in evs:
                stream.wait_event(ev)

    e2e_steps(max(2, args.warmup))
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    e_start, e_stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e_start.record(stream)
    e2e_steps(args.steps, start_event=e_start)
    e_stop.record(stream)
    torch.cuda.synchronize()
    if int(status.item()) != 0:
        raise RuntimeError(C.cosa_status_string(int(status.item())))
    if not np.array_equal(houts[(args.steps - 1) % 2].numpy(), out.view(torch.int16).cpu().numpy()):
        raise RuntimeError("end-to-end output differs from the device-resident run")
    e2e_ms = max_over_ranks(e_start.elapsed_time(e_stop) / args.steps, world, dev)
    gathered = None
    if by_heads and args.gather_out:
        # the optional exchange of the head split: O of every head on every rank (outside the timed region)
        from block_sparse_long_gb300 import shard
        G = w_full.spec.num_q_heads // w_full.spec.num_kv_heads
        torch.cuda.synchronize()
        g0 = time.perf_counter()
        full = shard.gather_heads(out, world, w_full.spec.num_kv_heads, G)
        torch.cuda.synchronize()
        gathered = {"ms": 1e3 * (time.perf_counter() - g0), "bytes_per_rank": full.numel() * full.element_size(),
                    "heads": int(full.shape[1])}
    h2d = sum(t.numel() * t.element_size() for t in (hq, hk, hv, hpt, hcu))
    d2h = hout.numel() * hout.element_size()

    if rank != 0:
        if world > 1:
            torch.distributed.destroy_process_group()
        return 0
    pk, pk_src = peaks()
    osk_avg = statistics.mean(osk_ms)
    achieved = ofl / (osk_avg * 1e-3) / 1e12
    peak = float(pk["bf16_tflops"])
    traffic = None if args.gqa_union else traffic_per_launch(workload_name)
    cl = clk.summary()
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
        "scaling": "strong" if by_heads else "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": workload_name, "num_reqs": spec.num_reqs, "seq_lens": list(spec.lengths),
                   "num_q_heads": w_full.spec.num_q_heads, "num_kv_heads": w_full.spec.num_kv_heads,
                   "head_dim": spec.head_dim,
                   "block_size": spec.block_size, "page_size": spec.page_size, "stride": spec.stride,
                   "stage1_budget": spec.budget_ppm / 1e6, "skip_delta": delta,
                   **({"osk_variant": "gqa_union (two query heads per K stream)"} if args.gqa_union else {}),
                   "l2": "inputs larger than L2 (q, k, v = %.2f GiB)" % ((q.numel() + k.numel() + v.numel()) * 2 / 2**30),
                   "parallelism": (f"kv heads [{kv_range[0]}, {kv_range[1]}) of {w_full.spec.num_kv_heads} on rank 0, "
                                   f"{world} ranks" if by_heads else f"independent replicas per GPU x{world}")},
        "osk_ms": osk_avg, "kap_ms": statistics.mean(kap_ms),
        "osk_tflops": achieved, "osk_pct_bf16_peak": 100.0 * achieved / peak,
        "dense_equiv_tflops": dense_equiv_flops(spec) / (osk_avg * 1e-3) / 1e12,
        "visits": visited, "computed": computed, "realized_stage1": visited / causal,
        "realized_stage2": computed / causal,
        "roofline": {"bound": "tensor",
                     "kernel": (f"osk_union_kernel<{spec.head_dim},{spec.page_size},"
                                f"{'true' if delta > 0 else 'false'},false>" if args.gqa_union else
                                f"osk_kernel<{spec.block_size},{spec.head_dim},{spec.page_size},false,"
                                f"{'true' if delta > 0 else 'false'},false>"),
                     "achieved": achieved, "peak": peak,
                     "unit": "TFLOP/s", "frac": achieved / peak, "traffic": traffic,
                     "peak_source": f"bf16_tflops ({pk_src}, burst)"},
        "e2e": {"value": job_flops / (e2e_ms * 1e-3) / 1e12, "unit": UNIT, "ms_per_step": e2e_ms,
                "pipelined": "two device input/output sets; step s's host-to-device copy and step s-1's "
                             "device-to-host read overlap the kernels",
                "copy_streams_per_direction": max(1, args.copy_streams),
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": 9 * args.steps,
        "clocks": cl,
    }
    if cpu is not None:
        line["cpu_baseline"] = cpu
    if gathered is not None:
        line["gather_out"] = gathered
    print(json.dumps(line))
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


def run_sweep(args):
    """Dense endpoint vs CoSA over context lengths (one JSON line per length, not the bench line).

    For each length N the 128K workload's structure is generated at N tokens; CoSA runs KAP + OSK at
    B1 = 10 % with Delta = 15000 N / 131072 (the same ln(Delta / N) as the calibrated 128K workload);
    the dense endpoint runs the same OSK over every causal block in ascending order with skipping off
    (B1 = 100 %, Delta = -1), i.e. exact causal attention on the same kernel."""
    import torch
    from block_sparse_long_gb300 import cosa as C
    dev = torch.device("cuda", 0)

    def bf(x):
        return torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).to(dev).view(torch.bfloat16)

    def timed(fn, reps):
        fn()
        torch.cuda.synchronize()
        ts = []
        for _ in range(reps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            fn()
            e1.record()
            torch.cuda.synchronize()
            ts.append(e0.elapsed_time(e1))
        return statistics.median(ts)

    for n_tok in (4096, 8192, 16384, 32768, 65536, 131072):
        spec = synth.spec_for("128k_gqa_student_t", lengths=(n_tok,), name=f"structure_{n_tok // 1024}k")
        delta = 15000.0 * n_tok / 131072
        w = synth.make_workload(spec)
        q, k, v = bf(w.q), bf(w.k_cache), bf(w.v_cache)
        pt = torch.from_numpy(w.page_table).to(dev)
        cu = torch.from_numpy(w.cu_seqlens).to(dev)
        nqb = -(-n_tok // spec.block_size)
        pitch = C.stage1_pitch(spec.budget_ppm, spec.max_seqlen, spec.block_size)
        p = C.params_for(q, k, pt, cu, block_size=spec.block_size, max_seqlen=spec.max_seqlen, stride=spec.stride,
                         budget_ppm=spec.budget_ppm, mask_pitch=pitch, skip_delta=delta)
        mask = torch.empty((1, spec.num_q_heads, nqb, pitch), dtype=torch.int32, device=dev)
        mask_len = torch.empty((1, spec.num_q_heads, nqb), dtype=torch.int32, device=dev)
        ws = torch.empty(C.cosa_proxy_workspace_size(p), dtype=torch.uint8, device=dev)
        out = torch.empty_like(q)
        kap_ms = timed(lambda: C.cosa_proxy_select(p, q, cu, k, pt, mask=mask, mask_len=mask_len, workspace=ws), 10)
        osk_ms = timed(lambda: C.cosa_sparse_prefill(p, q, cu, k, v, pt, mask, mask_len, out=out), 10)
        # dense endpoint: every causal block, ascending, skipping off
        ar = torch.arange(nqb, dtype=torch.int32, device=dev)
        dmask = torch.where(ar[None, :] <= ar[:, None], ar[None, :], torch.full_like(ar[None, :], -1))
        dmask = dmask.expand(spec.num_q_heads, nqb, nqb).reshape(1, spec.num_q_heads, nqb, nqb).contiguous()
        dlen = (ar + 1).expand(spec.num_q_heads, nqb).reshape(1, spec.num_q_heads, nqb).contiguous()
        pd = C.params_for(q, k, pt, cu, block_size=spec.block_size, max_seqlen=spec.max_seqlen, stride=spec.stride,
                          budget_ppm=1_000_000, mask_pitch=nqb, skip_delta=-1.0)
        dense_ms = timed(lambda: C.cosa_sparse_prefill(pd, q, cu, k, v, pt, dmask, dlen, out=out), 5)
        causal_pairs = spec.num_q_heads * nqb * (nqb + 1) // 2
        dense_tflops = 4.0 * spec.block_size * spec.block_size * spec.head_dim * causal_pairs / (dense_ms * 1e-3) / 1e12
        print(json.dumps({"sweep": "cosa_vs_dense_endpoint", "tokens": n_tok, "workload": spec.name,
                          "skip_delta": delta, "stage1_budget": spec.budget_ppm / 1e6,
                          "cosa_ms": kap_ms + osk_ms, "kap_ms": kap_ms, "osk_ms": osk_ms, "dense_ms": dense_ms,
                          "dense_tflops": dense_tflops, "speedup_vs_dense": dense_ms / (kap_ms + osk_ms)}),
              flush=True)
        del q, k, v, mask, ws, out, dmask
        torch.cuda.empty_cache()
    return 0


def group_loads(orders):
    """Loads of a traversal shared by a GQA group whose heads keep their own visiting orders: each
    load serves every head whose next pending block it is; greedily the block next for the most
    heads (ties: lowest ID).  Returns (sum of |S_i|, |U_G|, shared loads)."""
    seqs = [list(dict.fromkeys(int(x) for x in o)) for o in orders]
    n_sel = sum(len(q) for q in seqs)
    n_union = len(set(x for q in seqs for x in q))
    pos = [0] * len(seqs)
    loads = 0
    while True:
        cand = {}
        for p_, q in zip(pos, seqs):
            if p_ < len(q):
                cand[q[p_]] = cand.get(q[p_], 0) + 1
        if not cand:
            break
        blk = min(cand, key=lambda b: (-cand[b], b))
        for h, q in enumerate(seqs):
            if pos[h] < len(q) and q[pos[h]] == blk:
                pos[h] += 1
        loads += 1
    return n_sel, n_union, loads


def union_stats(mask: np.ndarray, mask_len: np.ndarray, group: int):
    """PageWeaver's page reuse rate over the GQA groups (q heads sharing a kv head, same query block):
    rho_Q = sum |S_i| / sum |U_G|, and the same with order-preserving shared loads."""
    B, H, nqb, _ = mask.shape
    tot_sel = tot_union = tot_loads = 0
    for b in range(B):
        for g0 in range(0, H, group):
            for i in range(nqb):
                rows = [mask[b, h, i, :mask_len[b, h, i]] for h in range(g0, g0 + group)]
                if not any(len(r) for r in rows):
                    continue
                s_, u_, l_ = group_loads(rows)
                tot_sel += s_
                tot_union += u_
                tot_loads += l_
    return {"selections": tot_sel, "union_blocks": tot_union, "ordered_loads": tot_loads,
            "rho_Q": tot_sel / max(1, tot_union), "rho_ordered": tot_sel / max(1, tot_loads)}


def run_ablation(args):
    """Kernel-side ablations on synthetic data (one JSON line per point, not the bench line).

    remap: in-kernel skip ratio and OSK time against Delta, visiting in the computation order of
      Eq. (14) (with KV page remapping) or in ascending block order (without), for stage-1 budgets
      B1 in {100, 54, 42, 32, 28} %: the kernel-side analogue of CoSA Fig. 6 and Fig. C.  Skip ratio =
      skipped / visited blocks; budget = computed blocks / causal candidate blocks.
    jump: OSK time with skipping off (Delta = -1) at budgets {25, 50, 75} % and 32K-128K tokens for the
      same selected blocks visited (a) as an ascending ID list (physical jumps), (b) through the binary
      mask with logical skipping of the unselected blocks (BSA-style loop), (c) in the computation
      order; each against the dense endpoint of the same kernel: the analogue of CoSA Fig. B.
    topp: the top-p stage-1 rule (p in {0.8, 0.9, 0.95, 0.99}; the paper runs Qwen at 0.95): realised
      stage-1 budget, KAP time, and OSK time with skipping off and at the workload's Delta.
    union: PageWeaver's page reuse rate rho_Q of the GQA groups on the KAP masks, with and without
      keeping each head's visiting order (the bound on what a shared K/V traversal could save).
    Inputs have the 128K workload's structure at the given length."""
    import torch
    from block_sparse_long_gb300 import cosa as C
    dev = torch.device("cuda", 0)

    def bf(x):
        return torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).to(dev).view(torch.bfloat16)

    def timed(fn, reps):
        fn()
        torch.cuda.synchronize()
        ts = []
        for _ in range(reps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            fn()
            e1.record()
            torch.cuda.synchronize()
            ts.append(e0.elapsed_time(e1))
        return statistics.median(ts)

    def setup(n_tok):
        spec = synth.spec_for("128k_gqa_student_t", lengths=(n_tok,), name=f"structure_{n_tok // 1024}k")
        w = synth.make_workload(spec)
        t = dict(q=bf(w.q), k=bf(w.k_cache), v=bf(w.v_cache), pt=torch.from_numpy(w.page_table).to(dev),
                 cu=torch.from_numpy(w.cu_seqlens).to(dev))
        return spec, t

    def params(spec, t, ppm, pitch, delta, flags=0):
        return C.params_for(t["q"], t["k"], t["pt"], t["cu"], block_size=spec.block_size, max_seqlen=spec.max_seqlen,
                            stride=spec.stride, budget_ppm=ppm, mask_pitch=pitch, skip_delta=delta, flags=flags)

    def kap(spec, t, ppm, flags):
        nqb = -(-spec.max_seqlen // spec.block_size)
        pitch = C.stage1_pitch(ppm, spec.max_seqlen, spec.block_size)
        p = params(spec, t, ppm, pitch, -1.0, flags)
        mask = torch.empty((1, spec.num_q_heads, nqb, pitch), dtype=torch.int32, device=dev)
        ml = torch.empty((1, spec.num_q_heads, nqb), dtype=torch.int32, device=dev)
        C.cosa_proxy_select(p, t["q"], t["cu"], t["k"], t["pt"], mask=mask, mask_len=ml)
        return mask, ml, pitch

    def binary(spec, ids, ml):
        nqb = ids.shape[2]
        ar = torch.arange(ids.shape[3], device=dev)
        live = ar[None, None, None, :] < ml[..., None]
        m01 = torch.zeros((1, spec.num_q_heads, nqb, nqb + 1), dtype=torch.int32, device=dev)
        m01.scatter_(3, torch.where(live, ids, nqb).long(), 1)
        l01 = torch.where(ml > 0, torch.arange(1, nqb + 1, dtype=torch.int32, device=dev)[None, None, :], 0)
        return m01[..., :nqb].contiguous(), l01.to(torch.int32).contiguous()

    if args.ablation == "union":
        for wl in ("32k_gqa_shuffled", "128k_gqa_student_t"):
            spec = synth.spec_for(wl)
            w = synth.make_workload(spec)
            t = dict(q=bf(w.q), k=bf(w.k_cache), pt=torch.from_numpy(w.page_table).to(dev),
                     cu=torch.from_numpy(w.cu_seqlens).to(dev))
            group = spec.num_q_heads // spec.num_kv_heads
            for flags, order in ((0, "rho"), (C.COSA_FLAG_ASCENDING_ORDER, "ascending")):
                mask, ml, _ = kap(spec, t, spec.budget_ppm, flags)
                st = union_stats(mask.cpu().numpy(), ml.cpu().numpy(), group)
                print(json.dumps({"ablation": "union", "workload": spec.name, "group": group, "order": order,
                                  "stage1_budget": spec.budget_ppm / 1e6, **st}), flush=True)
            del t
            torch.cuda.empty_cache()
        return 0
    if args.ablation == "union-kernel":
        # the GQA page-union OSK (COSA_FLAG_GQA_UNION) against the default OSK on the same KAP masks
        for wl in ("32k_gqa_shuffled", "128k_gqa_student_t", "ragged4_gqa_noisy_masks"):
            spec = synth.spec_for(wl)
            w = synth.make_workload(spec)
            delta = delta_for(wl)
            t = dict(q=bf(w.q), k=bf(w.k_cache), v=bf(w.v_cache), pt=torch.from_numpy(w.page_table).to(dev),
                     cu=torch.from_numpy(w.cu_seqlens).to(dev))
            pitch = C.stage1_pitch(spec.budget_ppm, spec.max_seqlen, spec.block_size) + (4 if spec.mask_noise_frac else 0)
            p = params(spec, t, spec.budget_ppm, pitch, delta)
            mask, ml = C.cosa_proxy_select(p, t["q"], t["cu"], t["k"], t["pt"])
            if spec.mask_noise_frac:
                m_np, l_np = synth.inject_mask_noise(mask.cpu().numpy(), ml.cpu().numpy(), spec.lengths,
                                                     spec.block_size, spec.mask_noise_frac, seed=spec.seed)
                mask, ml = torch.from_numpy(m_np).to(dev), torch.from_numpy(l_np).to(dev)
            out = torch.empty_like(t["q"])
            pu = params(spec, t, spec.budget_ppm, pitch, delta, C.COSA_FLAG_GQA_UNION)
            rec = {"ablation": "union-kernel", "workload": spec.name, "skip_delta": delta}
            flags = {}
            for name, pp in (("per_head", p), ("union", pu)):
                rec[f"{name}_osk_ms"] = timed(lambda: C.cosa_sparse_prefill(pp, t["q"], t["cu"], t["k"], t["v"], t["pt"],
                                                                            mask, ml, out=out), 5)
                # rows of absent query blocks (shorter requests) are not written: 255 marks them
                f = torch.full(mask.shape, 255, dtype=torch.uint8, device=dev)
                C.cosa_sparse_prefill(pp, t["q"], t["cu"], t["k"], t["v"], t["pt"], mask, ml, out=out, visit_flags=f)
                flags[name] = f.cpu().numpy()
            live = flags["per_head"] != 255
            visits = int((live & ((flags["per_head"] & 3) != C.VISIT_IGNORED)).sum())
            shared = int((live & ((flags["union"] & C.VISIT_SHARED_LOAD) != 0)).sum())
            rec.update({"visits": visits, "computed": int((flags["per_head"] == C.VISIT_COMPUTED).sum()),
                        "per_head_k_loads": visits, "union_k_loads": visits - shared // 2,
                        "k_loads_saved": (shared // 2) / max(1, visits),
                        "decisions_equal": bool(np.array_equal(np.where(live, flags["union"] & 3, 255),
                                                               flags["per_head"]))})
            print(json.dumps(rec), flush=True)
            del t, mask, ml, out, flags
            torch.cuda.empty_cache()
        return 0
    if args.ablation == "topp":
        n_tok = args.ablation_tokens
        spec, t = setup(n_tok)
        out = torch.empty_like(t["q"])
        nqb = -(-n_tok // spec.block_size)
        cand = spec.num_q_heads * nqb * (nqb + 1) // 2
        delta = 15000.0 * n_tok / 131072
        mask = torch.empty((1, spec.num_q_heads, nqb, nqb), dtype=torch.int32, device=dev)
        ml = torch.empty((1, spec.num_q_heads, nqb), dtype=torch.int32, device=dev)
        for ppm in (800_000, 900_000, 950_000, 990_000):
            p = params(spec, t, ppm, nqb, delta, C.COSA_FLAG_TOP_P)
            ws = torch.empty(C.cosa_proxy_workspace_size(p), dtype=torch.uint8, device=dev)
            kap_ms = timed(lambda: C.cosa_proxy_select(p, t["q"], t["cu"], t["k"], t["pt"], mask=mask, mask_len=ml,
                                                       workspace=ws), 3)
            rec = {"ablation": "topp", "workload": spec.name, "tokens": n_tok, "top_p": ppm / 1e6,
                   "stage1_budget": int(ml.sum()) / cand, "kap_ms": kap_ms}
            for name, d in (("osk_no_skip_ms", -1.0), ("osk_ms", delta)):
                pd = params(spec, t, ppm, nqb, d)
                rec[name] = timed(lambda: C.cosa_sparse_prefill(pd, t["q"], t["cu"], t["k"], t["v"], t["pt"], mask,
                                                                ml, out=out), 3)
            flags = torch.empty(mask.shape, dtype=torch.uint8, device=dev)
            C.cosa_sparse_prefill(params(spec, t, ppm, nqb, delta), t["q"], t["cu"], t["k"], t["v"], t["pt"], mask, ml,
                                  out=out, visit_flags=flags)
            rec["skip_delta"] = delta
            rec["budget_after_skip"] = int((flags == C.VISIT_COMPUTED).sum()) / cand
            print(json.dumps(rec), flush=True)
            del ws, flags
        return 0
    if args.ablation == "remap":
        n_tok = args.ablation_tokens
        spec, t = setup(n_tok)
        out = torch.empty_like(t["q"])
        for ppm in (1_000_000, 540_000, 420_000, 320_000, 280_000):
            masks = {"remap": kap(spec, t, ppm, 0), "ascending": kap(spec, t, ppm, C.COSA_FLAG_ASCENDING_ORDER)}
            nqb = masks["remap"][0].shape[2]
            cand = spec.num_q_heads * nqb * (nqb + 1) // 2
            for delta in (-1.0, 250.0, 500.0, 1000.0, 2000.0, 3000.0, 5000.0, 10000.0, 15000.0, 30000.0):
                rec = {"ablation": "remap", "workload": spec.name, "tokens": n_tok, "stage1_budget": ppm / 1e6,
                       "skip_delta": delta}
                for mode, (mask, ml, pitch) in masks.items():
                    p = params(spec, t, ppm, pitch, delta)
                    flags = torch.empty(mask.shape, dtype=torch.uint8, device=dev)
                    ms = timed(lambda: C.cosa_sparse_prefill(p, t["q"], t["cu"], t["k"], t["v"], t["pt"], mask, ml,
                                                             out=out, visit_flags=flags), 3)
                    computed = int((flags == C.VISIT_COMPUTED).sum())
                    skipped = int((flags == C.VISIT_SKIPPED).sum())
                    rec[f"{mode}_skip_ratio"] = skipped / max(1, computed + skipped)
                    rec[f"{mode}_budget"] = computed / cand
                    rec[f"{mode}_osk_ms"] = ms
                print(json.dumps(rec), flush=True)
            del masks
            torch.cuda.empty_cache()
    else:
        for n_tok in (32768, 65536, 131072):
            spec, t = setup(n_tok)
            out = torch.empty_like(t["q"])
            nqb = -(-n_tok // spec.block_size)
            full, fl, fpitch = kap(spec, t, 1_000_000, C.COSA_FLAG_ASCENDING_ORDER)
            dense_ms = timed(lambda: C.cosa_sparse_prefill(params(spec, t, 1_000_000, fpitch, -1.0), t["q"], t["cu"],
                                                           t["k"], t["v"], t["pt"], full, fl, out=out), 3)
            for ppm in (250_000, 500_000, 750_000):
                ids, ml, pitch = kap(spec, t, ppm, C.COSA_FLAG_ASCENDING_ORDER)
                rho, rl, _ = kap(spec, t, ppm, 0)
                m01, l01 = binary(spec, ids, ml)
                p = params(spec, t, ppm, pitch, -1.0)
                pb = params(spec, t, ppm, nqb, -1.0, C.COSA_FLAG_BINARY_MASK)
                jump_ms = timed(lambda: C.cosa_sparse_prefill(p, t["q"], t["cu"], t["k"], t["v"], t["pt"], ids, ml,
                                                              out=out), 5)
                logical_ms = timed(lambda: C.cosa_sparse_prefill(pb, t["q"], t["cu"], t["k"], t["v"], t["pt"], m01,
                                                                 l01, out=out), 5)
                order_ms = timed(lambda: C.cosa_sparse_prefill(p, t["q"], t["cu"], t["k"], t["v"], t["pt"], rho, rl,
                                                               out=out), 5)
                print(json.dumps({"ablation": "jump", "workload": spec.name, "tokens": n_tok, "budget": ppm / 1e6,
                                  "dense_ms": dense_ms, "jump_ascending_ms": jump_ms,
                                  "logical_binary_ms": logical_ms, "jump_rho_order_ms": order_ms,
                                  "speedup_jump": dense_ms / jump_ms, "speedup_logical": dense_ms / logical_ms}),
                      flush=True)
                del ids, rho, m01
            del t, full
            torch.cuda.empty_cache()
    return 0


def run_link_probe(args):
    """Host-link bandwidth for one step's copies of a workload: its inputs (q, K and V caches) host to
    device and its output device to host, from pinned memory, each alone and both at once, with one
    or more copy streams per direction.  Prints one JSON line per configuration."""
    import torch
    spec = synth.spec_for(args.workload)
    dev = torch.device("cuda", 0)
    w = synth.make_workload(spec)
    nb_in = int(w.q.nbytes + w.k_cache.nbytes + w.v_cache.nbytes)
    nb_out = int(w.q.nbytes)
    h_in = torch.empty(nb_in, dtype=torch.uint8).pin_memory()
    h_out = torch.empty(nb_out, dtype=torch.uint8).pin_memory()
    d_in = torch.empty(nb_in, dtype=torch.uint8, device=dev)
    d_out = torch.empty(nb_out, dtype=torch.uint8, device=dev)
    cur = torch.cuda.current_stream(dev)

    def timed(n_h2d, n_d2h, reps=5, warm=True):
        if warm:
            timed(n_h2d, n_d2h, reps=1, warm=False)   # one untimed pass of the same copies first
        streams = [torch.cuda.Stream(device=dev) for _ in range(n_h2d + n_d2h)]
        jobs = [(d_in, h_in, nb_in, n_h2d, k) for k in range(n_h2d)] + \
               [(h_out, d_out, nb_out, n_d2h, k) for k in range(n_d2h)]
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(cur)
        for _ in range(reps):
            done = []
            for s, (dst, src, nb, parts, k) in zip(streams, jobs):
                s.wait_event(e0)
                with torch.cuda.stream(s):
                    lo, hi = nb * k // parts, nb * (k + 1) // parts
                    dst[lo:hi].copy_(src[lo:hi], non_blocking=True)
                    ev = torch.cuda.Event()
                    ev.record(s)
                    done.append(ev)
            for ev in done:
                cur.wait_event(ev)
        e1.record(cur)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / reps

    for n_h2d, n_d2h in [(1, 0), (2, 0), (4, 0), (0, 1), (0, 2), (0, 4), (1, 1), (2, 2)]:
        ms = timed(n_h2d, n_d2h)
        nbytes = (nb_in if n_h2d else 0) + (nb_out if n_d2h else 0)
        print(json.dumps({"link_probe": spec.name, "h2d_bytes": nb_in if n_h2d else 0,
                          "d2h_bytes": nb_out if n_d2h else 0, "h2d_streams": n_h2d, "d2h_streams": n_d2h,
                          "ms": round(ms, 3), "GB_per_s": round(nbytes / ms / 1e6, 1)}), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--workload", default="128k_gqa_student_t", choices=sorted(synth.WORKLOADS),
                    help="workload name (default: one 128K-token request, 32 q / 8 kv heads)")
    ap.add_argument("--impl", choices=["cosa", "reference"], default="cosa")
    ap.add_argument("--shard", choices=["heads", "replicas"], default="heads",
                    help="with N > 1 ranks: split the workload's kv heads (and their query heads) across the ranks "
                         "(one job, strong scaling), or run a replica of the whole workload on every rank (weak)")
    ap.add_argument("--kv-slice", default=None, metavar="A:B",
                    help="run only kv heads [A, B) of the workload and their query heads (a full-length slice, "
                         "for profiling); not a bench line of the whole workload")
    ap.add_argument("--gather-out", action="store_true",
                    help="with --shard heads: all-gather O over heads after the timed region (reported apart)")
    ap.add_argument("--gqa-union", action="store_true",
                    help="run the OSK as the GQA page-union kernel (COSA_FLAG_GQA_UNION: two query heads of a kv "
                         "group share one K stream); a measurement of that variant, not the bench line")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--clocks-log", default=None, help="also write the raw nvidia-smi clock samples here")
    ap.add_argument("--sweep", action="store_true",
                    help="time CoSA against the dense endpoint of the same kernel from 4K to 128K tokens")
    ap.add_argument("--ablation", choices=["remap", "jump", "topp", "union", "union-kernel"],
                    help="remap: skip ratio vs Delta with and without remapping over stage-1 budgets; "
                         "jump: physical jumps vs logical skipping of a binary mask; topp: the top-p stage-1 rule; "
                         "union: GQA page reuse rates; union-kernel: the GQA page-union OSK against the default OSK")
    ap.add_argument("--ablation-tokens", type=int, default=131072, help="context length of --ablation remap/topp")
    ap.add_argument("--copy-streams", type=int, default=1,
                    help="copy streams per direction in the end-to-end loop (each tensor split into that many chunks)")
    ap.add_argument("--link-probe", action="store_true",
                    help="host-link bandwidth of one step's input and output copies (the end-to-end floor)")
    args = ap.parse_args()
    if args.link_probe:
        return run_link_probe(args)
    if args.sweep:
        return run_sweep(args)
    if args.ablation:
        return run_ablation(args)
    spec = synth.spec_for(args.workload)
    delta = delta_for(args.workload)
    name = spec.name
    if args.impl == "reference":
        return run_reference(args, spec, name, delta)
    return run_cosa(args, spec, name, delta)


if __name__ == "__main__":
    sys.exit(main())

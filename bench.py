#!/usr/bin/env python3
"""Benchmark: one decode step of one HySparse2 Cross group (FA + selection, 5 SA layers).

Workload (synthetic, seeded): batch 64, context lengths uniform in [16384, 32768],
Hq=32, Hkv=4, head_dim=128, window w=128, top-k=1024, bf16 paged KV (page 64,
permuted block table), queries x @ W_Q with a distinct W_Q per layer, 32 needles
per sequence. One step = hs2_fa_select + 5 x hs2_sa_reuse on resident inputs.

Prints ONE JSON line (rank 0). ``--impl reference`` times the CPU oracle instead.
Multi-GPU (torchrun): every rank runs its own independent batch (weak scaling, no
data-path collective); the reported time is the max over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import signal
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "decode queries/s and HBM GB/s (FA+5 SA group); prefill tok/s and TFLOP/s"
WORKLOAD = "decode_bf16_b64_t16k-32k"
B, T_LO, T_HI, HQ, HKV, D, WIN, TOPK, NSA = 64, 16384, 32768, 32, 4, 128, 128, 1024, 5
FA_KERNEL = "fa_decode_mma_kernel"
FA_SOURCE = os.path.join(ROOT, "top_hs2_fa_gb300", "csrc", "fa_decode.cu")
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.json")
CLOCK_QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
               "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
               "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        j = json.load(open(p))
        return float(j["hbm_gbs"]), float(j["bf16_tflops"]), "measured"
    return 6800.0, 1900.0, "fallback"


def source_sha() -> str:
    return hashlib.sha256(open(FA_SOURCE, "rb").read()).hexdigest()[:16]


def recorded_traffic():
    """ncu DRAM bytes per FA-scan launch, if taken on the current kernel source."""
    try:
        j = json.load(open(TRAFFIC_FILE))
        e = j.get(WORKLOAD, {}).get(FA_KERNEL)
        if e and e.get("source_sha") == source_sha():
            return float(e["dram_bytes_per_launch"])
    except (OSError, ValueError, KeyError):
        pass
    return None


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons while the GPU is busy."""

    def __init__(self, gpu_index: int):
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={CLOCK_QUERY}", "--format=csv,noheader,nounits", "-lms", "200",
                 "-i", str(gpu_index)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.send_signal(signal.SIGTERM)
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        rows = []
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                rows.append(dict(sm=float(f[1]), smax=float(f[2]), power=float(f[3]), hw=f[5], hwt=f[6], swt=f[7],
                                 swp=f[8]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        smax = max(r["smax"] for r in rows)
        busy = [r for r in rows if r["power"] > 0] or rows
        busy = sorted(busy, key=lambda r: r["power"])[len(busy) // 2:] or busy  # upper half by power
        reasons = set()
        for r in rows:
            for key, name in (("hw", "hw_slowdown"), ("hwt", "hw_thermal_slowdown"), ("swt", "sw_thermal_slowdown"),
                              ("swp", "sw_power_cap")):
                if r[key].lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(r["sm"] for r in busy), "sm_max_mhz": smax,
                "power_w_max": max(r["power"] for r in rows), "samples": len(rows), "reasons": sorted(reasons)}


# ---------------------------------------------------------------------------- workload
def make_workload(seed: int):
    from top_hs2_fa_gb300 import workloads as W

    return W.decode_bf16_workload(seed=seed)


def algorithmic(grp):
    from top_hs2_fa_gb300 import counting as C

    m = C.decode_group_bytes(grp.kv.seq_len, HQ, HKV, D, WIN, TOPK, 2, NSA, grp.kv.max_pages)
    return m


# ---------------------------------------------------------------------------- reference arm
def cpu_baseline(grp, budget_s: float = 15.0):
    """The oracle as it stands, on the host cores, over the first sequences of the same
    workload until ``budget_s`` of CPU work has been spent."""
    done, elapsed = 0, 0.0
    while elapsed < budget_s and done < B:
        elapsed += oracle_sample_time_offset(grp, done, 1)
        done += 1
    return {"value": done / elapsed, "unit": "queries/s", "cores": os.cpu_count(), "kind": "oracle",
            "sample": f"{done} of the {B} decode queries (FA + 5 SA each), numpy float64 on host cores "
                      f"(BLAS threads = {os.cpu_count()})", "seconds": round(elapsed, 2)}


def oracle_sample_time_offset(grp, start: int, n: int):
    import numpy as np
    from oracle import hs2_oracle as O
    from top_hs2_fa_gb300 import workloads as W

    kv = grp.kv
    sel = list(range(start, start + n))
    sub = W.PagedKV(k=kv.k, v=kv.v, block_table=kv.block_table[sel], seq_len=kv.seq_len[sel], dtype=kv.dtype,
                    page=kv.page)
    t0 = time.perf_counter()
    _, _, idx, cnt = O.fa_decode(grp.q_fa[sel], sub, WIN, TOPK, grp.scale)
    for j in range(NSA):
        O.sa_decode(grp.q_sa[j][sel], sub, WIN, idx, cnt, grp.scale)
    return time.perf_counter() - t0


def run_reference(args, rank, world):
    if rank != 0:
        return 0
    grp = make_workload(seed=0)
    per_step = 2  # sequences per reference step (bounded sample of the workload)
    for i in range(args.warmup):
        oracle_sample_time_offset(grp, (i * per_step) % B, per_step)
    times = []
    for i in range(args.steps):
        times.append(oracle_sample_time_offset(grp, ((args.warmup + i) * per_step) % B, per_step))
    total = sum(times)
    value = args.steps * per_step / total
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "queries/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": WORKLOAD, "sample_per_step": f"{per_step} of {B} queries"},
            "cpu_baseline": {"value": value, "unit": "queries/s", "cores": os.cpu_count(), "kind": "oracle",
                             "sample": f"{per_step} decode queries (FA + 5 SA) per step, numpy float64"},
            "e2e": {"value": value, "unit": "queries/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------------------- GPU arm
def run_gpu(args, rank, world, local_rank):
    import numpy as np
    import torch

    from top_hs2_fa_gb300 import build as _build
    from top_hs2_fa_gb300 import hs2

    torch.cuda.set_device(local_rank)
    if rank == 0 or not os.path.exists(_build.LIB):
        _build.build()
    if world > 1:
        torch.distributed.barrier()
    hs2.load()
    dev = torch.device("cuda", local_rank)
    grp = make_workload(seed=rank)
    kv = grp.kv
    alg = algorithmic(grp)

    def up(a, bf16=False):
        t = torch.from_numpy(np.ascontiguousarray(a).view(np.int16) if bf16 else np.ascontiguousarray(a))
        t = t.to(dev)
        return t.view(torch.bfloat16) if bf16 else t

    dkv = hs2.KV(k=up(kv.k, True), v=up(kv.v, True), block_table=up(kv.block_table), seq_len=up(kv.seq_len))
    max_t = int(kv.seq_len.max())
    q_fa = up(grp.q_fa, True)
    q_sa = [up(q, True) for q in grp.q_sa]
    o = torch.empty((B, HQ, D), dtype=torch.float32, device=dev)
    lse = torch.empty((B, HQ), dtype=torch.float32, device=dev)
    idx = torch.empty((B, HKV, TOPK), dtype=torch.int32, device=dev)
    cnt = torch.empty((B, HKV), dtype=torch.int32, device=dev)
    o_sa = [torch.empty((B, HQ, D), dtype=torch.float32, device=dev) for _ in range(NSA)]
    ws_fa = torch.empty(hs2.hs2_fa_select_workspace(B, HQ, dkv, max_t, TOPK), dtype=torch.uint8, device=dev)
    ws_sa = torch.empty(hs2.hs2_sa_reuse_workspace(B, HQ, dkv, WIN, TOPK), dtype=torch.uint8, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream()
    launches_per_step = 2 + 2 * NSA

    def step(qf=q_fa, qs=q_sa, outs=None):
        oo = outs if outs is not None else (o, lse, idx, cnt, o_sa)
        hs2.hs2_fa_select(qf, dkv, WIN, TOPK, grp.scale, max_t=max_t, out=oo[:4], workspace=ws_fa, dev_err=err,
                          stream=stream)
        for j in range(NSA):
            hs2.hs2_sa_reuse(qs[j], dkv, WIN, oo[2], oo[3], TOPK, grp.scale, out=oo[4][j], workspace=ws_sa,
                             dev_err=err, stream=stream)

    sampler = ClockSampler(local_rank) if rank == 0 else None
    for _ in range(max(3, args.warmup)):
        step()
    # keep the GPU busy (untimed) long enough for the clock sampler to see it under load
    torch.cuda.synchronize()
    t_w = time.perf_counter()
    while time.perf_counter() - t_w < args.clock_warm_s:
        step()
        torch.cuda.synchronize()

    # FA-scan events, one pair per timed step
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    for a_, b_ in ev:
        a_.record(stream)
        b_.record(stream)
    t_start = torch.cuda.Event(enable_timing=True)
    t_stop = torch.cuda.Event(enable_timing=True)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    t_start.record(stream)
    for i in range(args.steps):
        hs2.hs2_profile_next(hs2.STAGE_FA_SCAN, ev[i][0], ev[i][1])
        step()
    t_stop.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    ms = t_start.elapsed_time(t_stop)
    fa_ms = sum(a_.elapsed_time(b_) for a_, b_ in ev) / args.steps

    # end to end through the C ABI with host buffers: H2D of the step's queries, table and
    # lengths from pinned memory, D2H of every layer's output and the index sets
    h_q = [torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).pin_memory() for x in [grp.q_fa, *grp.q_sa]]
    h_bt = torch.from_numpy(np.ascontiguousarray(kv.block_table)).pin_memory()
    h_sl = torch.from_numpy(np.ascontiguousarray(kv.seq_len)).pin_memory()
    d_q = [torch.empty(x.shape, dtype=torch.int16, device=dev) for x in h_q]
    h_out = [torch.empty((B, HQ, D), dtype=torch.float32).pin_memory() for _ in range(1 + NSA)]
    h_idx = torch.empty((B, HKV, TOPK), dtype=torch.int32).pin_memory()
    h_cnt = torch.empty((B, HKV), dtype=torch.int32).pin_memory()
    h2d = sum(x.numel() * 2 for x in h_q) + h_bt.numel() * 4 + h_sl.numel() * 4
    d2h = (1 + NSA) * B * HQ * D * 4 + h_idx.numel() * 4 + h_cnt.numel() * 4

    def e2e_step():
        for hq, dq in zip(h_q, d_q):
            dq.copy_(hq, non_blocking=True)
        dkv.block_table.copy_(h_bt, non_blocking=True)
        dkv.seq_len.copy_(h_sl, non_blocking=True)
        qs = [x.view(torch.bfloat16) for x in d_q]
        step(qs[0], qs[1:])
        h_out[0].copy_(o, non_blocking=True)
        for j in range(NSA):
            h_out[1 + j].copy_(o_sa[j], non_blocking=True)
        h_idx.copy_(idx, non_blocking=True)
        h_cnt.copy_(cnt, non_blocking=True)

    for _ in range(3):
        e2e_step()
    torch.cuda.synchronize()
    e_start = torch.cuda.Event(enable_timing=True)
    e_stop = torch.cuda.Event(enable_timing=True)
    e_start.record(stream)
    for _ in range(args.steps):
        e2e_step()
    e_stop.record(stream)
    torch.cuda.synchronize()
    e_ms = e_start.elapsed_time(e_stop)
    clocks = sampler.stop() if sampler else None
    bad = int(err.item())

    if world > 1:
        tt = torch.tensor([ms, e_ms, fa_ms], device=dev)
        torch.distributed.all_reduce(tt, op=torch.distributed.ReduceOp.MAX)
        ms, e_ms, fa_ms = [float(x) for x in tt.tolist()]
    if rank != 0:
        return 0
    hbm, tflops, src = peaks()
    per_step_s = ms / 1e3 / args.steps
    value = world * B / per_step_s
    fa_bytes = alg["fa"]
    achieved = fa_bytes / (fa_ms / 1e3) / 1e9
    traffic = recorded_traffic()
    line = {
        "metric": METRIC, "value": value, "unit": "queries/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": WORKLOAD, "batch": B, "seq_len": f"U[{T_LO},{T_HI}]", "Hq": HQ, "Hkv": HKV,
                   "head_dim": D, "window": WIN, "top_k": TOPK, "sa_layers": NSA, "page": 64,
                   "parallelism": "replicas" if world > 1 else "single",
                   "l2": "inputs larger than L2 (%.2f GB of K/V read per step)" % (fa_bytes / 1e9),
                   "hbm_gbs_step": alg["total"] / per_step_s / 1e9 * world,
                   "algorithmic_bytes_per_step": alg["total"]},
        "roofline": {"bound": "hbm", "kernel": FA_KERNEL, "achieved": achieved, "peak": hbm, "unit": "GB/s",
                     "frac": achieved / hbm, "traffic": traffic, "peak_source": f"hbm_gbs ({src})",
                     "algorithmic_bytes_per_launch": fa_bytes, "launch_ms": fa_ms},
        "e2e": {"value": world * B / (e_ms / 1e3 / args.steps), "unit": "queries/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clocks,
        "device_errors": bad,
    }
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(grp)
    print(json.dumps(line), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--clock-warm-s", type=float, default=1.0,
                    help="seconds of untimed steps before timing, so the clock sampler sees load")
    args = ap.parse_args()
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        return run_reference(args, rank, world)
    if world > 1:
        import torch

        torch.cuda.set_device(local_rank)
        torch.distributed.init_process_group("nccl")
    try:
        return run_gpu(args, rank, world, local_rank)
    finally:
        if world > 1:
            import torch

            torch.distributed.destroy_process_group()


if __name__ == "__main__":
    sys.exit(main())

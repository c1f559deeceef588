#!/usr/bin/env python3
"""Benchmark of the group-shared top-k sparse attention hot path on one GB300.

Default workload (the decode metric's configuration): one decode step of one
HySparse2 Cross group — batch 64, context lengths uniform in [16384, 32768],
Hq=32, Hkv=4, head_dim=128, window 128, top-k 1024, bf16 paged KV (page 64,
permuted block table), queries x @ W_Q with a distinct W_Q per layer, 32
needles per sequence. One step = hs2_fa_select + 5 x hs2_sa_reuse on resident
inputs. ``--workload`` selects the other configurations for measurement:
``prefill`` (n=32768), ``long_decode`` (batch 16 x 131072, 4 independent
caches, 24 layers), ``csa2`` (Full + Reindex indexer, 5 MQA layers), and the
decode variants ``decode_block`` (block-level selection, 64-position blocks),
``decode_fp8`` / ``decode_fp4`` (E4M3 / E2M1 paged KV), ``decode_append`` and
``long_decode_append`` (the current token's K/V appended inside the step).

Prints ONE JSON line (rank 0). ``--impl reference`` times the CPU oracle on a
bounded sample of the same workload. Under torchrun every rank runs its own
independent batch (weak scaling, no data-path collective); the reported time is
the max over ranks.
"""
from __future__ import annotations

import argparse
import dataclasses
import hashlib
import json
import os
import signal
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "decode queries/s and HBM GB/s (FA+5 SA group); prefill tok/s and TFLOP/s"
NSA = 5
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.json")
CLOCK_QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
               "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
               "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        j = json.load(open(p))
        return {"hbm": float(j["hbm_gbs"]), "bf16": float(j["bf16_tflops"]),
                "bf16_sustained": float(j.get("bf16_tflops_sustained", j["bf16_tflops"])), "src": "measured"}
    return {"hbm": 6800.0, "bf16": 1900.0, "bf16_sustained": 1700.0, "src": "fallback"}


def source_sha(paths) -> str:
    h = hashlib.sha256()
    for p in ([paths] if isinstance(paths, str) else paths):
        h.update(open(os.path.join(ROOT, p), "rb").read())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str, kernel: str, source: str):
    """ncu DRAM bytes per launch of the roofline kernel, if taken on the current kernel source."""
    try:
        e = json.load(open(TRAFFIC_FILE)).get(workload, {}).get(kernel)
        if e and e.get("source_sha") == source_sha(source):
            return float(e["dram_bytes_per_launch"])
    except (OSError, ValueError, KeyError):
        pass
    return None


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons while the GPU is busy."""

    def __init__(self, gpu_index: int):
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
        busy = sorted(rows, key=lambda r: r["power"])[len(rows) // 2:] or rows  # upper half by power draw
        reasons = set()
        for r in rows:
            for key, name in (("hw", "hw_slowdown"), ("hwt", "hw_thermal_slowdown"), ("swt", "sw_thermal_slowdown"),
                              ("swp", "sw_power_cap")):
                if r[key].lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(r["sm"] for r in busy), "sm_max_mhz": smax,
                "power_w_max": max(r["power"] for r in rows), "samples": len(rows), "reasons": sorted(reasons)}


def up(a, dev, bf16=False):
    import numpy as np
    import torch

    t = torch.from_numpy(np.ascontiguousarray(a).view(np.int16) if bf16 else np.ascontiguousarray(a)).to(dev)
    return t.view(torch.bfloat16) if bf16 else t


def pinned_copies(h_in, d_in, xs, dev, as_bf16):
    """Append pinned host buffers for inputs xs (uploaded into fresh device tensors)."""
    import numpy as np
    import torch

    for x in xs:
        if as_bf16:
            h_in.append(torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).pin_memory())
        else:
            h_in.append(torch.from_numpy(np.ascontiguousarray(x)).pin_memory())
        d_in.append(torch.empty(h_in[-1].shape, dtype=h_in[-1].dtype, device=dev))


class StepIO:
    """Host <-> device traffic of one end-to-end step, overlapped with the step's kernels.

    Inputs and outputs are tagged by the layer that reads or writes them. At the start of a
    step a copy stream (after everything before the step) uploads the inputs in tag order,
    recording an event per tag; a layer waits only for its own inputs (need). When a layer
    is done, the copy stream downloads its outputs (done) while later layers compute; the
    step ends when both streams have finished (end). Every byte still crosses every step."""

    def __init__(self, dev):
        import torch

        self.cs = torch.cuda.Stream(device=dev)
        self.inputs, self.outputs, self.ev_in, self.ev_out = {}, {}, {}, {}

    def add_in(self, tag, h, d):
        import torch

        self.inputs.setdefault(tag, []).append((h, d))
        self.ev_in.setdefault(tag, torch.cuda.Event())

    def add_out(self, tag, h, d):
        import torch

        self.outputs.setdefault(tag, []).append((h, d))
        self.ev_out.setdefault(tag, torch.cuda.Event())

    def begin(self, st):
        import torch

        self.cs.wait_stream(st)
        with torch.cuda.stream(self.cs):
            for tag, pairs in self.inputs.items():
                for h, d in pairs:
                    d.copy_(h, non_blocking=True)
                self.ev_in[tag].record(self.cs)

    def need(self, st, tag):
        if tag in self.ev_in:
            st.wait_event(self.ev_in[tag])

    def done(self, st, tag):
        import torch

        if tag not in self.outputs:
            return
        self.ev_out[tag].record(st)
        self.cs.wait_event(self.ev_out[tag])
        with torch.cuda.stream(self.cs):
            for h, d in self.outputs[tag]:
                h.copy_(d, non_blocking=True)

    def end(self, st):
        st.wait_stream(self.cs)


class _NoIO:
    def need(self, st, tag):
        pass

    def done(self, st, tag):
        pass


NO_IO = _NoIO()


# ============================================================================ scenarios
class Decode:
    """Decode step of one or more Cross groups: per group hs2_fa_select + 5 x hs2_sa_reuse."""

    roofline_kernel, bound = "fa_decode_mma_kernel", "hbm"
    roofline_source = ("top_hs2_fa_gb300/csrc/fa_decode.cu", "top_hs2_fa_gb300/csrc/mma_attn.cuh")
    unit = "queries/s"

    def __init__(self, name, B, t_lo, t_hi, groups, needles, qproj, sel_block=1, kv_fmt=None, append=None):
        self.name, self.B, self.t_lo, self.t_hi, self.groups = name, B, t_lo, t_hi, groups
        self.needles, self.qproj, self.sel_block, self.kv_fmt = needles, qproj, sel_block, kv_fmt
        self.kv_fp8 = kv_fmt is not None  # a low-precision cache (FP8 or FP4 codes with scales)
        # the current token's K/V enter the cache in the step: None (already there), "fused"
        # (each group's FA call appends its own rows) or "batched" (one hs2_kv_append for all
        # groups' caches before the first group runs)
        self.append = append
        # arithmetic type: an FP8 cache converts to f16 MMA operands (fp32 accumulation)
        self.dtype = "f16" if self.kv_fp8 else "bf16"
        self.Hq, self.Hkv, self.D, self.w, self.k = 32, 4, 128, 128, 1024

    def host_setup(self, seed):
        import numpy as np
        from top_hs2_fa_gb300 import workloads as W

        self.host = []
        for gi in range(self.groups):
            s_len, s_grp = np.random.SeedSequence([seed, gi]).spawn(2)
            lens = W.uniform_lengths(self.B, self.t_lo, self.t_hi, s_len)
            grp = W.decode_group(lens, self.Hq, self.Hkv, self.D, self.w, self.k, "bf16", s_grp, n_sa=NSA,
                                 needles=self.needles, qproj=self.qproj)
            if self.kv_fmt == "fp8":  # the same values stored as FP8 E4M3 with per-(page, KV head) scales
                grp.kv = W.quantize_kv_fp8(grp.kv)
            elif self.kv_fmt == "fp4":  # E2M1 with E4M3 scales of 16 channels and per-(page, KV head) scales
                grp.kv = W.quantize_kv_fp4(grp.kv)
            if self.append:  # the new token's K and V rows ([B][Hkv][d], bf16)
                rng = np.random.default_rng(np.random.SeedSequence([seed, gi, 7]))
                shape = (self.B, self.Hkv, self.D)
                grp.k_new = W.store(rng.standard_normal(shape, dtype=np.float32), "bf16")
                grp.v_new = W.store(rng.standard_normal(shape, dtype=np.float32), "bf16")
            self.host.append(grp)

    def setup(self, dev, seed):
        import torch
        from top_hs2_fa_gb300 import counting as C, hs2

        self.hs2 = hs2
        self.host_setup(seed)
        self.dev = []
        fa, total = [], 0
        for grp in self.host:
            kv = grp.kv
            bf = not self.kv_fp8
            fp4 = self.kv_fmt == "fp4"
            d = {"kv": hs2.KV(k=up(kv.k, dev, bf), v=up(kv.v, dev, bf), block_table=up(kv.block_table, dev),
                              seq_len=up(kv.seq_len, dev),
                              k_scale=None if bf else up(kv.k_scale, dev), v_scale=None if bf else up(kv.v_scale, dev),
                              k_sf=up(kv.k_sf, dev) if fp4 else None, v_sf=up(kv.v_sf, dev) if fp4 else None),
                 "max_t": int(kv.seq_len.max()), "q": [up(x, dev, True) for x in [grp.q_fa, *grp.q_sa]]}
            B = self.B
            d["o"] = [torch.empty((B, self.Hq, self.D), dtype=torch.float32, device=dev) for _ in range(1 + NSA)]
            d["lse"] = torch.empty((B, self.Hq), dtype=torch.float32, device=dev)
            d["idx"] = torch.empty((B, self.Hkv, self.k), dtype=torch.int32, device=dev)
            d["cnt"] = torch.empty((B, self.Hkv), dtype=torch.int32, device=dev)
            d["ws_fa"] = torch.empty(hs2.hs2_fa_select_workspace(B, self.Hq, d["kv"], d["max_t"], self.k),
                                     dtype=torch.uint8, device=dev)
            d["ws_sa"] = torch.empty(hs2.hs2_sa_reuse_workspace(B, self.Hq, d["kv"], self.w, self.k),
                                     dtype=torch.uint8, device=dev)
            if self.append:
                d["k_new"], d["v_new"] = up(grp.k_new, dev, True), up(grp.v_new, dev, True)
                total += 2 * grp.k_new.nbytes  # the rows written into the cache
            self.dev.append(d)
            elem = {"fp8": 1, "fp4": 0.5 + 1 / 16}.get(self.kv_fmt, 2)  # cache bytes per channel
            m = C.decode_group_bytes(kv.seq_len, self.Hq, self.Hkv, self.D, self.w, self.k, elem, NSA,
                                     kv.max_pages, q_elem=2)
            fa.append(m["fa"])
            total += m["total"]
        self.alg_per_launch = fa[0]  # the profiled launch is group 0's FA scan
        self.alg_total = total
        self.units_per_step = self.B
        # kernels per step, as the library reports them for these calls
        d0 = self.dev[0]
        per_group = (hs2.hs2_fa_select_launches(self.B, self.Hq, d0["kv"], d0["max_t"], self.w, self.k,
                                                sel_block=self.sel_block, append=self.append == "fused") +
                     NSA * hs2.hs2_sa_reuse_launches(self.B, self.Hq, d0["kv"], self.w, self.k))
        self.launches_per_step = self.groups * per_group + (1 if self.append == "batched" else 0)

    def step(self, stream, err, qs=None, profile=None, io=NO_IO):
        hs2 = self.hs2
        if self.append == "batched":  # every group's new entry in one launch
            io.need(stream, "append")
            hs2.hs2_kv_append([d["kv"] for d in self.dev], [d["k_new"] for d in self.dev],
                              [d["v_new"] for d in self.dev], dev_err=err, stream=stream)
        fused = self.append == "fused"
        for gi, d in enumerate(self.dev):
            q = qs[gi] if qs is not None else d["q"]
            if profile is not None and gi == 0:
                hs2.hs2_profile_next(hs2.STAGE_FA_SCAN, *profile)
            io.need(stream, ("fa", gi))
            hs2.hs2_fa_select(q[0], d["kv"], self.w, self.k, self.host[gi].scale, max_t=d["max_t"],
                              out=(d["o"][0], d["lse"], d["idx"], d["cnt"]), workspace=d["ws_fa"], dev_err=err,
                              stream=stream, sel_block=self.sel_block, k_new=d["k_new"] if fused else None,
                              v_new=d["v_new"] if fused else None)
            io.done(stream, ("fa", gi))
            for j in range(NSA):
                io.need(stream, ("sa", gi, j))
                # layers after the first follow an SA launch that wrote none of idx, cnt, table, lengths
                hs2.hs2_sa_reuse(q[1 + j], d["kv"], self.w, d["idx"], d["cnt"], self.k, self.host[gi].scale,
                                 out=d["o"][1 + j], workspace=d["ws_sa"], dev_err=err, stream=stream,
                                 overlap=j > 0)
                io.done(stream, ("sa", gi, j))

    def e2e_buffers(self, dev):
        """Pinned host inputs (every layer's queries, table, lengths, new rows) and outputs (all
        layers, indices), tagged by the layer that reads or writes them (StepIO)."""
        import torch

        self.h_in, self.d_in, self.h_out, self.d_out, self.q_views = [], [], [], [], []
        self.io = StepIO(dev)
        for gi, (grp, d) in enumerate(zip(self.host, self.dev)):
            n0 = len(self.d_in)
            pinned_copies(self.h_in, self.d_in, [grp.kv.block_table, grp.kv.seq_len], dev, False)
            self.d_in[-2:] = [d["kv"].block_table, d["kv"].seq_len]
            tags = [("fa", gi), ("fa", gi)]
            pinned_copies(self.h_in, self.d_in, [grp.q_fa, *grp.q_sa], dev, True)
            self.q_views.append([x.view(torch.bfloat16) for x in self.d_in[-(1 + NSA):]])
            tags += [("fa", gi)] + [("sa", gi, j) for j in range(NSA)]
            if self.append:  # the new token's rows arrive with the step's inputs
                pinned_copies(self.h_in, self.d_in, [grp.k_new, grp.v_new], dev, True)
                self.d_in[-2:] = [d["k_new"].view(torch.int16), d["v_new"].view(torch.int16)]
                tags += [("fa", gi) if self.append == "fused" else "append"] * 2
            for tag, h, dd in zip(tags, self.h_in[n0:], self.d_in[n0:]):
                self.io.add_in(tag, h, dd)
            outs = [(("fa", gi), d["o"][0]), (("fa", gi), d["idx"]), (("fa", gi), d["cnt"])]
            outs += [(("sa", gi, j), d["o"][1 + j]) for j in range(NSA)]
            for tag, t in outs:
                self.h_out.append(torch.empty(t.shape, dtype=t.dtype).pin_memory())
                self.d_out.append(t)
                self.io.add_out(tag, self.h_out[-1], t)
        if self.append == "batched":  # the append runs first: its rows lead the uploads
            first = self.io.inputs.pop("append")
            self.io.inputs = {"append": first, **self.io.inputs}

    def config(self):
        return {"workload": self.name, "batch": self.B,
                "seq_len": f"U[{self.t_lo},{self.t_hi}]" if self.t_lo != self.t_hi else self.t_lo,
                "groups": self.groups, "Hq": self.Hq, "Hkv": self.Hkv, "head_dim": self.D, "window": self.w,
                "top_k": self.k, "sa_layers_per_group": NSA, "page": 64,
                "kv_dtype": {"fp8": "fp8_e4m3 (scale per page and KV head)",
                             "fp4": "fp4_e2m1 (e4m3 scale per 16 channels, scale per page and KV head)"}.get(
                                 self.kv_fmt, "bf16"),
                "selection": "token" if self.sel_block == 1 else f"blocks of {self.sel_block}",
                "kv_append": self.append or "none"}

    def oracle_sample(self, budget_s):
        """Oracle FA + 5 SA per query (in every group) on the host cores, query by query."""
        from oracle import hs2_oracle as O
        from top_hs2_fa_gb300 import workloads as W

        done, elapsed = 0, 0.0
        while done < self.B and (done == 0 or elapsed < budget_s):
            t0 = time.perf_counter()
            for grp in self.host:
                kv, sel = grp.kv, [done]
                sub = dataclasses.replace(kv, block_table=kv.block_table[sel], seq_len=kv.seq_len[sel])
                if self.append:
                    sub = O.kv_append(sub, grp.k_new[sel], grp.v_new[sel])
                _, _, idx, cnt = O.fa_decode(grp.q_fa[sel], sub, self.w, self.k, grp.scale, blk=self.sel_block)
                for j in range(NSA):
                    O.sa_decode(grp.q_sa[j][sel], sub, self.w, idx, cnt, grp.scale)
            elapsed += time.perf_counter() - t0
            done += 1
        return done, elapsed, f"{done} of the {self.B} queries (FA + 5 SA in each of {self.groups} group(s))"


class Prefill:
    """Prefill of one sequence: hs2_fa_select (causal FA + per-row top-k) + 5 x hs2_sa_reuse."""

    roofline_kernel, roofline_source, bound = "fa_prefill_fwd_kernel", "top_hs2_fa_gb300/csrc/fa_prefill.cu", "tensor"
    unit = "tok/s"

    def __init__(self, n=32768):
        self.name = f"prefill_bf16_n{n}"
        self.n, self.Hq, self.Hkv, self.D, self.w, self.k = n, 32, 4, 128, 128, 1024

    def host_setup(self, seed):
        from top_hs2_fa_gb300 import workloads as W

        self.host = [W.prefill_group(self.n, self.Hq, self.Hkv, self.D, self.w, self.k, "bf16", seed, n_sa=NSA,
                                     rho=0.999)]

    def setup(self, dev, seed):
        import torch
        from top_hs2_fa_gb300 import counting as C, hs2

        self.hs2 = hs2
        self.host_setup(seed)
        g, n = self.host[0], self.n
        kv = g.kv
        d = {"kv": hs2.KV(k=up(kv.k, dev, True), v=up(kv.v, dev, True), block_table=up(kv.block_table, dev),
                          seq_len=up(kv.seq_len, dev)), "q": [up(x, dev, True) for x in [g.q_fa, *g.q_sa]]}
        d["o"] = [torch.empty((n, self.Hq, self.D), dtype=torch.float32, device=dev) for _ in range(1 + NSA)]
        d["lse"] = torch.empty((n, self.Hq), dtype=torch.float32, device=dev)
        d["idx"] = torch.empty((n, self.Hkv, self.k), dtype=torch.int32, device=dev)
        d["cnt"] = torch.empty((n, self.Hkv), dtype=torch.int32, device=dev)
        d["ws_fa"] = torch.empty(hs2.hs2_fa_select_workspace(n, self.Hq, d["kv"], n, self.k, True), dtype=torch.uint8,
                                 device=dev)
        d["ws_sa"] = torch.empty(hs2.hs2_sa_reuse_workspace(n, self.Hq, d["kv"], self.w, self.k, True),
                                 dtype=torch.uint8, device=dev)
        self.dev = [d]
        f = C.prefill_flops(n, self.Hq, self.D, self.w, self.k)
        self.alg_per_launch = f["fa"]
        self.alg_total = f["fa"] + NSA * f["sa_per_layer"]
        self.units_per_step = n
        self.launches_per_step = (hs2.hs2_fa_select_launches(n, self.Hq, d["kv"], n, self.w, self.k, prefill=True) +
                                  NSA * hs2.hs2_sa_reuse_launches(n, self.Hq, d["kv"], self.w, self.k, prefill=True))

    def step(self, stream, err, qs=None, profile=None, io=NO_IO):
        hs2, d, g = self.hs2, self.dev[0], self.host[0]
        q = qs[0] if qs is not None else d["q"]
        if profile is not None:
            hs2.hs2_profile_next(hs2.STAGE_FA_SCAN, *profile)
        io.need(stream, ("fa", 0))
        hs2.hs2_fa_select(q[0], d["kv"], self.w, self.k, g.scale, prefill=True,
                          out=(d["o"][0], d["lse"], d["idx"], d["cnt"]), workspace=d["ws_fa"], dev_err=err,
                          stream=stream)
        io.done(stream, ("fa", 0))
        for j in range(NSA):
            io.need(stream, ("sa", 0, j))
            hs2.hs2_sa_reuse(q[1 + j], d["kv"], self.w, d["idx"], d["cnt"], self.k, g.scale, prefill=True,
                             out=d["o"][1 + j], workspace=d["ws_sa"], dev_err=err, stream=stream)
            io.done(stream, ("sa", 0, j))

    e2e_buffers = Decode.e2e_buffers
    append = None
    groups = 1

    def config(self):
        return {"workload": self.name, "n": self.n, "Hq": self.Hq, "Hkv": self.Hkv, "head_dim": self.D,
                "window": self.w, "top_k": self.k, "sa_layers": NSA, "keys": "AR(1) drifting mean, rho=0.999",
                "fa_tflop": 4.0 * self.D * self.Hq * self.n * (self.n + 1) / 2 / 1e12}

    def oracle_sample(self, budget_s):
        import numpy as np
        from oracle import hs2_oracle as O

        g = self.host[0]
        rng = np.random.default_rng(5)
        full_idx = np.full((self.n, self.Hkv, self.k), -1, np.int32)
        full_cnt = np.zeros((self.n, self.Hkv), np.int32)
        done, elapsed = 0, 0.0
        while done < 64 and (done == 0 or elapsed < budget_s):
            i = int(rng.integers(0, self.n))
            t0 = time.perf_counter()
            _, _, idx, cnt = O.fa_prefill_rows(g.q_fa, g.kv, [i], self.w, self.k, g.scale)
            full_idx[i], full_cnt[i] = idx[0], cnt[0]
            for j in range(NSA):
                O.sa_prefill_rows(g.q_sa[j], g.kv, [i], self.w, full_idx, full_cnt, g.scale)
            elapsed += time.perf_counter() - t0
            done += 1
        return done, elapsed, f"{done} uniformly drawn rows (FA + top-k + 5 SA each) of the n={self.n} prefill"


class Csa2:
    """CSA2 decode group: Full indexer -> SA, Reindex -> SA, 3 x Reuse SA (MQA, w = 0)."""

    roofline_kernel, roofline_source, bound = "lightning_scan_kernel", "top_hs2_fa_gb300/csrc/indexer.cu", "hbm"
    unit = "queries/s"
    groups = 1

    def __init__(self):
        self.name = "csa2_decode_bf16_b8_t131072"
        self.B, self.t, self.Hq, self.D, self.k_top, self.max_blocks = 8, 131072, 32, 128, 512, 2048

    def host_setup(self, seed):
        from top_hs2_fa_gb300 import workloads as W

        self.host = [W.csa2_group([self.t] * self.B, Hq=self.Hq, d=self.D, Hi=64, di=128, k_top=self.k_top, blk=8,
                                  max_blocks=self.max_blocks, n_reuse=3, needles=32, seed=seed)]

    def setup(self, dev, seed):
        import torch
        from top_hs2_fa_gb300 import counting as C, hs2

        self.hs2 = hs2
        self.host_setup(seed)
        g, B = self.host[0], self.B
        d = {"kv": hs2.KV(k=up(g.kv.k, dev, True), v=up(g.kv.v, dev, True), block_table=up(g.kv.block_table, dev),
                          seq_len=up(g.kv.seq_len, dev)),
             "kidx": hs2.KV(k=up(g.kidx.k, dev, True), v=None, block_table=up(g.kidx.block_table, dev),
                            seq_len=up(g.kidx.seq_len, dev)),
             "qi": [up(x, dev, True) for x in g.q_idx], "wi": [up(x, dev) for x in g.w_idx],
             "q": [up(x, dev, True) for x in g.q_main]}
        d["o"] = [torch.empty((B, self.Hq, self.D), dtype=torch.float32, device=dev) for _ in range(5)]
        d["pool"] = torch.empty((B, self.max_blocks), dtype=torch.int32, device=dev)
        d["pcnt"] = torch.empty((B,), dtype=torch.int32, device=dev)
        d["idx"] = [torch.empty((B, 1, self.k_top), dtype=torch.int32, device=dev) for _ in range(2)]
        d["cnt"] = [torch.empty((B, 1), dtype=torch.int32, device=dev) for _ in range(2)]
        d["ws_i"] = torch.empty(max(hs2.hs2_hier_reindex_workspace(m, 64, d["kidx"], self.t, self.k_top, 8,
                                                                   self.max_blocks) for m in (0, 1)),
                                dtype=torch.uint8, device=dev)
        d["ws_sa"] = torch.empty(hs2.hs2_sa_reuse_workspace(B, self.Hq, d["kv"], 0, self.k_top), dtype=torch.uint8,
                                 device=dev)
        self.dev = [d]
        m = C.csa2_decode_bytes([self.t] * B, self.D, 128, 2, self.k_top, self.max_blocks * 8, 5)
        self.alg_per_launch = m["full"]
        self.alg_total = m["total"]
        self.units_per_step = B
        # Full: indexer scan + one launch for the position and block selections; Reindex: scan +
        # selection; 5 SA calls
        self.launches_per_step = 2 + 2 + 5 * hs2.hs2_sa_reuse_launches(B, self.Hq, d["kv"], 0, self.k_top)

    def step(self, stream, err, qs=None, profile=None, io=NO_IO):
        hs2, d, g = self.hs2, self.dev[0], self.host[0]
        q = qs[0] if qs is not None else d["q"]
        if profile is not None:
            hs2.hs2_profile_next(hs2.STAGE_INDEXER, *profile)
        for mode in (hs2.FULL, hs2.REINDEX):
            io.need(stream, ("layer", mode))
            hs2.hs2_hier_reindex(mode, d["qi"][mode], d["wi"][mode], d["kidx"], self.k_top, 8, self.max_blocks,
                                 pool_blocks=d["pool"], pool_cnt=d["pcnt"], max_t=self.t,
                                 out=(d["idx"][mode].view(self.B, self.k_top), d["cnt"][mode].view(self.B)),
                                 workspace=d["ws_i"], dev_err=err, stream=stream)
            hs2.hs2_sa_reuse(q[mode], d["kv"], 0, d["idx"][mode], d["cnt"][mode], self.k_top, g.scale,
                             out=d["o"][mode], workspace=d["ws_sa"], dev_err=err, stream=stream)
            io.done(stream, ("layer", mode))
        for j in range(2, 5):  # Reuse layers read the Reindex layer's indices
            io.need(stream, ("layer", j))
            hs2.hs2_sa_reuse(q[j], d["kv"], 0, d["idx"][1], d["cnt"][1], self.k_top, g.scale, out=d["o"][j],
                             workspace=d["ws_sa"], dev_err=err, stream=stream, overlap=True)
            io.done(stream, ("layer", j))

    def e2e_buffers(self, dev):
        import torch

        g, d = self.host[0], self.dev[0]
        self.h_in, self.d_in, self.h_out, self.d_out = [], [], [], []
        self.io = StepIO(dev)
        pinned_copies(self.h_in, self.d_in, g.q_idx, dev, True)
        self.d_in[-2:] = [t.view(torch.int16) for t in d["qi"]]
        pinned_copies(self.h_in, self.d_in, g.w_idx, dev, False)
        self.d_in[-2:] = d["wi"]
        pinned_copies(self.h_in, self.d_in, g.q_main, dev, True)
        self.q_views = [[x.view(torch.bfloat16) for x in self.d_in[-5:]]]
        tags = [("layer", 0), ("layer", 1)] * 2 + [("layer", j) for j in range(5)]
        order = [0, 2, 4, 1, 3, 5, 6, 7, 8]  # by the layer that needs them: Full's first
        for i in order:
            self.io.add_in(tags[i], self.h_in[i], self.d_in[i])
        outs = [(("layer", j), d["o"][j]) for j in range(5)]
        outs += [(("layer", m), d["idx"][m]) for m in range(2)] + [(("layer", m), d["cnt"][m]) for m in range(2)]
        outs += [(("layer", 1), d["pool"]), (("layer", 1), d["pcnt"])]
        for tag, t in outs:
            self.h_out.append(torch.empty(t.shape, dtype=t.dtype).pin_memory())
            self.d_out.append(t)
            self.io.add_out(tag, self.h_out[-1], t)

    def config(self):
        return {"workload": self.name, "batch": self.B, "seq_len": self.t, "Hq": self.Hq, "Hkv": 1,
                "head_dim": self.D, "indexer_heads": 64, "indexer_dim": 128, "top_k": self.k_top, "block": 8,
                "max_blocks": self.max_blocks, "layers": "Full, Reindex, 3 x Reuse"}

    def oracle_sample(self, budget_s):
        from oracle import hs2_oracle as O
        from top_hs2_fa_gb300 import workloads as W

        g = self.host[0]
        done, elapsed = 0, 0.0
        while done < self.B and (done == 0 or elapsed < budget_s):
            sel = [done]
            sub_i = W.PagedKV(k=g.kidx.k, v=None, block_table=g.kidx.block_table[sel], seq_len=g.kidx.seq_len[sel],
                              dtype="bf16")
            sub = W.PagedKV(k=g.kv.k, v=g.kv.v, block_table=g.kv.block_table[sel], seq_len=g.kv.seq_len[sel],
                            dtype="bf16")
            t0 = time.perf_counter()
            fi, fc, pool, pc = O.indexer_full(g.q_idx[0][sel], g.w_idx[0][sel], sub_i, self.k_top, 8, self.max_blocks)
            ri, rc = O.indexer_reindex(g.q_idx[1][sel], g.w_idx[1][sel], sub_i, self.k_top, 8, pool, pc)
            O.sa_decode(g.q_main[0][sel], sub, 0, fi[:, None], fc[:, None], g.scale)
            for j in range(1, 5):
                O.sa_decode(g.q_main[j][sel], sub, 0, ri[:, None], rc[:, None], g.scale)
            elapsed += time.perf_counter() - t0
            done += 1
        return done, elapsed, f"{done} of the {self.B} queries (Full, Reindex and 5 SA layers each)"


SCENARIOS = {
    "decode": lambda: Decode("decode_bf16_b64_t16k-32k", 64, 16384, 32768, 1, 32, True),
    "long_decode": lambda: Decode("long_decode_bf16_b16_t131072_x4", 16, 131072, 131072, 4, 64, False),
    # the decode workload with HySparse's first-version block-level selection (16 blocks of 64)
    "decode_block": lambda: Decode("decode_bf16_b64_t16k-32k_block64", 64, 16384, 32768, 1, 32, True, sel_block=64),
    # the decode workload with its cache stored as FP8 E4M3 (queries bf16)
    "decode_fp8": lambda: Decode("decode_fp8kv_b64_t16k-32k", 64, 16384, 32768, 1, 32, True, kv_fmt="fp8"),
    # ... and as FP4 E2M1 with an E4M3 scale per 16 channels
    "decode_fp4": lambda: Decode("decode_fp4kv_b64_t16k-32k", 64, 16384, 32768, 1, 32, True, kv_fmt="fp4"),
    # decode with the current token's K/V appended by the FA call itself
    "decode_append": lambda: Decode("decode_bf16_b64_t16k-32k_append", 64, 16384, 32768, 1, 32, True,
                                    append="fused"),
    # the four Cross-group caches: one batched append of the new token, then each group in turn
    "long_decode_append": lambda: Decode("long_decode_bf16_b16_t131072_x4_append", 16, 131072, 131072, 4, 64, False,
                                         append="batched"),
    "prefill": lambda: Prefill(32768),
    "csa2": lambda: Csa2(),
}


# ============================================================================ arms
def run_reference(args, rank, world):
    """The oracle on the host cores, on bounded samples of the selected workload."""
    if rank != 0:
        return 0
    sc = SCENARIOS[args.workload]()
    sc.host_setup(0)
    for _ in range(args.warmup):
        sc.oracle_sample(0.0)
    tot_units, tot_s, sample = 0, 0.0, ""
    for _ in range(args.steps):
        u, s, sample = sc.oracle_sample(2.0)
        tot_units += u
        tot_s += s
    value = tot_units / tot_s
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": sc.unit, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * tot_s / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": sc.config(),
            "cpu_baseline": {"value": value, "unit": sc.unit, "cores": os.cpu_count(), "kind": "oracle",
                             "sample": f"per step: {sample}; numpy float64"},
            "e2e": {"value": value, "unit": sc.unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def graph_of(body, stream):
    """Capture body() (stream-ordered library calls and copies) once as a CUDA graph; return
    a function that replays it on `stream`."""
    import torch

    body()  # warm on the capture path: kernel attributes set, nothing allocated later
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, capture_error_mode="relaxed"):
        body()
    torch.cuda.synchronize()

    def replay():
        with torch.cuda.stream(stream):
            g.replay()

    return replay


def max_over_ranks(values, world, device=None):
    """Element-wise max of per-rank timings over all ranks (the slowest rank sets the time)."""
    if world <= 1:
        return [float(v) for v in values]
    import torch

    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return [float(x) for x in t.tolist()]


def whole_job_rate(world, units_per_step, ms_total, steps):
    """Units per second of the whole job: every rank processes its own batch (weak scaling)."""
    return world * units_per_step / (ms_total / 1e3 / steps)


def run_gpu(args, rank, world, local_rank):
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
    sc = SCENARIOS[args.workload]()
    sc.setup(dev, seed=rank)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream()

    sampler = ClockSampler(local_rank) if rank == 0 else None
    for _ in range(max(3, args.warmup)):
        sc.step(stream, err)
    torch.cuda.synchronize()
    t_w = time.perf_counter()
    while time.perf_counter() - t_w < args.clock_warm_s:  # untimed: lets the clock sampler see load
        sc.step(stream, err)
        torch.cuda.synchronize()

    # the roofline kernel's launch time: eager steps, one event pair per step around it
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    for a_, b_ in ev:
        a_.record(stream)
        b_.record(stream)
    torch.cuda.synchronize()
    for i in range(args.steps):
        sc.step(stream, err, profile=ev[i])
    torch.cuda.synchronize()
    k_ms = sum(a_.elapsed_time(b_) for a_, b_ in ev) / args.steps

    # the step itself: captured once as a CUDA graph and replayed (no per-launch gaps)
    run_step = graph_of(lambda: sc.step(torch.cuda.current_stream(), err), stream) if args.graph \
        else (lambda: sc.step(stream, err))
    for _ in range(3):
        run_step()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    t0.record(stream)
    for i in range(args.steps):
        run_step()
    t1.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    ms = t0.elapsed_time(t1)

    # end to end through the C ABI with host buffers: H2D of every layer's queries (and the
    # indexer inputs, tables, lengths) from pinned memory, D2H of every output and index set
    sc.e2e_buffers(dev)
    h2d = sum(x.numel() * x.element_size() for x in sc.h_in)
    d2h = sum(x.numel() * x.element_size() for x in sc.h_out)

    def e2e_body():
        # uploads and downloads on a copy stream, each layer waiting for its own inputs and
        # its outputs leaving while later layers run (StepIO)
        st = torch.cuda.current_stream()
        sc.io.begin(st)
        sc.step(st, err, qs=sc.q_views, io=sc.io)
        sc.io.end(st)

    e2e_step = graph_of(e2e_body, stream) if args.graph else e2e_body

    for _ in range(3):
        e2e_step()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize()
    e_ms = e0.elapsed_time(e1)
    clocks = sampler.stop() if sampler else None
    bad = int(err.item())

    ms, e_ms, k_ms = max_over_ranks([ms, e_ms, k_ms], world, dev)
    if rank != 0:
        return 0
    pk = peaks()
    per_step_s = ms / 1e3 / args.steps
    value = whole_job_rate(world, sc.units_per_step, ms, args.steps)
    cfg = sc.config()
    cfg["parallelism"] = f"replicas x{world}" if world > 1 else "single"
    cfg["cuda_graph"] = bool(args.graph)
    if sc.bound == "hbm":
        achieved = sc.alg_per_launch / (k_ms / 1e3) / 1e9
        peak, unit, psrc = pk["hbm"], "GB/s", f"hbm_gbs ({pk['src']})"
        traffic = recorded_traffic(sc.name, sc.roofline_kernel, sc.roofline_source)
        cfg["l2"] = "inputs larger than L2 (%.2f GB read by the roofline kernel per step)" % (sc.alg_per_launch / 1e9)
        cfg["hbm_gbs_step"] = world * sc.alg_total / per_step_s / 1e9
        cfg["algorithmic_bytes_per_step"] = sc.alg_total
    else:
        achieved = sc.alg_per_launch / (k_ms / 1e3) / 1e12
        peak, unit = pk["bf16_sustained"], "TFLOP/s"
        psrc = f"bf16_tflops_sustained ({pk['src']}; kernel timed inside a long step)"
        traffic = None
        cfg["l2"] = "sequence K/V (64 MB) L2-resident by design; queries and outputs larger than L2"
        cfg["algorithmic_tflop_per_step"] = sc.alg_total / 1e12
        cfg["tflops_step"] = world * sc.alg_total / per_step_s / 1e12
    line = {
        "metric": METRIC, "value": value, "unit": sc.unit, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": getattr(sc, "dtype", "bf16"), "data": "synthetic", "config": cfg,
        "roofline": {"bound": sc.bound, "kernel": sc.roofline_kernel, "achieved": achieved, "peak": peak, "unit": unit,
                     "frac": achieved / peak, "traffic": traffic, "peak_source": psrc,
                     "algorithmic_per_launch": sc.alg_per_launch, "launch_ms": k_ms},
        "e2e": {"value": whole_job_rate(world, sc.units_per_step, e_ms, args.steps), "unit": sc.unit,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": sc.launches_per_step * args.steps,
        "clocks": clocks,
        "device_errors": bad,
    }
    if not args.no_cpu_baseline:
        u, s, sample = sc.oracle_sample(15.0)
        line["cpu_baseline"] = {"value": u / s, "unit": sc.unit, "cores": os.cpu_count(), "kind": "oracle",
                                "sample": f"{sample}; numpy float64 on the host cores (BLAS threads = "
                                          f"{os.cpu_count()})", "seconds": round(s, 2)}
    print(json.dumps(line), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(SCENARIOS), default="decode")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--graph", action=argparse.BooleanOptionalAction, default=True,
                    help="replay each step as a captured CUDA graph (default) or launch eagerly")
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

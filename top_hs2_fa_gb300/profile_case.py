"""Run a few steps of one group at a chosen (small) size, for profilers.

A self-contained driver for ``ncu -k regex:<kernel>`` captures of one workload shape:

  decode   FA + selection, then SA layers (``--batch`` sequences, lengths in [t-lo, t-hi];
           ``--kv-fp8``: the KV stored as FP8 E4M3)
  prefill  causal FA + per-row selection, then SA layers over ``--n`` rows
  csa2     Full indexer + SA, Reindex indexer + SA (``--batch`` sequences of ``--t`` keys)

e.g. ``python -m top_hs2_fa_gb300.profile_case --mode prefill --n 8192 --steps 1``.
"""
from __future__ import annotations

import argparse

import numpy as np
import torch

from . import build, hs2, workloads as W


def up(x, bf16=False):
    t = torch.from_numpy(np.ascontiguousarray(x).view(np.int16) if bf16 else np.ascontiguousarray(x)).cuda()
    return t.view(torch.bfloat16) if bf16 else t


def run_decode(a) -> float:
    grp = W.decode_bf16_workload(seed=0, B=a.batch, t_lo=a.t_lo, t_hi=a.t_hi, qproj=False)
    if a.kv_fp8:
        grp.kv = W.quantize_kv_fp8(grp.kv)
    kv = grp.kv
    if a.kv_fp8:
        dkv = hs2.KV(k=up(kv.k), v=up(kv.v), block_table=up(kv.block_table), seq_len=up(kv.seq_len),
                     k_scale=up(kv.k_scale), v_scale=up(kv.v_scale))
    else:
        dkv = hs2.KV(k=up(kv.k, True), v=up(kv.v, True), block_table=up(kv.block_table), seq_len=up(kv.seq_len))
    q = up(grp.q_fa, True)
    qs = [up(x, True) for x in grp.q_sa[:a.sa_layers]]
    max_t = int(kv.seq_len.max())
    for _ in range(a.steps):
        o, lse, idx, cnt = hs2.hs2_fa_select(q, dkv, grp.w, grp.k, grp.scale, max_t=max_t)
        for x in qs:
            hs2.hs2_sa_reuse(x, dkv, grp.w, idx, cnt, grp.k, grp.scale)
    return float(o.abs().mean())


def run_prefill(a) -> float:
    grp = W.prefill_group(a.n, 32, 4, 128, w=128, k=1024, dtype="bf16", seed=0, n_sa=a.sa_layers, rho=0.999)
    kv = grp.kv
    dkv = hs2.KV(k=up(kv.k, True), v=up(kv.v, True), block_table=up(kv.block_table), seq_len=up(kv.seq_len))
    q = up(grp.q_fa, True)
    qs = [up(x, True) for x in grp.q_sa[:a.sa_layers]]
    for _ in range(a.steps):
        o, lse, idx, cnt = hs2.hs2_fa_select(q, dkv, grp.w, grp.k, grp.scale, prefill=True)
        for x in qs:
            hs2.hs2_sa_reuse(x, dkv, grp.w, idx, cnt, grp.k, grp.scale, prefill=True)
    return float(o.abs().mean())


def run_csa2(a) -> float:
    B, k_top, max_blocks = a.batch, 512, 2048
    g = W.csa2_group([a.t] * B, Hq=32, d=128, Hi=64, di=128, k_top=k_top, blk=8, max_blocks=max_blocks, n_reuse=3,
                     needles=32, seed=0)
    dkv = hs2.KV(k=up(g.kv.k, True), v=up(g.kv.v, True), block_table=up(g.kv.block_table), seq_len=up(g.kv.seq_len))
    kidx = hs2.KV(k=up(g.kidx.k, True), v=None, block_table=up(g.kidx.block_table), seq_len=up(g.kidx.seq_len))
    qi = [up(x, True) for x in g.q_idx]
    wi = [up(x) for x in g.w_idx]
    q = [up(x, True) for x in g.q_main]
    pool = torch.empty((B, max_blocks), dtype=torch.int32, device="cuda")
    pcnt = torch.empty((B,), dtype=torch.int32, device="cuda")
    for _ in range(a.steps):
        for mode in (hs2.FULL, hs2.REINDEX):
            idx, cnt, _, _ = hs2.hs2_hier_reindex(mode, qi[mode], wi[mode], kidx, k_top, 8, max_blocks,
                                                  pool_blocks=pool, pool_cnt=pcnt, max_t=a.t)
            o = hs2.hs2_sa_reuse(q[mode], dkv, 0, idx.view(B, 1, k_top), cnt.view(B, 1), k_top, g.scale)
    return float(o.abs().mean())


def main() -> None:
    ap = argparse.ArgumentParser()
    ap.add_argument("--mode", choices=("decode", "prefill", "csa2"), default="decode")
    ap.add_argument("--batch", type=int, default=8)
    ap.add_argument("--t-lo", type=int, default=16384)
    ap.add_argument("--t-hi", type=int, default=32768)
    ap.add_argument("--n", type=int, default=8192, help="prefill rows")
    ap.add_argument("--t", type=int, default=131072, help="csa2 keys per sequence")
    ap.add_argument("--steps", type=int, default=3)
    ap.add_argument("--sa-layers", type=int, default=5)
    ap.add_argument("--kv-fp8", action="store_true", help="decode: FP8 E4M3 paged KV")
    a = ap.parse_args()
    build.build()
    v = {"decode": run_decode, "prefill": run_prefill, "csa2": run_csa2}[a.mode](a)
    torch.cuda.synchronize()
    print("ok", v)


if __name__ == "__main__":
    main()

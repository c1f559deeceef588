"""Run a few decode steps of one group (FA + selection, SA layers) at a chosen size.

A small, self-contained driver for profilers (e.g. ``ncu -k regex:fa_decode``):
``python -m top_hs2_fa_gb300.profile_case --batch 8 --steps 3``.
"""
from __future__ import annotations

import argparse

import numpy as np
import torch

from . import build, hs2, workloads as W


def main() -> None:
    ap = argparse.ArgumentParser()
    ap.add_argument("--batch", type=int, default=8)
    ap.add_argument("--t-lo", type=int, default=16384)
    ap.add_argument("--t-hi", type=int, default=32768)
    ap.add_argument("--steps", type=int, default=3)
    ap.add_argument("--sa-layers", type=int, default=5)
    a = ap.parse_args()
    build.build()
    grp = W.decode_bf16_workload(seed=0, B=a.batch, t_lo=a.t_lo, t_hi=a.t_hi, qproj=False)
    kv = grp.kv

    def up(x, bf16=False):
        t = torch.from_numpy(np.ascontiguousarray(x).view(np.int16) if bf16 else np.ascontiguousarray(x)).cuda()
        return t.view(torch.bfloat16) if bf16 else t

    dkv = hs2.KV(k=up(kv.k, True), v=up(kv.v, True), block_table=up(kv.block_table), seq_len=up(kv.seq_len))
    q = up(grp.q_fa, True)
    qs = [up(x, True) for x in grp.q_sa[:a.sa_layers]]
    max_t = int(kv.seq_len.max())
    for _ in range(a.steps):
        o, lse, idx, cnt = hs2.hs2_fa_select(q, dkv, grp.w, grp.k, grp.scale, max_t=max_t)
        for x in qs:
            hs2.hs2_sa_reuse(x, dkv, grp.w, idx, cnt, grp.k, grp.scale)
    torch.cuda.synchronize()
    print("ok", float(o.abs().mean()))


if __name__ == "__main__":
    main()

"""Helpers shared by the tests: device upload of seeded workloads and the acceptance rules."""
from __future__ import annotations

import numpy as np

TOL_BF16 = 2e-2  # max-abs error on outputs, bf16 inputs, fp32 accumulation
TOL_F32 = 1e-4   # max-abs error on outputs, fp32 inputs
SCORE_BAND = 1e-3  # relative band around the k-th oracle score where set differences are allowed


def tol(dtype: str) -> float:
    return TOL_BF16 if dtype == "bf16" else TOL_F32


def to_torch(arr: np.ndarray, dtype: str, device="cuda"):
    import torch

    if dtype == "bf16" and arr.dtype == np.uint16:
        return torch.from_numpy(np.ascontiguousarray(arr).view(np.int16)).to(device).view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(arr)).to(device)


def kv_to_device(kv, device="cuda"):
    from top_hs2_fa_gb300.hs2 import KV

    lowp = kv.dtype in ("fp8", "fp4")  # uint8 codes with per-(page, KV head) scales
    fp4 = kv.dtype == "fp4"  # plus E4M3 scales of 16 channels
    return KV(k=to_torch(kv.k, kv.dtype, device),
              v=None if kv.v is None else to_torch(kv.v, kv.dtype, device),
              block_table=to_torch(kv.block_table, "i32", device),
              seq_len=to_torch(kv.seq_len, "i32", device),
              k_scale=to_torch(kv.k_scale, "f32", device) if lowp else None,
              v_scale=to_torch(kv.v_scale, "f32", device) if lowp and kv.v is not None else None,
              k_sf=to_torch(kv.k_sf, "u8", device) if fp4 else None,
              v_sf=to_torch(kv.v_sf, "u8", device) if fp4 and kv.v is not None else None)


def check_index_sets(gpu_idx, gpu_cnt, ora_idx, ora_cnt, ora_scores, label=""):
    """Equal counts; every position in the symmetric difference has an oracle score within
    SCORE_BAND relative of the oracle's k-th (last selected) score; GPU sets sorted ascending,
    -1 padded, without repeats. ``ora_scores[key]`` is the oracle score array over F.
    Returns the number of (query, head) sets that differ at all."""
    gpu_idx = np.asarray(gpu_idx)
    gpu_cnt = np.asarray(gpu_cnt)
    differ = 0
    for key in np.ndindex(*gpu_cnt.shape):
        n = int(ora_cnt[key])
        assert int(gpu_cnt[key]) == n, f"{label}{key}: count {gpu_cnt[key]} != {n}"
        g = gpu_idx[key][:n]
        assert np.all(gpu_idx[key][n:] == -1), f"{label}{key}: padding not -1"
        assert np.all(np.diff(g) > 0), f"{label}{key}: not strictly ascending"
        o = np.asarray(ora_idx[key][:n])
        if n == 0 or np.array_equal(g, o):
            continue
        differ += 1
        sc = ora_scores[key]
        assert g.min() >= 0 and g.max() < len(sc), f"{label}{key}: index outside the far range"
        kth = sc[o].min()
        sym = np.setxor1d(g, o)
        rel = np.abs(sc[sym] - kth) / max(abs(kth), 1e-300)
        assert np.all(rel <= SCORE_BAND), f"{label}{key}: set differs outside the 1e-3 band (max rel {rel.max():.3g})"
    return differ


def max_abs(a, b) -> float:
    return float(np.max(np.abs(np.asarray(a, np.float64) - np.asarray(b, np.float64)))) if np.size(a) else 0.0

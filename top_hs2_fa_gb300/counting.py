"""Algorithmic work model (bytes moved, flops, selector comparisons).

The benchmark divides these *algorithmic* amounts by measured kernel time to
get achieved GB/s or TFLOP/s; scratch traffic (e.g. the decode logits buffer)
is deliberately excluded, so overheads show up as a lower roofline fraction.

The selector-comparison and byte-crossover formulas restate the counting
examples of "2.3.1 · CSA、HCA 与 CSA2" (§5.1 "一个层组的成本明细", §6.1) and of
"Lecture 10 · 混合架构与稀疏注意力" (§5.3, Exercise 6); the tests pin them to
the numbers printed there.
"""
from __future__ import annotations

import numpy as np


def union_size(t: int, w: int, k: int) -> int:
    """|W(t) ∪ S(t)| = min(w, t) + min(k, max(0, t - w))."""
    return min(w, t) + min(k, max(0, t - w))


def decode_group_bytes(seq_len, Hq: int, Hkv: int, d: int, w: int, k: int, elem: float,
                       n_sa: int, max_pages: int | None = None, q_elem: float | None = None) -> dict:
    """HBM bytes one decode step of one group must move (FA + n_sa SA layers).

    FA reads every visible K and V row once; each SA layer reads the K and V rows
    of W ∪ S once per KV head (its query heads share the gathered row). Small
    terms: queries, fp32 outputs, indices and the block table. ``elem``: cache bytes
    per channel (2 bf16, 1 FP8, 0.5625 FP4 with its E4M3 scale per 16 channels);
    ``q_elem``: query bytes per channel (default ``elem``).
    """
    seq_len = [int(t) for t in seq_len]
    B = len(seq_len)
    row = d * elem
    fa = sum(t * Hkv * row * 2 for t in seq_len)
    sa_layer = sum(Hkv * union_size(t, w, k) * row * 2 for t in seq_len)
    q = B * Hq * d * (elem if q_elem is None else q_elem)
    o = B * Hq * d * 4
    idx = B * Hkv * k * 4
    mp = max_pages if max_pages is not None else max((t + 63) // 64 for t in seq_len)
    table = B * mp * 4
    io = (1 + n_sa) * (q + o + table) + idx * (1 + n_sa)
    return {"fa": fa, "sa_per_layer": sa_layer, "sa": n_sa * sa_layer, "io": io,
            "total": fa + n_sa * sa_layer + io}


def prefill_flops(n: int, Hq: int, d: int, w: int, k: int) -> dict:
    """Algorithmic flops of causal FA over n rows (QK^T and PV, 2 flops per MAC) and of
    one SA layer (the same over |W ∪ S| keys per row)."""
    t = np.arange(1, n + 1, dtype=np.float64)
    fa = 4.0 * d * Hq * float(t.sum())
    u = np.minimum(w, t) + np.minimum(k, np.maximum(0, t - w))
    sa = 4.0 * d * Hq * float(u.sum())
    return {"fa": fa, "sa_per_layer": sa}


def selector_comparisons(n_c: int, pool: int, n_full: int, n_reindex: int, n_reuse: int):
    """Entries scored by the selectors of one CSA2 layer group.

    Flat: every layer scores all n_c entries. Hierarchical: the Full layer scores all
    n_c, each Reindex layer only the pool, Reuse layers score nothing.
    Returns (flat, hierarchical)."""
    flat = (n_full + n_reindex + n_reuse) * n_c
    hier = n_full * n_c + n_reindex * pool
    return flat, hier


def dsa_decode_bytes(L: int, latent_bytes: int, index_key_bytes: int, k: int):
    """Bytes read per layer per decode step: dense reads every latent; DSA reads every
    index key plus k latents. Returns (dense, dsa)."""
    return latent_bytes * L, index_key_bytes * L + latent_bytes * min(k, L)


def dsa_crossover(latent_bytes: int, index_key_bytes: int, k: int) -> float:
    """Context length above which DSA reads fewer bytes than dense attention."""
    return latent_bytes * k / (latent_bytes - index_key_bytes)


def csa2_decode_bytes(seq_len, d: int, di: int, elem: int, k_top: int, pool_positions: int,
                      n_layers: int) -> dict:
    """HBM bytes of one CSA2 decode group: the Full indexer reads every indexer key, the
    Reindex indexer reads the pool's keys, every layer's MQA attention reads k_top K and
    V rows."""
    seq_len = [int(t) for t in seq_len]
    full = sum(t * di * elem for t in seq_len)
    reindex = sum(min(pool_positions, t) * di * elem for t in seq_len)
    attn = n_layers * sum(min(k_top, t) * d * elem * 2 for t in seq_len)
    return {"full": full, "reindex": reindex, "attention": attn, "total": full + reindex + attn}

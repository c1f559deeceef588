"""Oracle for group-shared top-k sparse attention — TEST INFRASTRUCTURE ONLY.

A plain, slow, float64 CPU restatement of what the pages define. Only
``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py``
may import or run it; the product path (the CUDA library and its binding) never
does. It shares no code with the CUDA path: inputs arrive as arrays in their
storage form (bfloat16 bit patterns as uint16, or float32) and are widened
exactly to float64 here.

Pages cited (by title, section):

* [HS2]  "HySparse2：整体架构、KV 生命周期与 PD 分离" — the HySparse2 explainer.
* [CSA2] "2.3.1 · CSA、HCA 与 CSA2: 压缩序列上的稀疏检索和跨层复用".
* [L10]  "Lecture 10 · 混合架构与稀疏注意力：Mamba、Marconi 与 DeepSeek-V3.2".

Readings taken where the pages are silent or their formulas were lost
(every one is listed with its basis in the design notes):

* positions are 0-based; a query that sees ``t`` keys sits at position t-1;
* window W(t) = the last min(w, t) positions [max(0,t-w), t-1]; far range
  F(t) = [0, t-w-1]; |S(t)| = min(k, max(0, t-w))            ([HS2] §7.2);
* softmax scale is the ``scale`` argument (1/sqrt(d) in every workload);
* GQA: query head h reads KV head g = h // (Hq/Hkv);
* selection score of far position s for KV head g is the FA attention
  probability summed over the query heads of g, normalised over all t visible
  keys: score_g(s) = sum_h exp(x_h(s) - lse_h)   ([HS2] §5, Appendix
  "Oracle 不能理解成对所有后层绝对正确": the FA's own exactly computed scores);
* ranking: higher score first, equal scores -> lower position first; the
  chosen set is returned sorted ascending and padded with -1;
* SA attends to W(t) ∪ S(t) under one softmax normalisation ([HS2] §7.2, §7.4);
* CSA2 indexer score I(s) = sum_j w_j * relu(q_j . k_s), unscaled ([L10] §5.1);
  Full: top-k_top over all s < t and top-max_blocks blocks of 8 positions by
  block maximum over visible members, equal maxima -> lower block id; Reindex:
  the same score restricted to the pool's positions ([CSA2] §3.2).

No function here is blocked, fused or reordered beyond these definitions.
"""
from __future__ import annotations

import copy
import math

import numpy as np

__all__ = [
    "to_f64", "gather_rows", "window", "far_count", "full_attention", "selection_scores",
    "topk_lower_index", "fa_decode", "sparse_attention", "sa_decode", "fa_prefill_rows",
    "sa_prefill_rows", "lightning_scores", "block_max", "indexer_full", "indexer_reindex",
    "pool_positions", "renormalisation_bound", "kv_append",
]


# ----------------------------------------------------------------------------- inputs
def fp8_e4m3_to_f64(b: np.ndarray) -> np.ndarray:
    """Exact value of FP8 E4M3 bytes (1 sign, 4 exponent bits with bias 7, 3 mantissa bits;
    exponent 0 is subnormal, m * 2^-9; exponent 15 with mantissa 7 is NaN, there is no
    infinity): the storage of the low-precision KV option (the pages' case for cutting main-KV
    bytes: [CSA2] §3, "KV 字节与 FP4")."""
    b = np.asarray(b, dtype=np.uint8).astype(np.int64)
    sign = np.where(b & 0x80, -1.0, 1.0)
    e, m = (b >> 3) & 0xF, b & 0x7
    mag = np.where(e == 0, m * 2.0 ** -9, (1.0 + m / 8.0) * np.exp2(e - 7.0))
    return np.where((e == 15) & (m == 7), np.nan, sign * mag)


def fp4_e2m1_to_f64(c: np.ndarray) -> np.ndarray:
    """Exact value of FP4 E2M1 codes (the low 4 bits of each entry: 1 sign, 2 exponent bits
    with bias 1, 1 mantissa bit; exponent 0 is subnormal, m * 0.5; no infinity or NaN, so the
    largest magnitude is 6): the main-KV format of the FP4 cache ([CSA2] §3, "KV 字节与 FP4":
    E2M1 values with one E4M3 scale per 16 channels)."""
    c = np.asarray(c, dtype=np.uint8).astype(np.int64) & 0xF
    sign = np.where(c & 0x8, -1.0, 1.0)
    e, m = (c >> 1) & 0x3, c & 0x1
    return sign * np.where(e == 0, m * 0.5, (1.0 + m / 2.0) * np.exp2(e - 1.0))


def fp4_unpack(packed: np.ndarray) -> np.ndarray:
    """Two E2M1 codes per byte along the last axis: channel 2i is the low nibble of byte i,
    channel 2i+1 the high nibble."""
    packed = np.asarray(packed, dtype=np.uint8)
    out = np.empty(packed.shape[:-1] + (2 * packed.shape[-1],), dtype=np.uint8)
    out[..., 0::2] = packed & 0xF
    out[..., 1::2] = packed >> 4
    return out


def to_f64(x: np.ndarray, dtype: str) -> np.ndarray:
    """Exact widening of stored values: bfloat16 bit patterns (uint16), float32, or FP8 E4M3
    bytes (uint8; scaling is applied by the caller)."""
    if dtype == "fp8":
        return fp8_e4m3_to_f64(x)
    if dtype == "bf16":
        u = np.ascontiguousarray(x, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
        return u.view(np.float32).astype(np.float64)
    if dtype == "f32":
        return np.asarray(x, dtype=np.float32).astype(np.float64)
    raise ValueError(dtype)


def gather_rows(pool: np.ndarray, bt_row: np.ndarray, g: int, positions: np.ndarray,
                page: int, dtype: str, scale=None) -> np.ndarray:
    """Block-table resolve: logical position s of one sequence -> row
    pool[bt[s // page]][g][s % page] of the paged pool, as float64 [len(positions)][d].
    Entries are read in place through the table ([HS2] §7.2: "按索引直接访问 paged KV").
    ``scale`` ([num_pages][Hkv], FP8 pools): row values are stored / scale[page][g].
    FP4 pools (``dtype`` "fp4"): ``scale`` is (slab, sf) with slab [num_pages][Hkv] float32
    and sf [num_pages][Hkv][page][d/16] E4M3 codes; channel c of a row is
    e2m1(code) * e4m3(sf[.., c // 16]) * slab[page][g]."""
    positions = np.asarray(positions, dtype=np.int64)
    pages = np.asarray(bt_row, dtype=np.int64)[positions // page]
    if positions.size and (pages < 0).any():
        raise ValueError("block table entry < 0 for a visible position")
    if dtype == "fp4":
        slab, sf = scale
        vals = fp4_e2m1_to_f64(fp4_unpack(pool[pages, g, positions % page, :]))
        gs = fp8_e4m3_to_f64(np.asarray(sf)[pages, g, positions % page, :])
        rows = vals * np.repeat(gs, 16, axis=-1)
        return rows * np.asarray(slab, dtype=np.float64)[pages, g][:, None]
    rows = to_f64(pool[pages, g, positions % page, :], dtype)
    if scale is not None:
        rows = rows * np.asarray(scale, dtype=np.float64)[pages, g][:, None]
    return rows


def _scale(kv, which: str):
    """The dequantisation scales of a low-precision pool: FP8, the per-(page, KV head)
    scale; FP4, that scale and the per-16-channel E4M3 scales; None otherwise."""
    if kv.dtype == "fp8":
        return getattr(kv, which + "_scale", None)
    if kv.dtype == "fp4":
        return getattr(kv, which + "_scale"), getattr(kv, which + "_sf")
    return None


def _qdtype(kv) -> str:
    """Queries are bf16 when the KV cache is FP8 or FP4, else the cache's dtype."""
    return "bf16" if kv.dtype in ("fp8", "fp4") else kv.dtype


# ----------------------------------------------------------------------------- decode KV append
def kv_append(kv, k_new: np.ndarray, v_new=None):
    """Decode KV append ([HS2] §10.1, step 3: once the source hidden state is ready, each
    Cross group's cache gains one entry for the new token). The new token is the last visible
    key of its sequence, position t-1 with t = seq_len[b] already counting it, so its rows
    k_new[b][g] (and v_new[b][g]) go to slot (t-1) % page of page bt[b][(t-1) // page].
    Returns a copy of the cache with those rows written in storage form; nothing else moves."""
    out = copy.copy(kv)
    out.k = np.array(kv.k, copy=True)
    out.v = None if kv.v is None else np.array(kv.v, copy=True)
    for b in range(len(kv.seq_len)):
        pos = int(kv.seq_len[b]) - 1
        if pos < 0:
            raise ValueError("a sequence with no visible key has no current token")
        pg = int(kv.block_table[b][pos // kv.page])
        if pg < 0:
            raise ValueError("block table entry < 0 for the current token")
        out.k[pg, :, pos % kv.page, :] = k_new[b]
        if out.v is not None:
            out.v[pg, :, pos % kv.page, :] = v_new[b]
    return out


# ----------------------------------------------------------------------------- window / far range
def window(t: int, w: int) -> np.ndarray:
    """Forced recent window: the last min(w, t) positions ([HS2] §7.2)."""
    return np.arange(max(0, t - w), t, dtype=np.int64)


def far_count(t: int, w: int) -> int:
    """|F(t)|: positions outside the window, [0, t-w-1] ([HS2] §7.2)."""
    return max(0, t - w)


# ----------------------------------------------------------------------------- FA layer
def full_attention(q: np.ndarray, K: np.ndarray, V: np.ndarray, scale: float):
    """Causal full attention of query heads ``q`` [H][d] over all visible keys K, V [t][d].

    Returns (x [H][t] logits, lse [H], o [H][d]) with x = scale * q.k,
    lse = log sum_s exp(x), o = sum_s exp(x - lse) v  ([HS2] §5: the FA layer scans
    the whole history with its own query).
    """
    x = (q @ K.T) * float(scale)
    m = x.max(axis=1, keepdims=True)
    lse = (m + np.log(np.exp(x - m).sum(axis=1, keepdims=True)))[:, 0]
    p = np.exp(x - lse[:, None])
    return x, lse, p @ V


def selection_scores(x: np.ndarray, lse: np.ndarray, n_far: int) -> np.ndarray:
    """score(s) = sum_h exp(x_h(s) - lse_h) for s in F = [0, n_far): the FA's own
    attention probabilities summed over the query heads of one KV head."""
    if n_far <= 0:
        return np.zeros(0)
    return np.exp(x[:, :n_far] - lse[:, None]).sum(axis=0)


def topk_lower_index(score: np.ndarray, k: int) -> np.ndarray:
    """The min(k, len(score)) best positions by (score descending, position ascending),
    returned sorted ascending."""
    n = len(score)
    kk = min(int(k), n)
    if kk <= 0:
        return np.zeros(0, dtype=np.int64)
    order = np.lexsort((np.arange(n), -np.asarray(score)))
    return np.sort(order[:kk])


def block_topk(score: np.ndarray, k: int, blk: int) -> np.ndarray:
    """Block-level selection of HySparse's first version ([HS2] §2 "第一版": 16 blocks of 64
    tokens = 1024 positions): far position s belongs to block s // blk; a block's key is the
    largest score among its far positions; the min(k // blk, #blocks) best blocks by (key
    descending, block ascending) are taken whole (their far positions), returned ascending.
    blk = 1 is token-level selection."""
    n = len(score)
    nb = (n + blk - 1) // blk
    kb = min(int(k) // blk, nb)
    if kb <= 0:
        return np.zeros(0, dtype=np.int64)
    keys = np.array([np.max(score[b * blk:min(n, b * blk + blk)]) for b in range(nb)])
    blocks = np.sort(np.lexsort((np.arange(nb), -keys))[:kb])
    return np.concatenate([np.arange(b * blk, min(n, b * blk + blk)) for b in blocks]).astype(np.int64)


def _pad(sel: np.ndarray, k: int) -> np.ndarray:
    out = np.full(k, -1, dtype=np.int32)
    out[:len(sel)] = sel
    return out


def fa_decode(q: np.ndarray, kv, w: int, k: int, scale: float, return_scores: bool = False, blk: int = 1):
    """FA layer for one decode query per sequence plus its window-excluding top-k
    (token-level; ``blk`` > 1: the block-level selection of ``block_topk``).

    ``q``: stored [B][Hq][d]; ``kv``: object with k, v, block_table, seq_len, dtype, page.
    Returns o float64 [B][Hq][d], lse [B][Hq], idx int32 [B][Hkv][k] (-1 padded,
    ascending), cnt int32 [B][Hkv]; with ``return_scores`` also a dict
    {(b, g): score array over F}.
    """
    qf = to_f64(q, _qdtype(kv))
    B, Hq, d = qf.shape
    Hkv = kv.k.shape[1]
    G = Hq // Hkv
    o = np.zeros((B, Hq, d))
    lse = np.zeros((B, Hq))
    idx = np.full((B, Hkv, k), -1, dtype=np.int32)
    cnt = np.zeros((B, Hkv), dtype=np.int32)
    scores = {}
    for b in range(B):
        t = int(kv.seq_len[b])
        pos = np.arange(t)
        for g in range(Hkv):
            K = gather_rows(kv.k, kv.block_table[b], g, pos, kv.page, kv.dtype, _scale(kv, "k"))
            V = gather_rows(kv.v, kv.block_table[b], g, pos, kv.page, kv.dtype, _scale(kv, "v"))
            hs = slice(g * G, (g + 1) * G)
            x, l, og = full_attention(qf[b, hs], K, V, scale)
            o[b, hs], lse[b, hs] = og, l
            sc = selection_scores(x, l, far_count(t, w))
            sel = topk_lower_index(sc, k) if blk == 1 else block_topk(sc, k, blk)
            idx[b, g], cnt[b, g] = _pad(sel, k), len(sel)
            if return_scores:
                scores[(b, g)] = sc
    if return_scores:
        return o, lse, idx, cnt, scores
    return o, lse, idx, cnt


# ----------------------------------------------------------------------------- SA layer
def sparse_attention(q: np.ndarray, K: np.ndarray, V: np.ndarray, scale: float, sink=None) -> np.ndarray:
    """One softmax over the gathered entries (window and far positions together,
    [HS2] §7.2 and §7.4: "一起参加同一次归一化").

    ``sink`` (one natural-log logit per query head, or None): the per-head learnable sink
    bias of the SA layers ([HS2] §17.1) read as one more key with that logit and a zero
    value, so it only enlarges the softmax denominator by exp(sink)."""
    x = (q @ K.T) * float(scale)
    if sink is None:
        x = x - x.max(axis=1, keepdims=True)
        p = np.exp(x)
        p /= p.sum(axis=1, keepdims=True)
        return p @ V
    b = np.asarray(sink, dtype=np.float64).reshape(-1)
    m = np.maximum(x.max(axis=1) if x.shape[1] else np.full(x.shape[0], -np.inf), b)
    p = np.exp(x - m[:, None])
    den = p.sum(axis=1) + np.exp(b - m)
    return (p @ V) / den[:, None]


def output_gate(o: np.ndarray, gate) -> np.ndarray:
    """The SA layers' output sigmoid gate ([HS2] §17.1), elementwise: o * sigmoid(gate);
    ``gate`` has o's shape (a per-head gate is the same value across d), None = no gate."""
    if gate is None:
        return o
    g = np.asarray(gate, dtype=np.float64)
    return o / (1.0 + np.exp(-g))


def _union(t: int, w: int, sel: np.ndarray) -> np.ndarray:
    win = window(t, w)
    sel = np.asarray(sel, dtype=np.int64)
    if sel.size and (sel.min() < 0 or sel.max() >= t):
        raise ValueError("selected position outside [0, t)")
    if np.intersect1d(win, sel).size or len(np.unique(sel)) != len(sel):
        raise ValueError("window and selection overlap or repeat")
    return np.concatenate([win, sel])


def sa_decode(q: np.ndarray, kv, w: int, idx: np.ndarray, cnt: np.ndarray, scale: float, sink=None,
              gate=None) -> np.ndarray:
    """SA layer reusing the FA's KV and indices with its own query ([HS2] §5):
    O_h = sum over U = W(t) ∪ S(t) of softmax_U(scale q_h.k) v. Optional sink bias [Hq] and
    output gate logits [B][Hq][d] ([HS2] §17.1, see sparse_attention / output_gate).
    Returns float64 [B][Hq][d]."""
    qf = to_f64(q, _qdtype(kv))
    B, Hq, d = qf.shape
    Hkv = kv.k.shape[1]
    G = Hq // Hkv
    o = np.zeros((B, Hq, d))
    for b in range(B):
        t = int(kv.seq_len[b])
        for g in range(Hkv):
            U = _union(t, w, idx[b, g, :cnt[b, g]])
            K = gather_rows(kv.k, kv.block_table[b], g, U, kv.page, kv.dtype, _scale(kv, "k"))
            V = gather_rows(kv.v, kv.block_table[b], g, U, kv.page, kv.dtype, _scale(kv, "v"))
            hs = slice(g * G, (g + 1) * G)
            o[b, hs] = sparse_attention(qf[b, hs], K, V, scale, None if sink is None else np.asarray(sink)[hs])
    return output_gate(o, None if gate is None else to_f64(gate, "f32"))


# ----------------------------------------------------------------------------- prefill (row by row)
def fa_prefill_rows(q: np.ndarray, kv, rows, w: int, k: int, scale: float, return_scores: bool = False):
    """FA prefill of a single sequence (kv.B == 1), evaluated at the listed query rows.

    Row i sees t_i = i + 1 keys (causal); each row is the decode computation at that
    length. Returns o [R][Hq][d], lse [R][Hq], idx int32 [R][Hkv][k], cnt [R][Hkv]
    (and per-(r, g) scores with ``return_scores``).
    """
    rows = np.asarray(rows, dtype=np.int64)
    qf = to_f64(q, _qdtype(kv))
    _, Hq, d = qf.shape
    Hkv = kv.k.shape[1]
    G = Hq // Hkv
    R = len(rows)
    o = np.zeros((R, Hq, d))
    lse = np.zeros((R, Hq))
    idx = np.full((R, Hkv, k), -1, dtype=np.int32)
    cnt = np.zeros((R, Hkv), dtype=np.int32)
    scores = {}
    Kall = [None] * Hkv
    Vall = [None] * Hkv
    tmax = int(rows.max()) + 1 if R else 0
    for g in range(Hkv):
        Kall[g] = gather_rows(kv.k, kv.block_table[0], g, np.arange(tmax), kv.page, kv.dtype, _scale(kv, "k"))
        Vall[g] = gather_rows(kv.v, kv.block_table[0], g, np.arange(tmax), kv.page, kv.dtype, _scale(kv, "v"))
    for r, i in enumerate(rows):
        t = int(i) + 1
        for g in range(Hkv):
            hs = slice(g * G, (g + 1) * G)
            x, l, og = full_attention(qf[i, hs], Kall[g][:t], Vall[g][:t], scale)
            o[r, hs], lse[r, hs] = og, l
            sc = selection_scores(x, l, far_count(t, w))
            sel = topk_lower_index(sc, k)
            idx[r, g], cnt[r, g] = _pad(sel, k), len(sel)
            if return_scores:
                scores[(r, g)] = sc
    if return_scores:
        return o, lse, idx, cnt, scores
    return o, lse, idx, cnt


def sa_prefill_rows(q: np.ndarray, kv, rows, w: int, idx: np.ndarray, cnt: np.ndarray,
                    scale: float, sink=None, gate=None) -> np.ndarray:
    """SA prefill at the listed rows; ``idx``/``cnt`` are indexed by the row itself
    ([n][Hkv][k] and [n][Hkv]); optional sink [Hq] and gate logits [n][Hq][d].
    Returns float64 [R][Hq][d]."""
    rows = np.asarray(rows, dtype=np.int64)
    qf = to_f64(q, _qdtype(kv))
    _, Hq, d = qf.shape
    Hkv = kv.k.shape[1]
    G = Hq // Hkv
    o = np.zeros((len(rows), Hq, d))
    for r, i in enumerate(rows):
        t = int(i) + 1
        for g in range(Hkv):
            U = _union(t, w, idx[i, g, :cnt[i, g]])
            K = gather_rows(kv.k, kv.block_table[0], g, U, kv.page, kv.dtype, _scale(kv, "k"))
            V = gather_rows(kv.v, kv.block_table[0], g, U, kv.page, kv.dtype, _scale(kv, "v"))
            hs = slice(g * G, (g + 1) * G)
            o[r, hs] = sparse_attention(qf[i, hs], K, V, scale, None if sink is None else np.asarray(sink)[hs])
    return output_gate(o, None if gate is None else to_f64(np.asarray(gate)[rows], "f32"))


# ----------------------------------------------------------------------------- CSA2 indexer
def lightning_scores(q_idx: np.ndarray, w_idx: np.ndarray, K: np.ndarray) -> np.ndarray:
    """I(s) = sum_j w_j * ReLU(q_j . k_s) over indexer heads j; the indexer key k_s is
    shared by all heads ([L10] §5.1). q_idx [Hi][di], w_idx [Hi], K [n][di] -> [n]."""
    return (np.asarray(w_idx, np.float64)[:, None] * np.maximum(q_idx @ K.T, 0.0)).sum(axis=0)


def block_max(I: np.ndarray, t: int, blk: int) -> np.ndarray:
    """Maximum of I over block b = [blk*b, blk*b + blk) ∩ [0, t), for b < ceil(t/blk)
    ([CSA2] §3.2: "给每个八位置块取最大值")."""
    nb = (t + blk - 1) // blk
    return np.array([I[b * blk:min(t, (b + 1) * blk)].max() for b in range(nb)])


def pool_positions(blocks: np.ndarray, t: int, blk: int) -> np.ndarray:
    """Ascending positions covered by the pool's blocks, clipped to [0, t)."""
    blocks = np.sort(np.asarray(blocks, dtype=np.int64))
    pos = (blocks[:, None] * blk + np.arange(blk)[None, :]).reshape(-1)
    return pos[pos < t]


def indexer_full(q_idx: np.ndarray, w_idx: np.ndarray, kidx, k_top: int, blk: int,
                 max_blocks: int, return_scores: bool = False):
    """CSA2 Full layer's hierarchical indexer ([CSA2] §3.2).

    Scores every visible position with the lightning indexer; the same scores give
    the layer's top-k_top positions and, through the per-block maximum, the
    top-max_blocks blocks that form the candidate pool for later Reindex layers.
    Returns idx int32 [B][k_top], cnt [B], pool int32 [B][max_blocks] (block ids,
    ascending, -1 padded), pool_cnt [B].
    """
    qf = to_f64(q_idx, kidx.dtype)
    B = qf.shape[0]
    idx = np.full((B, k_top), -1, dtype=np.int32)
    cnt = np.zeros(B, dtype=np.int32)
    pool = np.full((B, max_blocks), -1, dtype=np.int32)
    pool_cnt = np.zeros(B, dtype=np.int32)
    scores = {}
    for b in range(B):
        t = int(kidx.seq_len[b])
        K = gather_rows(kidx.k, kidx.block_table[b], 0, np.arange(t), kidx.page, kidx.dtype)
        I = lightning_scores(qf[b], w_idx[b], K)
        sel = topk_lower_index(I, k_top)
        idx[b, :len(sel)], cnt[b] = sel, len(sel)
        bm = block_max(I, t, blk)
        blocks = topk_lower_index(bm, max_blocks)
        pool[b, :len(blocks)], pool_cnt[b] = blocks, len(blocks)
        if return_scores:
            scores[b] = (I, bm)
    if return_scores:
        return idx, cnt, pool, pool_cnt, scores
    return idx, cnt, pool, pool_cnt


def indexer_reindex(q_idx: np.ndarray, w_idx: np.ndarray, kidx, k_top: int, blk: int,
                    pool: np.ndarray, pool_cnt: np.ndarray, return_scores: bool = False):
    """CSA2 Reindex layer: its own indexer query rescores only the pool's positions and
    keeps the top-k_top of them ([CSA2] §3.2: "后续 Reindex 只在这些位置重新打分").
    Returns idx int32 [B][k_top] (ascending positions, -1 padded), cnt [B]."""
    qf = to_f64(q_idx, kidx.dtype)
    B = qf.shape[0]
    idx = np.full((B, k_top), -1, dtype=np.int32)
    cnt = np.zeros(B, dtype=np.int32)
    scores = {}
    for b in range(B):
        t = int(kidx.seq_len[b])
        pos = pool_positions(pool[b, :pool_cnt[b]], t, blk)
        K = gather_rows(kidx.k, kidx.block_table[b], 0, pos, kidx.page, kidx.dtype)
        I = lightning_scores(qf[b], w_idx[b], K)
        sel = pos[topk_lower_index(I, k_top)]
        idx[b, :len(sel)], cnt[b] = np.sort(sel), len(sel)
        if return_scores:
            scores[b] = (pos, I)
    if return_scores:
        return idx, cnt, scores
    return idx, cnt


# ----------------------------------------------------------------------------- error bound
def renormalisation_bound(p: np.ndarray, keep: np.ndarray, V: np.ndarray) -> float:
    """Bound on |o_keep - o| for one head: with missed mass eps = 1 - sum_{keep} p and
    |v| <= Bv, the renormalised output over ``keep`` differs from the dense output by at
    most 2 * eps * Bv ([HS2] §18 and the appendix "可以怎样用数学解释", whose
    formulas were lost in extraction; this is the plainest reading of the prose)."""
    eps = 1.0 - float(p[keep].sum())
    Bv = float(np.sqrt((V * V).sum(axis=1)).max())
    return 2.0 * max(eps, 0.0) * Bv

"""Seeded synthetic inputs for group-shared top-k sparse attention.

This module only *builds inputs*: random tensors, the paged KV layout with a
permuted block table, and planted "needle" keys. It holds none of the
attention, selection or indexer arithmetic, so both the CUDA path (through the
tests and the benchmark) and the CPU oracle can consume its output without
sharing any of the method's code.

Storage conventions (identical for every consumer):

* ``dtype == "bf16"``: tensors are ``uint16`` arrays holding bfloat16 bit
  patterns, produced by round-to-nearest-even from float32 draws.
* ``dtype == "f32"``: tensors are ``float32`` arrays.
* K/V pools: ``[num_pages][Hkv][page][d]``; block table ``int32[B][max_pages]``
  (unused entries are -1); ``seq_len`` is ``int32[B]`` = number of visible keys,
  the current query's own key included.
* Slots of a page beyond ``seq_len`` are filled with a large constant so that a
  kernel that reads past the visible range produces visibly wrong results.

Workload shapes follow the pages' settings: a Cross group of one FA and five SA
layers sharing one KV cache, window w=128 and top-k=1024 (HySparse2：整体架构、
KV 生命周期与 PD 分离, §7.2-7.3); the CSA2 indexer with 64 heads, 8-position
blocks, up to 2048 blocks and top-512 (2.3.1 · CSA、HCA 与 CSA2, §3.2).
"""
from __future__ import annotations

import math
import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field

import numpy as np

PAGE = 64
POISON = 300.0  # value written into never-visible page slots
_CHUNK = 1 << 22  # values per generator chunk (fixed: results do not depend on thread count)


# ----------------------------------------------------------------------------- rounding helpers
def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bfloat16 (nearest-even) and return the uint16 bit patterns."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    r = (u + (np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1)))) >> np.uint32(16)
    return r.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def _fp8_e4m3_table() -> np.ndarray:
    """Values of the 127 non-negative finite FP8 E4M3 codes 0x00..0x7E, ascending (the
    format's magnitude order is its code order): exponent e (bias 7, 0 = subnormal), 3-bit m."""
    c = np.arange(127)
    e, m = c >> 3, c & 7
    return np.where(e == 0, m * 2.0 ** -9, (1.0 + m / 8.0) * np.exp2(e - 7.0))


_E4M3 = _fp8_e4m3_table()


def f32_to_fp8_e4m3(x: np.ndarray) -> np.ndarray:
    """Round to the nearest FP8 E4M3 value (ties to the even code), saturating at +-448;
    returns the uint8 codes."""
    x = np.asarray(x, dtype=np.float64)
    a = np.minimum(np.abs(x), 448.0)
    hi = np.clip(np.searchsorted(_E4M3, a), 1, 126)
    lo = hi - 1
    dl, dh = a - _E4M3[lo], _E4M3[hi] - a
    code = np.where(dl < dh, lo, np.where(dh < dl, hi, np.where(lo % 2 == 0, lo, hi)))
    code = np.where(a <= 0.0, 0, code)
    return (code | np.where(np.signbit(x), 0x80, 0)).astype(np.uint8)


def store(x: np.ndarray, dtype: str) -> np.ndarray:
    """Convert float32 values to the storage form of ``dtype``."""
    if dtype == "bf16":
        return f32_to_bf16_bits(x)
    if dtype == "f32":
        return np.ascontiguousarray(x, dtype=np.float32)
    raise ValueError(dtype)


def values(x: np.ndarray, dtype: str) -> np.ndarray:
    """Float32 view of stored values (exact for both storage forms)."""
    return bf16_bits_to_f32(x) if dtype == "bf16" else np.asarray(x, dtype=np.float32)


# ----------------------------------------------------------------------------- random fill
def _ss(seed) -> np.random.SeedSequence:
    return seed if isinstance(seed, np.random.SeedSequence) else np.random.SeedSequence(seed)


def _threads() -> int:
    return max(1, min(16, os.cpu_count() or 1))


def normal_fill(out: np.ndarray, seed, scale: float = 1.0, dtype: str = "f32") -> None:
    """Fill ``out`` (flat-contiguous) with N(0, scale^2) draws in storage form ``dtype``.

    The array is cut into fixed chunks, each drawn from its own PCG64 stream
    spawned from ``seed``; the result is independent of the number of threads.
    """
    flat = out.reshape(-1)
    n = flat.size
    nchunks = max(1, (n + _CHUNK - 1) // _CHUNK)
    seeds = _ss(seed).spawn(nchunks)

    def work(i: int) -> None:
        lo, hi = i * _CHUNK, min(n, (i + 1) * _CHUNK)
        rng = np.random.Generator(np.random.PCG64(seeds[i]))
        buf = rng.standard_normal(hi - lo, dtype=np.float32)
        if scale != 1.0:
            buf *= np.float32(scale)
        flat[lo:hi] = store(buf, dtype)

    if nchunks == 1:
        work(0)
    else:
        with ThreadPoolExecutor(_threads()) as ex:
            list(ex.map(work, range(nchunks)))


def normal(shape, seed, scale: float = 1.0, dtype: str = "f32") -> np.ndarray:
    out = np.empty(shape, dtype=np.uint16 if dtype == "bf16" else np.float32)
    normal_fill(out, seed, scale, dtype)
    return out


# ----------------------------------------------------------------------------- paged layout
@dataclass
class PagedKV:
    """One group's paged KV cache (shared by its FA and its SA layers)."""

    k: np.ndarray  # [num_pages][Hkv][page][d] (storage form)
    v: np.ndarray | None  # same shape, or None for an indexer-key cache
    block_table: np.ndarray  # int32 [B][max_pages]
    seq_len: np.ndarray  # int32 [B]
    dtype: str
    page: int = PAGE
    k_scale: np.ndarray | None = None  # FP8 / FP4 pools: float32 [num_pages][Hkv] per-slab scale
    v_scale: np.ndarray | None = None
    k_sf: np.ndarray | None = None  # FP4 pools: uint8 E4M3 codes [num_pages][Hkv][page][d/16]
    v_sf: np.ndarray | None = None

    @property
    def num_pages(self) -> int:
        return int(self.k.shape[0])

    @property
    def Hkv(self) -> int:
        return int(self.k.shape[1])

    @property
    def d(self) -> int:
        return int(self.k.shape[3]) * (2 if self.dtype == "fp4" else 1)  # FP4: two codes per byte

    @property
    def B(self) -> int:
        return int(self.seq_len.shape[0])

    @property
    def max_pages(self) -> int:
        return int(self.block_table.shape[1])

    def locate(self, b: int, s) -> tuple:
        """(physical page, slot) of logical position(s) ``s`` of sequence ``b``."""
        s = np.asarray(s)
        return self.block_table[b][s // self.page], s % self.page


def make_block_table(seq_len: np.ndarray, page: int, seed, permute: bool = True):
    """Assign every (sequence, logical page) a distinct physical page.

    Returns (block_table int32[B][max_pages] with -1 for unused entries, num_pages).
    With ``permute`` the physical pages are a random permutation of all pages.
    """
    npg = [(int(t) + page - 1) // page for t in seq_len]
    total = int(sum(npg))
    max_pages = max(1, max(npg) if npg else 1)
    phys = np.arange(total, dtype=np.int64)
    if permute:
        phys = np.random.Generator(np.random.PCG64(seed)).permutation(total)
    bt = np.full((len(npg), max_pages), -1, dtype=np.int32)
    off = 0
    for b, n in enumerate(npg):
        bt[b, :n] = phys[off:off + n]
        off += n
    return bt, total


def poison_tail(kv: PagedKV) -> None:
    """Write POISON into every slot beyond seq_len (and into pages no sequence owns)."""
    pv = store(np.array([POISON], np.float32), kv.dtype)[0]
    owned = np.zeros(kv.num_pages, dtype=bool)
    for b in range(kv.B):
        t = int(kv.seq_len[b])
        npg = (t + kv.page - 1) // kv.page
        owned[kv.block_table[b, :npg]] = True
        if t % kv.page:
            last = kv.block_table[b, npg - 1]
            kv.k[last, :, t % kv.page:, :] = pv
            if kv.v is not None:
                kv.v[last, :, t % kv.page:, :] = pv
    kv.k[~owned] = pv
    if kv.v is not None:
        kv.v[~owned] = pv


def random_paged_kv(seq_len, Hkv: int, d: int, dtype: str, seed, with_v: bool = True,
                    page: int = PAGE, permute: bool = True, scale: float = 1.0) -> PagedKV:
    """K (and V) i.i.d. N(0, scale^2) in a paged pool with a (permuted) block table."""
    seq_len = np.asarray(seq_len, dtype=np.int32)
    ss = _ss(seed)
    s_bt, s_k, s_v = ss.spawn(3)
    bt, total = make_block_table(seq_len, page, s_bt, permute)
    shape = (max(total, 1), Hkv, page, d)
    k = normal(shape, s_k, scale, dtype)
    v = normal(shape, s_v, scale, dtype) if with_v else None
    kv = PagedKV(k=k, v=v, block_table=bt, seq_len=seq_len, dtype=dtype, page=page)
    poison_tail(kv)
    return kv


def write_rows(kv: PagedKV, b: int, g: int, pos: np.ndarray, rows_f32: np.ndarray, which: str = "k") -> None:
    pg, sl = kv.locate(b, pos)
    arr = kv.k if which == "k" else kv.v
    arr[pg, g, sl, :] = store(rows_f32.astype(np.float32), kv.dtype)


def plant_needles(kv: PagedKV, q_vals: np.ndarray, n_needles: int, w: int, seed,
                  lam: float = 8.0) -> list:
    """Plant keys aligned with the mean query head of each KV head.

    For each sequence b, ``n_needles`` positions are drawn without replacement
    from the far range [0, t-w-1]; at each, for each KV head g, the key is set
    to lam*sqrt(d)*qbar/|qbar|^2 with qbar the mean of the query heads of g, so
    that the mean-head logit (scaled by 1/sqrt(d)) equals lam.
    ``q_vals``: float32 [B][Hq][d]. Returns the planted positions per sequence.
    """
    rng = np.random.Generator(np.random.PCG64(seed))
    B, Hq, d = q_vals.shape
    Hkv = kv.Hkv
    G = Hq // Hkv
    out = []
    for b in range(B):
        t = int(kv.seq_len[b])
        nfar = max(0, t - w)
        m = min(n_needles, nfar)
        pos = np.sort(rng.choice(nfar, size=m, replace=False)) if m > 0 else np.zeros(0, np.int64)
        for g in range(Hkv):
            qbar = q_vals[b, g * G:(g + 1) * G].astype(np.float64).mean(0)
            key = lam * math.sqrt(d) * qbar / max(float(qbar @ qbar), 1e-30)
            write_rows(kv, b, g, pos, np.repeat(key[None, :], m, 0))
        out.append(pos)
    return out


# ----------------------------------------------------------------------------- group workloads
@dataclass
class DecodeGroup:
    """One decode step of one Cross group: FA query + n_sa SA queries over one paged KV."""

    kv: PagedKV
    q_fa: np.ndarray  # [B][Hq][d] storage form
    q_sa: list  # n_sa x [B][Hq][d] storage form
    Hq: int
    w: int
    k: int
    scale: float
    needles: list = field(default_factory=list)


def decode_group(seq_len, Hq: int, Hkv: int, d: int, w: int, k: int, dtype: str, seed,
                 n_sa: int = 5, needles: int = 32, qproj: bool = False, page: int = PAGE,
                 permute: bool = True, qscale: float = 1.0, kvscale: float = 1.0) -> DecodeGroup:
    """Decode workload. With ``qproj`` the queries are x @ W_Q (x ~ N(0,1)^(Hq*d),
    W_Q ~ N(0, 1/(Hq*d))), one W_Q per layer; otherwise they are N(0, qscale^2)."""
    seq_len = np.asarray(seq_len, dtype=np.int32)
    B = len(seq_len)
    ss = _ss(seed)
    s_kv, s_q, s_needle = ss.spawn(3)
    kv = random_paged_kv(seq_len, Hkv, d, dtype, s_kv, page=page, permute=permute, scale=kvscale)
    qs = []
    qseeds = s_q.spawn(1 + n_sa + 1)
    if qproj:
        hid = Hq * d
        x = normal((B, hid), qseeds[-1])
        for j in range(1 + n_sa):
            W = normal((hid, hid), qseeds[j], scale=1.0 / math.sqrt(hid))
            qs.append(store((x @ W).reshape(B, Hq, d), dtype))
    else:
        for j in range(1 + n_sa):
            qs.append(normal((B, Hq, d), qseeds[j], qscale, dtype))
    q_fa_vals = values(qs[0], dtype).reshape(B, Hq, d)
    pos = plant_needles(kv, q_fa_vals, needles, w, s_needle) if needles else []
    return DecodeGroup(kv=kv, q_fa=qs[0], q_sa=qs[1:], Hq=Hq, w=w, k=k, scale=1.0 / math.sqrt(d),
                       needles=pos)


def quantize_kv_fp8(kv: PagedKV) -> PagedKV:
    """FP8 E4M3 copy of a paged pool with one scale per (page, KV head) slab for K and for V:
    scale = max |value| / 448 (1 for an all-zero slab), code = E4M3(value / scale)."""
    out = {}
    for name in ("k", "v"):
        src = getattr(kv, name)
        codes = np.empty(src.shape, dtype=np.uint8)
        sc = np.empty(src.shape[:2], dtype=np.float32)
        for p0 in range(0, src.shape[0], 2048):  # page chunks bound the temporaries
            x = values(src[p0:p0 + 2048], kv.dtype).astype(np.float64)
            amax = np.abs(x).max(axis=(2, 3))
            s_ = np.where(amax > 0, amax / 448.0, 1.0).astype(np.float32)
            codes[p0:p0 + 2048] = f32_to_fp8_e4m3(x / s_[:, :, None, None].astype(np.float64))
            sc[p0:p0 + 2048] = s_
        out[name], out[name + "_scale"] = codes, sc
    return PagedKV(k=out["k"], v=out["v"], block_table=kv.block_table, seq_len=kv.seq_len, dtype="fp8", page=kv.page,
                   k_scale=out["k_scale"], v_scale=out["v_scale"])


_E2M1 = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])  # magnitudes of E2M1 codes 0..7


def f32_to_fp4_e2m1(x: np.ndarray) -> np.ndarray:
    """Round to the nearest FP4 E2M1 value (ties to the even code), saturating at +-6;
    returns the 4-bit codes (uint8 0..15, bit 3 = sign)."""
    x = np.asarray(x, dtype=np.float64)
    a = np.minimum(np.abs(x), 6.0)
    hi = np.clip(np.searchsorted(_E2M1, a), 1, 7)
    lo = hi - 1
    dl, dh = a - _E2M1[lo], _E2M1[hi] - a
    code = np.where(dl < dh, lo, np.where(dh < dl, hi, np.where(lo % 2 == 0, lo, hi)))
    code = np.where(a <= 0.0, 0, code)
    return (code | np.where(np.signbit(x) & (code > 0), 8, 0)).astype(np.uint8)


def quantize_kv_fp4(kv: PagedKV) -> PagedKV:
    """FP4 copy of a paged pool: E2M1 codes (two per byte, channel 2i in the low nibble) with
    one E4M3 scale per 16 channels of a row and one float32 scale per (page, KV head) slab.
    slab = max |value| / (6 * 448) (1 for an all-zero slab); a group's E4M3 scale is the
    smallest E4M3 value >= its max |value / slab| / 6 (so no code saturates); code =
    E2M1(value / slab / group scale)."""
    out = {}
    for name in ("k", "v"):
        src = getattr(kv, name)
        P, Hh, S, d = src.shape
        codes = np.empty((P, Hh, S, d // 2), dtype=np.uint8)
        sf = np.empty((P, Hh, S, d // 16), dtype=np.uint8)
        slab = np.empty((P, Hh), dtype=np.float32)
        for p0 in range(0, P, 1024):  # page chunks bound the temporaries
            x = values(src[p0:p0 + 1024], kv.dtype).astype(np.float64)
            amax = np.abs(x).max(axis=(2, 3))
            sl = np.where(amax > 0, amax / (6.0 * 448.0), 1.0).astype(np.float32)
            y = x / sl[:, :, None, None].astype(np.float64)
            yg = y.reshape(y.shape[:3] + (d // 16, 16))
            need = np.abs(yg).max(axis=-1) / 6.0
            gc = np.clip(np.searchsorted(_E4M3, need, side="left"), 0, 126)  # smallest value >= need
            gs = _E4M3[gc]
            q = f32_to_fp4_e2m1(np.where(gs[..., None] > 0, yg / np.where(gs > 0, gs, 1.0)[..., None], 0.0))
            q = q.reshape(y.shape)
            codes[p0:p0 + 1024] = q[..., 0::2] | (q[..., 1::2] << 4)
            sf[p0:p0 + 1024] = gc.astype(np.uint8)
            slab[p0:p0 + 1024] = sl
        out[name], out[name + "_sf"], out[name + "_scale"] = codes, sf, slab
    return PagedKV(k=out["k"], v=out["v"], block_table=kv.block_table, seq_len=kv.seq_len, dtype="fp4", page=kv.page,
                   k_scale=out["k_scale"], v_scale=out["v_scale"], k_sf=out["k_sf"], v_sf=out["v_sf"])


def decode_group_fp4(seq_len, Hq: int, Hkv: int, d: int, w: int, k: int, seed, **kw) -> DecodeGroup:
    """The bf16 decode workload with its paged KV stored as FP4 E2M1 + E4M3 group scales."""
    grp = decode_group(seq_len, Hq, Hkv, d, w, k, "bf16", seed, **kw)
    grp.kv = quantize_kv_fp4(grp.kv)
    return grp


def decode_group_fp8(seq_len, Hq: int, Hkv: int, d: int, w: int, k: int, seed, **kw) -> DecodeGroup:
    """The bf16 decode workload with its paged KV stored as FP8 E4M3 (queries stay bf16)."""
    grp = decode_group(seq_len, Hq, Hkv, d, w, k, "bf16", seed, **kw)
    grp.kv = quantize_kv_fp8(grp.kv)
    return grp


@dataclass
class PrefillGroup:
    """Prefill of one sequence of n tokens: FA + n_sa SA layers over one paged KV (B=1)."""

    kv: PagedKV
    q_fa: np.ndarray  # [n][Hq][d]
    q_sa: list  # n_sa x [n][Hq][d]
    Hq: int
    w: int
    k: int
    scale: float


def drifting_keys(n: int, Hkv: int, d: int, rho: float, seed) -> np.ndarray:
    """K_i = mu_i + eps_i with mu an AR(1) process per KV head (float32 [n][Hkv][d]).

    mu_0 ~ N(0, I); mu_i = rho*mu_{i-1} + sqrt(1-rho^2)*eta_i; eps, eta ~ N(0, I).
    """
    s_eta, s_eps = _ss(seed).spawn(2)
    eta = normal((n, Hkv, d), s_eta)
    eps = normal((n, Hkv, d), s_eps)
    c = np.float32(math.sqrt(1.0 - rho * rho))
    mu = np.empty((n, Hkv, d), np.float32)
    mu[0] = eta[0]
    r = np.float32(rho)
    for i in range(1, n):
        mu[i] = r * mu[i - 1] + c * eta[i]
    return mu + eps


def prefill_group(n: int, Hq: int, Hkv: int, d: int, w: int, k: int, dtype: str, seed,
                  n_sa: int = 5, rho: float | None = None, scale_in: float = 1.0,
                  needles: int = 0, page: int = PAGE, permute: bool = False) -> PrefillGroup:
    """Prefill workload on a single sequence (B=1). ``rho`` selects AR(1)-drifting keys."""
    ss = _ss(seed)
    s_kv, s_k, s_q, s_needle = ss.spawn(4)
    kv = random_paged_kv([n], Hkv, d, dtype, s_kv, page=page, permute=permute, scale=scale_in)
    if rho is not None:
        K = drifting_keys(n, Hkv, d, rho, s_k) * np.float32(scale_in)
        pos = np.arange(n)
        for g in range(Hkv):
            write_rows(kv, 0, g, pos, K[:, g, :])
    qseeds = s_q.spawn(1 + n_sa)
    qs = [normal((n, Hq, d), qseeds[j], scale_in, dtype) for j in range(1 + n_sa)]
    if needles:
        # align needles with the last row's FA query so that its selection is non-trivial
        qlast = values(qs[0], dtype).reshape(n, Hq, d)[n - 1:n]
        kv1 = PagedKV(k=kv.k, v=kv.v, block_table=kv.block_table, seq_len=kv.seq_len, dtype=dtype, page=page)
        plant_needles(kv1, qlast, needles, w, s_needle)
    return PrefillGroup(kv=kv, q_fa=qs[0], q_sa=qs[1:], Hq=Hq, w=w, k=k, scale=1.0 / math.sqrt(d))


@dataclass
class TinyGroup:
    """Tiny fp32 group: prefill over n rows plus one decode query at position n."""

    prefill: PrefillGroup  # its kv holds n+1 keys; prefill rows use the first n
    decode: DecodeGroup  # B=1, seq_len = n+1, same kv arrays


def tiny_group(n: int = 2048, Hq: int = 4, Hkv: int = 1, d: int = 64, w: int = 16, k: int = 64,
               dtype: str = "f32", needles: int = 8, seed=0, page: int = PAGE) -> TinyGroup:
    """Q, K, V ~ N(0,1)/sqrt(d); needles aligned to the decode query; one SA layer."""
    sc = 1.0 / math.sqrt(d)
    ss = _ss(seed)
    s_kv, s_q, s_needle = ss.spawn(3)
    kv = random_paged_kv([n + 1], Hkv, d, dtype, s_kv, page=page, permute=True, scale=sc)
    qseeds = s_q.spawn(4)
    q_fa = normal((n + 1, Hq, d), qseeds[0], sc, dtype)
    q_sa = normal((n + 1, Hq, d), qseeds[1], sc, dtype)
    qdec = values(q_fa, dtype).reshape(n + 1, Hq, d)[n:n + 1]
    pos = plant_needles(kv, qdec, needles, w, s_needle)
    pre = PrefillGroup(kv=PagedKV(k=kv.k, v=kv.v, block_table=kv.block_table,
                                  seq_len=np.array([n], np.int32), dtype=dtype, page=page),
                       q_fa=q_fa[:n], q_sa=[q_sa[:n]], Hq=Hq, w=w, k=k, scale=sc)
    dec = DecodeGroup(kv=kv, q_fa=q_fa[n:n + 1], q_sa=[q_sa[n:n + 1]], Hq=Hq, w=w, k=k, scale=sc,
                      needles=pos)
    return TinyGroup(prefill=pre, decode=dec)


@dataclass
class Csa2Group:
    """CSA2 decode group: main paged KV (Hkv=1), indexer-key pool, two indexer queries
    (Full and Reindex layers) and one main query per layer (Full, Reindex, Reuse x n_reuse)."""

    kv: PagedKV  # main KV, Hkv = 1
    kidx: PagedKV  # indexer keys, Hkv = 1, v = None
    q_idx: list  # [Full, Reindex] each [B][Hi][di] storage form
    w_idx: list  # [Full, Reindex] each float32 [B][Hi]
    q_main: list  # (2 + n_reuse) x [B][Hq][d]
    Hq: int
    k_top: int
    blk: int
    max_blocks: int
    scale: float
    needles: list = field(default_factory=list)


def csa2_group(seq_len, Hq: int = 32, d: int = 128, Hi: int = 64, di: int = 128, k_top: int = 512,
               blk: int = 8, max_blocks: int = 2048, n_reuse: int = 3, needles: int = 32,
               dtype: str = "bf16", seed=0, page: int = PAGE) -> Csa2Group:
    seq_len = np.asarray(seq_len, dtype=np.int32)
    B = len(seq_len)
    ss = _ss(seed)
    s_kv, s_ki, s_q, s_w, s_m, s_needle = ss.spawn(6)
    kv = random_paged_kv(seq_len, 1, d, dtype, s_kv, page=page)
    kidx = random_paged_kv(seq_len, 1, di, dtype, s_ki, with_v=False, page=page)
    qseeds = s_q.spawn(2)
    q_idx = [normal((B, Hi, di), qseeds[j], 1.0, dtype) for j in range(2)]
    wseeds = s_w.spawn(2)
    w_idx = [np.random.Generator(np.random.PCG64(wseeds[j])).uniform(0.0, 1.0, (B, Hi)).astype(np.float32)
             for j in range(2)]
    mseeds = s_m.spawn(2 + n_reuse)
    q_main = [normal((B, Hq, d), mseeds[j], 1.0, dtype) for j in range(2 + n_reuse)]
    # needles in the indexer keys, aligned with the Full layer's weighted query direction
    rng = np.random.Generator(np.random.PCG64(s_needle))
    qv = values(q_idx[0], dtype).reshape(B, Hi, di).astype(np.float64)
    pos_all = []
    for b in range(B):
        t = int(seq_len[b])
        m = min(needles, t)
        pos = np.sort(rng.choice(t, size=m, replace=False)) if m else np.zeros(0, np.int64)
        u = (w_idx[0][b].astype(np.float64)[:, None] * qv[b]).sum(0)
        u = u / max(np.linalg.norm(u), 1e-30)
        key = 4.0 * math.sqrt(di) * u
        write_rows(kidx, b, 0, pos, np.repeat(key[None, :], m, 0))
        pos_all.append(pos)
    return Csa2Group(kv=kv, kidx=kidx, q_idx=q_idx, w_idx=w_idx, q_main=q_main, Hq=Hq, k_top=k_top,
                     blk=blk, max_blocks=max_blocks, scale=1.0 / math.sqrt(d), needles=pos_all)


# ----------------------------------------------------------------------------- named workloads
def uniform_lengths(B: int, lo: int, hi: int, seed) -> np.ndarray:
    return np.random.Generator(np.random.PCG64(seed)).integers(lo, hi + 1, size=B).astype(np.int32)


WORKLOADS = {
    "tiny_fp32": dict(n=2048, Hq=4, Hkv=1, d=64, w=16, k=64, dtype="f32", needles=8),
    "decode_bf16_b64_t16k-32k": dict(B=64, t_lo=16384, t_hi=32768, Hq=32, Hkv=4, d=128, w=128,
                                     k=1024, dtype="bf16", needles=32, n_sa=5),
    "prefill_bf16_n32768": dict(n=32768, Hq=32, Hkv=4, d=128, w=128, k=1024, dtype="bf16",
                                rho=0.999, n_sa=5),
    "long_decode_bf16_b16_t131072_x4": dict(B=16, t=131072, groups=4, Hq=32, Hkv=4, d=128, w=128,
                                            k=1024, dtype="bf16", needles=64, n_sa=5),
    "csa2_decode_bf16_b8_t131072": dict(B=8, t=131072, Hq=32, d=128, Hi=64, di=128, k_top=512,
                                        blk=8, max_blocks=2048, n_reuse=3, needles=32, dtype="bf16"),
}


def decode_bf16_workload(seed: int = 0, B: int = 64, t_lo: int = 16384, t_hi: int = 32768,
                         qproj: bool = True) -> DecodeGroup:
    """Decode, bf16 KV: lengths uniform in [t_lo, t_hi], Hq=32, Hkv=4, d=128, w=128, k=1024,
    page 64 with a permuted table, 32 needles per sequence, five SA layers."""
    c = WORKLOADS["decode_bf16_b64_t16k-32k"]
    ss = _ss(seed)
    s_len, s_grp = ss.spawn(2)
    lens = uniform_lengths(B, t_lo, t_hi, s_len)
    return decode_group(lens, c["Hq"], c["Hkv"], c["d"], c["w"], c["k"], c["dtype"], s_grp,
                        n_sa=c["n_sa"], needles=c["needles"], qproj=qproj)

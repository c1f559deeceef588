"""Thin Python binding of libhs2 (argument marshalling only).

Functions carry the C names (``hs2_fa_select``, ``hs2_sa_reuse``,
``hs2_hier_reindex``, the ``*_workspace`` queries) and take torch CUDA tensors;
every step of the path runs in the library's kernels. PyTorch only provides
device memory and the current stream. There is no fallback: if the library
cannot be loaded, every call raises.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

import torch

from . import build as _build

ABI_VERSION = 6  # include/hs2.h HS2_ABI_VERSION this binding marshals for
F32, BF16, FP8_E4M3, FP4_E2M1 = 0, 1, 2, 3
FULL, REINDEX = 0, 1
DEV_BAD_PAGE, DEV_BAD_INDEX, DEV_TIMEOUT, DEV_BAD_LENGTH, DEV_SELECT = 1, 2, 4, 8, 16
EXPORTS = (
    "hs2_fa_select_workspace", "hs2_fa_select", "hs2_fa_select_ex", "hs2_sa_reuse_workspace", "hs2_sa_reuse", "hs2_sa_reuse_ex",
    "hs2_hier_reindex_workspace", "hs2_hier_reindex", "hs2_strerror", "hs2_last_cuda_error",
    "hs2_abi_version", "hs2_profile_next", "hs2_selftest_wait_timeout", "hs2_fa_select_noalloc", "hs2_fa_select_noalloc_capacity",
    "hs2_kv_append", "hs2_fa_select_append", "hs2_fa_select_launches", "hs2_sa_reuse_launches",
)
STAGE_FA_SCAN, STAGE_SA_GATHER, STAGE_INDEXER = 0, 1, 2
SA_OVERLAP = 1  # HS2_SA_OVERLAP


class hs2_kv(ctypes.Structure):
    _fields_ = [
        ("k", ctypes.c_void_p), ("v", ctypes.c_void_p), ("block_table", ctypes.c_void_p),
        ("seq_len", ctypes.c_void_p), ("batch", ctypes.c_int32), ("num_pages", ctypes.c_int32),
        ("max_pages", ctypes.c_int32), ("page_size", ctypes.c_int32), ("Hkv", ctypes.c_int32),
        ("d", ctypes.c_int32), ("dtype", ctypes.c_int32), ("k_scale", ctypes.c_void_p), ("v_scale", ctypes.c_void_p),
        ("k_sf", ctypes.c_void_p), ("v_sf", ctypes.c_void_p),
    ]


class HS2Error(RuntimeError):
    pass


_lib = None


def load(path: str | None = None) -> ctypes.CDLL:
    """Load libhs2.so (built in-tree by ``build.build()``); raises if it is missing."""
    global _lib
    if _lib is not None:
        return _lib
    path = path or _build.LIB
    if not os.path.exists(path):
        raise HS2Error(f"libhs2 not built ({path}); run top_hs2_fa_gb300.build.build()")
    lib = ctypes.CDLL(path)
    vp, i32, f32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    kvp = ctypes.POINTER(hs2_kv)
    lib.hs2_fa_select_workspace.argtypes = [i32, i32, kvp, i32, i32, i32]
    lib.hs2_fa_select_workspace.restype = sz
    lib.hs2_fa_select.argtypes = [vp, i32, i32, kvp, i32, i32, i32, f32, i32, vp, vp, vp, vp, vp, sz, vp, vp]
    lib.hs2_fa_select.restype = i32
    lib.hs2_fa_select_ex.argtypes = [vp, i32, i32, kvp, i32, i32, i32, f32, i32, i32, vp, vp, vp, vp, vp, sz, vp,
                                     vp]
    lib.hs2_fa_select_ex.restype = i32
    lib.hs2_sa_reuse_workspace.argtypes = [i32, i32, kvp, i32, i32, i32]
    lib.hs2_sa_reuse_workspace.restype = sz
    lib.hs2_sa_reuse.argtypes = [vp, i32, i32, kvp, i32, vp, vp, i32, f32, i32, vp, vp, sz, vp, vp]
    lib.hs2_sa_reuse.restype = i32
    lib.hs2_sa_reuse_ex.argtypes = [vp, i32, i32, kvp, i32, vp, vp, i32, f32, i32, vp, vp, i32, vp, vp, sz, vp, vp]
    lib.hs2_sa_reuse_ex.restype = i32
    lib.hs2_hier_reindex_workspace.argtypes = [i32, i32, kvp, i32, i32, i32, i32]
    lib.hs2_hier_reindex_workspace.restype = sz
    lib.hs2_hier_reindex.argtypes = [i32, vp, vp, i32, kvp, i32, i32, i32, i32, vp, vp, vp, vp, vp, sz, vp, vp]
    lib.hs2_hier_reindex.restype = i32
    lib.hs2_selftest_wait_timeout.argtypes = [i32, vp, vp]
    lib.hs2_selftest_wait_timeout.restype = i32
    lib.hs2_strerror.argtypes = [i32]
    lib.hs2_strerror.restype = ctypes.c_char_p
    lib.hs2_last_cuda_error.restype = i32
    lib.hs2_abi_version.restype = i32
    lib.hs2_profile_next.argtypes = [i32, vp, vp]
    lib.hs2_profile_next.restype = None
    lib.hs2_fa_select_noalloc.argtypes = [vp, i32, i32, kvp, i32, i32, i32, f32, i32, vp, vp, vp, vp, vp, vp]
    lib.hs2_fa_select_noalloc.restype = i32
    lib.hs2_kv_append.argtypes = [i32, kvp, ctypes.POINTER(vp), ctypes.POINTER(vp), vp, vp]
    lib.hs2_kv_append.restype = i32
    lib.hs2_fa_select_append.argtypes = [vp, i32, i32, kvp, i32, i32, i32, f32, i32, vp, vp, vp, vp, vp, vp, vp, sz,
                                         vp, vp]
    lib.hs2_fa_select_append.restype = i32
    lib.hs2_fa_select_noalloc_capacity.argtypes = []
    lib.hs2_fa_select_noalloc_capacity.restype = sz
    lib.hs2_fa_select_launches.argtypes = [i32, i32, kvp, i32, i32, i32, i32, i32, i32]
    lib.hs2_fa_select_launches.restype = i32
    lib.hs2_sa_reuse_launches.argtypes = [i32, i32, kvp, i32, i32, i32]
    lib.hs2_sa_reuse_launches.restype = i32
    if lib.hs2_abi_version() != ABI_VERSION:
        raise HS2Error(f"libhs2 ABI {lib.hs2_abi_version()} != binding ABI {ABI_VERSION}: rebuild the library")
    _lib = lib
    return lib


def _check(st: int) -> None:
    if st != 0:
        lib = load()
        msg = lib.hs2_strerror(st).decode()
        if st == -3:
            msg += f" (cudaError {lib.hs2_last_cuda_error()})"
        raise HS2Error(f"hs2 status {st}: {msg}")


def _ptr(t) -> int | None:
    return None if t is None else t.data_ptr()


def _stream(stream) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


@dataclass
class KV:
    """Device tensors of one group's paged KV cache."""

    k: torch.Tensor  # [num_pages][Hkv][64][d], float32, bfloat16 or uint8 (FP8 E4M3 codes);
    v: torch.Tensor | None  # FP4: uint8 [num_pages][Hkv][64][d/2], two E2M1 codes per byte
    block_table: torch.Tensor  # int32 [B][max_pages]
    seq_len: torch.Tensor  # int32 [B]
    k_scale: torch.Tensor | None = None  # FP8 / FP4: float32 [num_pages][Hkv]
    v_scale: torch.Tensor | None = None
    k_sf: torch.Tensor | None = None  # FP4: uint8 E4M3 [num_pages][Hkv][64][d/16]
    v_sf: torch.Tensor | None = None

    def c(self) -> hs2_kv:
        d = int(self.k.shape[3])
        if self.k.dtype == torch.uint8 and self.k_sf is not None:
            dt, d = FP4_E2M1, 2 * d
            if self.k_scale is None or (self.v is not None and (self.v_scale is None or self.v_sf is None)):
                raise HS2Error("an FP4 KV cache needs k_scale, v_scale, k_sf and v_sf")
        elif self.k.dtype == torch.uint8:
            dt = FP8_E4M3
            if self.k_scale is None or (self.v is not None and self.v_scale is None):
                raise HS2Error("an FP8 KV cache needs k_scale and v_scale")
        elif self.k.dtype in (torch.bfloat16, torch.float32):
            dt = BF16 if self.k.dtype == torch.bfloat16 else F32
        else:
            raise HS2Error(f"unsupported KV dtype {self.k.dtype}")
        for t in (self.k, self.v, self.block_table, self.seq_len, self.k_scale, self.v_scale, self.k_sf, self.v_sf):
            if t is not None and not t.is_contiguous():
                raise HS2Error("KV tensors must be contiguous")
        return hs2_kv(_ptr(self.k), _ptr(self.v), _ptr(self.block_table), _ptr(self.seq_len),
                      int(self.seq_len.shape[0]), int(self.k.shape[0]), int(self.block_table.shape[1]),
                      int(self.k.shape[2]), int(self.k.shape[1]), d, dt,
                      _ptr(self.k_scale), _ptr(self.v_scale), _ptr(self.k_sf), _ptr(self.v_sf))


def _workspace(nbytes: int, device, ws):
    if ws is not None:
        if ws.numel() * ws.element_size() < nbytes:
            raise HS2Error("workspace too small")
        return ws
    return torch.empty(max(nbytes, 256), dtype=torch.uint8, device=device)


def hs2_fa_select_workspace(B_or_n: int, Hq: int, kv: KV, max_t: int, k: int, prefill: bool = False) -> int:
    c = kv.c()
    return int(load().hs2_fa_select_workspace(B_or_n, Hq, ctypes.byref(c), max_t, k, int(prefill)))


def hs2_fa_select_launches(B_or_n: int, Hq: int, kv: KV, max_t: int, w: int, k: int, prefill: bool = False,
                           sel_block: int = 1, append: bool = False) -> int:
    """Kernels one hs2_fa_select call with these arguments launches (-1: rejected)."""
    c = kv.c()
    return int(load().hs2_fa_select_launches(B_or_n, Hq, ctypes.byref(c), max_t, w, k, int(prefill), sel_block,
                                              int(append)))


def hs2_sa_reuse_launches(B_or_n: int, Hq: int, kv: KV, w: int, k: int, prefill: bool = False) -> int:
    """Kernels one hs2_sa_reuse call with these arguments launches (-1: rejected)."""
    c = kv.c()
    return int(load().hs2_sa_reuse_launches(B_or_n, Hq, ctypes.byref(c), w, k, int(prefill)))


def hs2_kv_append(kvs, k_new, v_new=None, dev_err=None, stream=None) -> None:
    """Decode KV append for several caches in one launch: row t-1 (t = seq_len[b]) of
    every sequence of cache c takes k_new[c][b] / v_new[c][b] ([batch][Hkv][d], the cache's
    dtype). ``kvs``: list of KV (bf16 or f32 pools, written in place)."""
    lib = load()
    n = len(kvs)
    if n != len(k_new) or (v_new is not None and n != len(v_new)):
        raise HS2Error("one k_new (and v_new) tensor per cache")
    for kv, kn, vn in zip(kvs, k_new, v_new if v_new is not None else [None] * n):
        for x in (kn, vn):
            if x is not None and (not x.is_contiguous() or x.dtype != kv.k.dtype):
                raise HS2Error("new rows must be contiguous and of the cache's dtype")
    cs = (hs2_kv * n)(*[kv.c() for kv in kvs])
    kp = (ctypes.c_void_p * n)(*[_ptr(x) for x in k_new])
    vpa = (ctypes.c_void_p * n)(*[_ptr(x) for x in v_new]) if v_new is not None else None
    _check(lib.hs2_kv_append(n, cs, kp, vpa, _ptr(dev_err), _stream(stream)))


def hs2_fa_select(q: torch.Tensor, kv: KV, w: int, k: int, scale: float, prefill: bool = False,
                  max_t: int | None = None, out=None, workspace=None, dev_err=None, stream=None,
                  sel_block: int = 1, k_new: torch.Tensor | None = None, v_new: torch.Tensor | None = None):
    """FA layer + window-excluding top-k. Returns (o, lse, idx, idx_cnt) (float32, float32,
    int32, int32). ``max_t`` defaults to the table's capacity (decode) or n (prefill).
    ``sel_block`` > 1 selects whole blocks of that many far positions (``hs2_fa_select_ex``).
    ``k_new`` / ``v_new`` ([B][Hkv][d], decode): the current token's rows, appended to the
    cache at position t-1 by the same call (``hs2_fa_select_append``).
    ``dev_err`` (int32 device tensor) collects the device-side error bits (``DEV_*``). Every
    row gets its exact top-k: a prefill row whose streamed candidates cannot prove it is
    recomputed over its whole far range in the same call."""
    lib = load()
    Bq, Hq, d = q.shape
    c = kv.c()
    Hkv = c.Hkv
    if max_t is None:
        max_t = Bq if prefill else c.max_pages * c.page_size
    dev = q.device
    if out is None:
        o = torch.empty((Bq, Hq, d), dtype=torch.float32, device=dev)
        lse = torch.empty((Bq, Hq), dtype=torch.float32, device=dev)
        idx = torch.empty((Bq, Hkv, k), dtype=torch.int32, device=dev)
        cnt = torch.empty((Bq, Hkv), dtype=torch.int32, device=dev)
    else:
        o, lse, idx, cnt = out
    nb = int(lib.hs2_fa_select_workspace(Bq, Hq, ctypes.byref(c), max_t, k, int(prefill)))
    ws = _workspace(nb, dev, workspace)
    if k_new is not None:
        if prefill:
            raise HS2Error("the fused append is decode only")
        for x in (k_new, v_new):
            if x is None or not x.is_contiguous() or x.dtype != kv.k.dtype:
                raise HS2Error("k_new and v_new must be contiguous and of the cache's dtype")
        st = lib.hs2_fa_select_append(_ptr(q), Bq, Hq, ctypes.byref(c), max_t, w, k, float(scale), int(sel_block),
                                      _ptr(k_new), _ptr(v_new), _ptr(o), _ptr(lse), _ptr(idx), _ptr(cnt), _ptr(ws),
                                      ws.numel() * ws.element_size(), _ptr(dev_err), _stream(stream))
    elif sel_block == 1:
        st = lib.hs2_fa_select(_ptr(q), Bq, Hq, ctypes.byref(c), max_t, w, k, float(scale), int(prefill),
                               _ptr(o), _ptr(lse), _ptr(idx), _ptr(cnt), _ptr(ws), ws.numel() * ws.element_size(),
                               _ptr(dev_err), _stream(stream))
    else:
        st = lib.hs2_fa_select_ex(_ptr(q), Bq, Hq, ctypes.byref(c), max_t, w, k, float(scale), int(prefill),
                                  int(sel_block), _ptr(o), _ptr(lse), _ptr(idx), _ptr(cnt), _ptr(ws),
                                  ws.numel() * ws.element_size(), _ptr(dev_err), _stream(stream))
    _check(st)
    return o, lse, idx, cnt


def hs2_sa_reuse_workspace(B_or_n: int, Hq: int, kv: KV, w: int, k: int, prefill: bool = False) -> int:
    c = kv.c()
    return int(load().hs2_sa_reuse_workspace(B_or_n, Hq, ctypes.byref(c), w, k, int(prefill)))


def hs2_sa_reuse(q: torch.Tensor, kv: KV, w: int, idx: torch.Tensor, idx_cnt: torch.Tensor, k: int,
                 scale: float, prefill: bool = False, out=None, workspace=None, dev_err=None, stream=None,
                 sink: torch.Tensor | None = None, gate: torch.Tensor | None = None, overlap: bool = False):
    """SA layer reusing the FA's KV and indices with its own query. Returns o (float32).

    ``sink`` (float32 [Hq]) and ``gate`` (float32 [Bq][Hq][d]) are the optional per-head sink
    logits and output gate logits. ``overlap`` (``HS2_SA_OVERLAP``, the SA layers of a group
    after the first): idx, idx_cnt, the block table and the lengths were complete before the
    previous launch on the stream began, and ``workspace`` is the one the previous SA call on
    this stream used with the same sizes, so the decode kernel is one launch that may read
    them while that launch finishes. Without these three this is ``hs2_sa_reuse``, else
    ``hs2_sa_reuse_ex``."""
    lib = load()
    Bq, Hq, d = q.shape
    c = kv.c()
    o = out if out is not None else torch.empty((Bq, Hq, d), dtype=torch.float32, device=q.device)
    nb = int(lib.hs2_sa_reuse_workspace(Bq, Hq, ctypes.byref(c), w, k, int(prefill)))
    if overlap and workspace is None:
        raise HS2Error("overlap continues the previous SA call's workspace: pass it")
    ws = _workspace(nb, q.device, workspace)
    if sink is not None:
        assert sink.dtype == torch.float32 and sink.is_contiguous() and sink.numel() == Hq
    if gate is not None:
        assert gate.dtype == torch.float32 and gate.is_contiguous() and tuple(gate.shape) == (Bq, Hq, d)
    if sink is None and gate is None and not overlap:
        st = lib.hs2_sa_reuse(_ptr(q), Bq, Hq, ctypes.byref(c), w, _ptr(idx), _ptr(idx_cnt), k, float(scale),
                              int(prefill), _ptr(o), _ptr(ws), ws.numel() * ws.element_size(), _ptr(dev_err),
                              _stream(stream))
    else:
        st = lib.hs2_sa_reuse_ex(_ptr(q), Bq, Hq, ctypes.byref(c), w, _ptr(idx), _ptr(idx_cnt), k, float(scale),
                                 int(prefill), _ptr(sink), _ptr(gate), SA_OVERLAP if overlap else 0, _ptr(o),
                                 _ptr(ws), ws.numel() * ws.element_size(), _ptr(dev_err), _stream(stream))
    _check(st)
    return o


def hs2_hier_reindex_workspace(mode: int, Hi: int, k_idx: KV, max_t: int, k_top: int, blk: int,
                               max_blocks: int) -> int:
    c = k_idx.c()
    return int(load().hs2_hier_reindex_workspace(mode, Hi, ctypes.byref(c), max_t, k_top, blk, max_blocks))


def hs2_hier_reindex(mode: int, q_idx: torch.Tensor, w_idx: torch.Tensor, k_idx: KV, k_top: int, blk: int,
                     max_blocks: int, pool_blocks=None, pool_cnt=None, max_t: int | None = None, out=None,
                     workspace=None, dev_err=None, stream=None):
    """CSA2 hierarchical indexer (Full or Reindex). Returns (idx, idx_cnt, pool_blocks, pool_cnt)."""
    lib = load()
    B, Hi, di = q_idx.shape
    c = k_idx.c()
    dev = q_idx.device
    if max_t is None:
        max_t = c.max_pages * c.page_size
    if pool_blocks is None:
        pool_blocks = torch.empty((B, max_blocks), dtype=torch.int32, device=dev)
        pool_cnt = torch.empty((B,), dtype=torch.int32, device=dev)
    if out is None:
        idx = torch.empty((B, k_top), dtype=torch.int32, device=dev)
        cnt = torch.empty((B,), dtype=torch.int32, device=dev)
    else:
        idx, cnt = out
    nb = int(lib.hs2_hier_reindex_workspace(mode, Hi, ctypes.byref(c), max_t, k_top, blk, max_blocks))
    ws = _workspace(nb, dev, workspace)
    st = lib.hs2_hier_reindex(mode, _ptr(q_idx), _ptr(w_idx), Hi, ctypes.byref(c), max_t, k_top, blk,
                              max_blocks, _ptr(pool_blocks), _ptr(pool_cnt), _ptr(idx), _ptr(cnt), _ptr(ws),
                              ws.numel() * ws.element_size(), _ptr(dev_err), _stream(stream))
    _check(st)
    return idx, cnt, pool_blocks, pool_cnt


def hs2_profile_next(stage: int, start, stop) -> None:
    """Have the next call running ``stage`` record torch.cuda.Event ``start``/``stop`` around
    its main kernel (events must already have been recorded once so that they exist)."""
    load().hs2_profile_next(stage, start.cuda_event if start is not None else None,
                            stop.cuda_event if stop is not None else None)


def hs2_fa_select_noalloc(q: torch.Tensor, kv: KV, w: int, k: int, scale: float, prefill: bool = False,
                          max_t: int | None = None, out=None, dev_err=None, stream=None):
    """hs2_fa_select without a workspace, for callers that cannot allocate device memory:
    the library's own static scratch (hs2_fa_select_noalloc_capacity() bytes) is used.
    Only the outputs are allocated here when ``out`` is None; pass ``out`` to allocate
    nothing. Concurrent calls on the GPU race on the shared scratch."""
    lib = load()
    Bq, Hq, d = q.shape
    c = kv.c()
    if max_t is None:
        max_t = Bq if prefill else c.max_pages * c.page_size
    if out is None:
        dev = q.device
        out = (torch.empty((Bq, Hq, d), dtype=torch.float32, device=dev),
               torch.empty((Bq, Hq), dtype=torch.float32, device=dev),
               torch.empty((Bq, c.Hkv, k), dtype=torch.int32, device=dev),
               torch.empty((Bq, c.Hkv), dtype=torch.int32, device=dev))
    o, lse, idx, cnt = out
    st = lib.hs2_fa_select_noalloc(_ptr(q), Bq, Hq, ctypes.byref(c), max_t, w, k, float(scale), int(prefill),
                                   _ptr(o), _ptr(lse), _ptr(idx), _ptr(cnt), _ptr(dev_err), _stream(stream))
    _check(st)
    return o, lse, idx, cnt


def hs2_selftest_wait_timeout(timeout_us: int, dev_err: torch.Tensor, stream=None) -> None:
    """One warp waits (bounded, timeout_us) on an mbarrier nothing arrives on: the wait must
    give up and set DEV_TIMEOUT in dev_err."""
    _check(load().hs2_selftest_wait_timeout(int(timeout_us), _ptr(dev_err), _stream(stream)))

// sa_stream.cu — SA gather-attention (bf16) for decode as a persistent, warp-granular stream.
//
// Each SA query attends to its forced recent window and to the positions its group's FA
// layer selected, under one softmax, reading the group's shared KV in place through the
// paged block table ("HySparse2：整体架构、KV 生命周期与 PD 分离", §5 (Cross group), §7.2
// (SA reads window plus top-k), §7.4 (reuse of the FA layer's KV and indices)).
//
// Decode has one query row per sequence, so there are few (row, KV head) pairs and each
// covers |W ∪ S| = w + k entries. Here every pair's entries are cut into 16-entry steps
// (ms steps per pair, empty steps where a pair has fewer entries), the steps of all pairs
// are laid end to end, and each warp of a grid sized to fill the GPU takes one contiguous,
// equal range of them. A warp
//   1. resolves every entry of its range (window positions directly, selected positions
//      through the index array, then through the block table) into pool row ids in its
//      own shared memory, lane-parallel, in three rounds of independent loads;
//   2. streams its steps through a ring of kStrStages slots: cp.async copies of the 16 K
//      rows and 16 V rows (whole 256-byte rows, zero rows for invalid entries) into the
//      128-byte swizzle layout while it computes an earlier step (staged_attn.cuh:
//      ldmatrix fragments, S^T = K.Q^T and O^T += V^T.P^T on mma.sync, one online
//      softmax over all of a pair's entries), without any CTA-wide barrier;
//   3. at the end of each pair in its range, writes the pair's output directly when it
//      covered the whole pair, otherwise writes a partial (m, l, o) and arrives on the
//      pair's counter; the last warp to arrive merges the partials and resets the counter.
//      When that arrival ends the warp's range (the usual case: a pair's last partial comes
//      from a warp that ends with it), the merge is left to the end of the kernel, where the
//      CTA's warps share the recorded merges, two heads per warp and pass.
// The merges leave every counter zero, so a call that follows another on the same workspace
// needs no clearing launch between the two. The kernel is launched with programmatic stream
// serialization: it waits on the previous launch (griddep_wait) before its first read of
// anything that launch may write, and lets the next launch start once its own wait is over;
// with sp.early the row resolve (reads of the indices, counts, block table and lengths only)
// runs before that wait, overlapping the previous launch's tail.
#include <algorithm>

#include "common.cuh"
#include "kernels.h"
#include "staged_attn.cuh"

namespace hs2 {

constexpr int kStrStages = 2;     // ring slots per warp
constexpr int kStrMaxSteps = 32;  // steps per warp (row-id capacity 512 entries)

template <int D>
constexpr uint32_t str_slot_bytes() {  // 16 K rows and 16 V rows
  return 2u * (D / 64) * 2048u;
}
// Cache formats of the kernel: bf16 rows, FP8 E4M3 codes, FP4 E2M1 codes with E4M3 group scales.
constexpr int kFmtBf16 = 0, kFmtFp8 = 1, kFmtFp4 = 2;

template <int D, int FMT>
constexpr uint32_t str_raw_bytes() {
  // FP8: 16 K rows, 16 V rows (D bytes each), then 16 + 16 slab scales.
  // FP4: 16 K rows, 16 V rows (D/2 bytes each), 16 + 16 rows of D/16 group scales, then
  //      16 + 16 slab scales.
  return FMT == kFmtFp8 ? 2u * 16u * D + 128u : 18u * D + 128u;
}
template <int D, int FMT>
constexpr uint32_t str_ring_bytes() {  // per warp, a multiple of 1024
  return FMT != kFmtBf16 ? (str_slot_bytes<D>() + kStrStages * str_raw_bytes<D, FMT>() + 1023u) / 1024u * 1024u
                         : kStrStages * str_slot_bytes<D>();
}
template <int D, int FMT>
constexpr size_t str_warp_bytes() {  // ring + row ids + step table
  return (size_t)str_ring_bytes<D, FMT>() + (kStrMaxSteps * 16 + 6 * kStrMaxSteps) * sizeof(int32_t);
}
template <int D, int FMT>
constexpr size_t str_smem_bytes() {
  return 1024 + 4 * str_warp_bytes<D, FMT>();
}

// Warp holding global step s when `total` steps are cut into `nw` equal ranges
// [floor(total*w/nw), floor(total*(w+1)/nw)) (every range non-empty when nw <= total).
HS2_DEVI int warp_of_step(long long s, long long total, int nw) { return (int)(((s + 1) * nw - 1) / total); }


// FMT = kFmtFp8: the cache holds E4M3 codes with one scale per (page, KV head). A warp's ring
// then holds raw slots (the 16 K and 16 V rows at D bytes each, plus each entry's K and V
// scale, staged by cp.async) and one f16 slot: every step converts its raw slot into the f16
// slot (exact, the same swizzled layout) and computes from there with per-entry scales.
// FMT = kFmtFp4: the same with E2M1 rows (D/2 bytes) and their E4M3 scales of 16 channels
// staged too; the conversion multiplies each value by its group scale (exact in f16) and the
// slab scales act as FP8's.
// EPI = true: the SA layer has a sink bias or an output gate (sa_norm_factor, sa_gate); false
// keeps the plain 1 / L epilogue, whose smaller register footprint the streaming loop feels.
// Registers are held to three CTAs per SM where shared memory fits three (bf16 rings, and
// every format at D = 64); the FP8 / FP4 rings at D = 128 fit two.
template <int D, int FMT, bool EPI>
__global__ void __launch_bounds__(128, (FMT == kFmtBf16 || D == 64) ? 3 : 1)
    sa_stream_kernel(const AttnArgs a, const SaStreamArgs sp) {
  constexpr bool LOWP = FMT != kFmtBf16;
  constexpr int NT = 1;  // 8 query heads per unit
  constexpr int HALVES = D / 64;
  constexpr int CPR = D / 8;  // 16-byte chunks per bf16 / f16 row
  constexpr int CP8 = D / 16;  // 16-byte chunks per FP8 row
  constexpr int CP4 = D / 32;  // 16-byte chunks per FP4 row
  constexpr uint32_t kSlot = str_slot_bytes<D>();
  constexpr uint32_t kSlot8 = str_raw_bytes<D, FMT>();
  constexpr uint32_t kRing = str_ring_bytes<D, FMT>();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int gid = lane >> 2, tig = lane & 3;
  const int wid = blockIdx.x * 4 + warp;
  // pairs whose last partial arrives at the end of a warp's range; merged by the CTA's warps
  __shared__ int pend_s[4];
  if (wid >= sp.nwarps) return;
  if (lane == 0) pend_s[warp] = -1;
  if (!sp.early) griddep_wait();
  const int G = a.G, HG = sp.hg, ms = sp.ms;
  const long long total = sp.total;
  const long long s0 = total * wid / sp.nwarps, s1 = total * (wid + 1) / sp.nwarps;
  const int ns = (int)(s1 - s0);  // <= kStrMaxSteps (host-checked)

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = (uint32_t)__cvta_generic_to_shared(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  const uint32_t ring = base + (uint32_t)warp * kRing;  // bf16: the slots; FP8: the f16 slot, then raw slots
  uint8_t* ring_g = smem_raw + (base - raw) + (size_t)warp * kRing;  // the same bytes, generic address
  int32_t* rowid = reinterpret_cast<int32_t*>(smem_raw + (base - raw) + 4 * (size_t)kRing) +
                   warp * (kStrMaxSteps * 16 + 6 * kStrMaxSteps);
  int32_t* st_p = rowid + kStrMaxSteps * 16;  // step table: unit, step within the unit,
  int32_t* st_i = st_p + kStrMaxSteps;         // t, sequence, |W|, |S|
  int32_t* st_t = st_i + kStrMaxSteps;
  int32_t* st_b = st_t + kStrMaxSteps;
  int32_t* st_nw = st_b + kStrMaxSteps;
  int32_t* st_ns = st_nw + kStrMaxSteps;

  // ---- 1a. step table: lane j < ns describes step j (32-bit from here on)
  const int p_first = (int)(s0 / ms), i_first = (int)(s0 % ms);
  if (lane < ns) {
    const int ii = i_first + lane;
    const int un = p_first + ii / ms, i = ii % ms, p = un / HG;
    const QueryGeom qg = query_geom(p / a.Hkv, a.prefill, a.seq_len);
    const int c0 = __ldg(&a.cnt[p]);
    const int t = qg.t;
    int nW = 0, nS = 0;
    if (t < 1 || t > a.max_t || (t + kPage - 1) / kPage > a.max_pages) {
      if (i == 0) flag_error(a.dev_err, HS2_DEV_BAD_LENGTH);
    } else {
      nW = min(a.w, t);
      if (i == 0 && (c0 < 0 || c0 > a.kcap)) flag_error(a.dev_err, HS2_DEV_BAD_INDEX);
      nS = max(0, min(a.kcap, c0));
    }
    st_p[lane] = un;
    st_i[lane] = i;
    st_t[lane] = t;
    st_b[lane] = qg.b;
    st_nw[lane] = nW;
    st_ns[lane] = nS;
  }
  __syncwarp();
  // ---- 1b. resolve the range's entries (lane takes entries lane, lane + 32, ...) into
  // pool row ids: window positions directly, selected ones through the index array, then
  // every position through the block table
  {
    int posv[16], aux[16];  // aux: selected-index slot, or -1 (window / none)
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const int e = lane + 32 * j, st = e >> 4;
      posv[j] = -1;
      aux[j] = -1;
      if (st < ns) {
        const int u = 16 * st_i[st] + (e & 15), nW = st_nw[st];
        if (u < nW) posv[j] = st_t[st] - nW + u;
        else if (u < nW + st_ns[st]) aux[j] = u - nW;
      }
    }
    // all loads of a round are issued before any check (a flagged error is an atomic
    // that later loads could not be moved across)
    int selv[16];
#pragma unroll
    for (int j = 0; j < 16; ++j)
      selv[j] = aux[j] >= 0 ? __ldg(&a.idx[(size_t)(st_p[(lane + 32 * j) >> 4] / HG) * a.kcap + aux[j]]) : 0;
    bool bad_idx = false;
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      if (aux[j] >= 0) {
        const int t = st_t[(lane + 32 * j) >> 4];
        const int lim = a.w > 0 ? t - a.w : t;
        if (selv[j] < 0 || selv[j] >= lim) bad_idx = true;
        else posv[j] = selv[j];
      }
    }
    int physv[16];
#pragma unroll
    for (int j = 0; j < 16; ++j)
      physv[j] = posv[j] >= 0 ? __ldg(&a.bt[(size_t)st_b[(lane + 32 * j) >> 4] * a.max_pages + posv[j] / kPage]) : -1;
    bool bad_page = false;
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const int e = lane + 32 * j, st = e >> 4;
      if (st < ns) {
        int r = -1;
        if (posv[j] >= 0) {
          if (physv[j] < 0 || physv[j] >= a.num_pages) bad_page = true;
          else r = (physv[j] * a.Hkv + (st_p[st] / HG) % a.Hkv) * kPage + posv[j] % kPage;
        }
        rowid[e] = r;
      }
    }
    if (bad_idx) flag_error(a.dev_err, HS2_DEV_BAD_INDEX);
    if (bad_page) flag_error(a.dev_err, HS2_DEV_BAD_PAGE);
  }
  __syncwarp();
  // everything below reads or writes what the previous launch may touch (queries, the
  // partials and counters of a shared workspace, the output)
  if (sp.early) griddep_wait();
  griddep_launch_dependents();

  // ---- 2. stream the steps
  const __nv_bfloat16* kb = reinterpret_cast<const __nv_bfloat16*>(a.k);
  const __nv_bfloat16* vb = reinterpret_cast<const __nv_bfloat16*>(a.v);
  // the group's SA layers re-read the same rows: ask L2 to keep them
  const uint64_t keep = l2_keep_policy();
  auto issue = [&](int j, int slot) {
    if constexpr (FMT == kFmtFp4) {
      const uint32_t dst = ring + kSlot + (uint32_t)slot * kSlot8;
      const uint8_t* kb4 = reinterpret_cast<const uint8_t*>(a.k);
      const uint8_t* vb4 = reinterpret_cast<const uint8_t*>(a.v);
#pragma unroll
      for (int m = 0; m < 16 * CP4 / 32; ++m) {
        const int c = lane + 32 * m;
        const int r = c / CP4, cc = c % CP4;
        const int rid = rowid[16 * j + r];
        const size_t off = (size_t)(rid >= 0 ? rid : 0) * (D / 2) + 16 * cc;
        cp_async16_keep(dst + r * (D / 2) + 16 * cc, kb4 + off, rid >= 0, keep);
        cp_async16_keep(dst + 8 * D + r * (D / 2) + 16 * cc, vb4 + off, rid >= 0, keep);
      }
      // lanes 0-15: the entries' K group scales, lanes 16-31: their V group scales (D/16 bytes)
      const int rs = rowid[16 * j + (lane & 15)];
      const uint8_t* sfs = (lane < 16 ? a.k_sf : a.v_sf) + (size_t)(rs >= 0 ? rs : 0) * (D / 16);
      const uint32_t sfd = dst + 16 * D + (lane < 16 ? 0 : D) + (lane & 15) * (D / 16);
      if constexpr (D == 128) cp_async8(sfd, sfs, rs >= 0);
      else cp_async4(sfd, sfs, rs >= 0);
      const float* src = (lane < 16 ? a.k_scale : a.v_scale) + (rs >= 0 ? (rs >> 6) : 0);
      cp_async4(dst + 18 * D + 4 * lane, src, rs >= 0);
      return;
    }
    if (FMT == kFmtFp8) {
      const uint32_t dst = ring + kSlot + (uint32_t)slot * kSlot8;
      const uint8_t* kb8 = reinterpret_cast<const uint8_t*>(a.k);
      const uint8_t* vb8 = reinterpret_cast<const uint8_t*>(a.v);
#pragma unroll
      for (int m = 0; m < 16 * CP8 / 32; ++m) {
        const int c = lane + 32 * m;
        const int r = c / CP8, cc = c % CP8;
        const int rid = rowid[16 * j + r];
        const size_t off = (size_t)(rid >= 0 ? rid : 0) * D + 16 * cc;
        cp_async16_keep(dst + r * D + 16 * cc, kb8 + off, rid >= 0, keep);
        cp_async16_keep(dst + 16 * D + r * D + 16 * cc, vb8 + off, rid >= 0, keep);
      }
      // lanes 0-15: the entries' K scales, lanes 16-31: their V scales (page-head = row id / 64)
      const int rid = rowid[16 * j + (lane & 15)];
      const float* src = (lane < 16 ? a.k_scale : a.v_scale) + (rid >= 0 ? (rid >> 6) : 0);
      cp_async4(dst + 32 * D + 4 * lane, src, rid >= 0);
      return;
    }
    const uint32_t dst = ring + (uint32_t)slot * kSlot;
#pragma unroll
    for (int m = 0; m < 16 * CPR / 32; ++m) {
      const int c = lane + 32 * m;
      const int r = c / CPR, cc = c % CPR;
      const int rid = rowid[16 * j + r];
      const size_t off = (size_t)(rid >= 0 ? rid : 0) * D + 8 * cc;
      const uint32_t so = (uint32_t)(cc >> 3) * 2048u + sw128(r, cc & 7);
      cp_async16_keep(dst + so, kb + off, rid >= 0, keep);
      cp_async16_keep(dst + HALVES * 2048u + so, vb + off, rid >= 0, keep);
    }
  };
#pragma unroll
  for (int j = 0; j < kStrStages - 1; ++j) {
    if (j < ns) issue(j, j);
    cp_async_commit();
  }
  StagedAttn<D, 1, LOWP> at;
  int cur_p = -1;
  for (int j = 0; j < ns; ++j) {
    if (j + kStrStages - 1 < ns) issue(j + kStrStages - 1, (j + kStrStages - 1) % kStrStages);
    cp_async_commit();
    cp_async_wait<kStrStages - 1>();
    __syncwarp();
    const int un = st_p[j], i = st_i[j];
    const int p = un / HG, h0 = (un % HG) * 8, Gh = min(8, G - h0);  // pair, first head, heads
    if (un != cur_p) {
      const int qi = p / a.Hkv, g = p % a.Hkv;
      at.init(reinterpret_cast<const __nv_bfloat16*>(a.q) + ((size_t)qi * a.Hq + (size_t)g * G + h0) * D, Gh);
      cur_p = un;
    }
    const bool okA = rowid[16 * j + gid] >= 0, okB = rowid[16 * j + gid + 8] >= 0;
    if constexpr (FMT == kFmtFp4) {
      // raw slot -> f16 slot: a 16-byte FP4 chunk (32 values of row r, two groups of 16)
      // becomes four f16 chunks, each value times its group's E4M3 scale
      const uint8_t* src = ring_g + kSlot + (size_t)(j % kStrStages) * kSlot8;
#pragma unroll
      for (int part = 0; part < 2; ++part) {  // K, V
#pragma unroll
        for (int m = 0; m < 16 * CP4 / 32; ++m) {
          const int c = lane + 32 * m;
          const int r = c / CP4, cc = c % CP4;
          const uint4 raw4 = *reinterpret_cast<const uint4*>(src + part * 8 * D + r * (D / 2) + 16 * cc);
          const uint8_t* sfr = src + 16 * D + part * D + r * (D / 16) + 2 * cc;
          const uint32_t s0 = e4m3_pair(sfr[0], sfr[0]), s1 = e4m3_pair(sfr[1], sfr[1]);
          const uint32_t words[4] = {raw4.x, raw4.y, raw4.z, raw4.w};
          uint8_t* dst = ring_g + part * HALVES * 2048;
#pragma unroll
          for (int q = 0; q < 4; ++q) {  // 8 values -> one f16 chunk
            uint32_t h0, h1, h2, h3;
            fp4x8_to_f16x8(words[q], h0, h1, h2, h3);
            const uint32_t sq = q < 2 ? s0 : s1;
            const int f = 4 * cc + q;  // f16 chunk index of the row
            *reinterpret_cast<uint4*>(dst + (f >> 3) * 2048 + sw128(r, f & 7)) =
                make_uint4(hmul2(h0, sq), hmul2(h1, sq), hmul2(h2, sq), hmul2(h3, sq));
          }
        }
      }
      __syncwarp();
      const float* scl = reinterpret_cast<const float*>(src + 18 * D);
      if (__any_sync(0xffffffffu, okA || okB))
        at.step(ring, okA, okB, a.scale_log2, scl[gid], scl[gid + 8], scl[16 + gid], scl[16 + gid + 8]);
    } else if (FMT == kFmtFp8) {
      // raw slot -> f16 slot: a 16-byte FP8 chunk (16 values of row r) becomes two f16 chunks
      const uint8_t* src = ring_g + kSlot + (size_t)(j % kStrStages) * kSlot8;
#pragma unroll
      for (int part = 0; part < 2; ++part) {  // K, V
#pragma unroll
        for (int m = 0; m < 16 * CP8 / 32; ++m) {
          const int c = lane + 32 * m;
          const int r = c / CP8, cc = c % CP8;
          const uint4 raw8 = *reinterpret_cast<const uint4*>(src + part * 16 * D + r * D + 16 * cc);
          const uint4 lo = fp8x8_to_f16x8(make_uint2(raw8.x, raw8.y));
          const uint4 hi = fp8x8_to_f16x8(make_uint2(raw8.z, raw8.w));
          const int f0 = 2 * cc, f1 = 2 * cc + 1;  // f16 chunk indices of the row
          uint8_t* dst = ring_g + part * HALVES * 2048;
          *reinterpret_cast<uint4*>(dst + (f0 >> 3) * 2048 + sw128(r, f0 & 7)) = lo;
          *reinterpret_cast<uint4*>(dst + (f1 >> 3) * 2048 + sw128(r, f1 & 7)) = hi;
        }
      }
      __syncwarp();
      const float* scl = reinterpret_cast<const float*>(src + 32 * D);
      if (__any_sync(0xffffffffu, okA || okB))
        at.step(ring, okA, okB, a.scale_log2, scl[gid], scl[gid + 8], scl[16 + gid], scl[16 + gid + 8]);
    } else if (__any_sync(0xffffffffu, okA || okB)) {
      at.step(ring + (uint32_t)(j % kStrStages) * kSlot, okA, okB, a.scale_log2);
    }
    __syncwarp();
    if (i != ms - 1 && j != ns - 1) continue;

    // ---- 3. the pair ends in this range: write its output or a partial
    const int qi = p / a.Hkv, g = p % a.Hkv;
    const int first = warp_of_step((long long)un * ms, total, sp.nwarps);
    const int last = warp_of_step((long long)(un + 1) * ms - 1, total, sp.nwarps);
    float lsum[NT][2];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int hs = 0; hs < 2; ++hs) {
        float lv = at.l[nt][hs];
        lv += __shfl_xor_sync(0xffffffffu, lv, 4);
        lv += __shfl_xor_sync(0xffffffffu, lv, 8);
        lv += __shfl_xor_sync(0xffffffffu, lv, 16);
        lsum[nt][hs] = lv;
      }
    float* out = a.out_o + ((size_t)qi * a.Hq + (size_t)g * G + h0) * D;
    if (first == last) {
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int hs = 0; hs < 2; ++hs) {
          const int hl = nt * 8 + 2 * tig + hs;
          if (hl < Gh) {
            if constexpr (EPI) {
              const int hq = g * G + h0 + hl;  // query head
              const float inv = sa_norm_factor(at.m[nt][hs], lsum[nt][hs], sink_b2(a.sink, hq)) * at.unit();
              const float* gl = a.gate ? a.gate + ((size_t)qi * a.Hq + hq) * D : nullptr;
#pragma unroll
              for (int mt = 0; mt < D / 16; ++mt) {
                const int d0 = 16 * mt + gid;
                out[hl * D + d0] = at.acc[mt][nt][hs] * inv * (gl ? sa_gate(gl[d0]) : 1.f);
                out[hl * D + d0 + 8] = at.acc[mt][nt][hs + 2] * inv * (gl ? sa_gate(gl[d0 + 8]) : 1.f);
              }
            } else {
              const float inv = (lsum[nt][hs] > 0.f ? 1.f / lsum[nt][hs] : 0.f) * at.unit();
#pragma unroll
              for (int mt = 0; mt < D / 16; ++mt) {
                out[hl * D + 16 * mt + gid] = at.acc[mt][nt][hs] * inv;
                out[hl * D + 16 * mt + gid + 8] = at.acc[mt][nt][hs + 2] * inv;
              }
            }
          }
        }
      continue;
    }
    const int slotc = wid - first, nc = last - first + 1;
    const size_t pbase = ((size_t)un * sp.maxc + slotc) * 8;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int hs = 0; hs < 2; ++hs) {
        const int hl = nt * 8 + 2 * tig + hs;
        if (hl < Gh) {
          if (gid == 0) a.part_ml[pbase + hl] = make_float2(at.m[nt][hs], lsum[nt][hs]);
          float* po = a.part_o + (pbase + hl) * D;
#pragma unroll
          for (int mt = 0; mt < D / 16; ++mt) {
            po[16 * mt + gid] = at.acc[mt][nt][hs] * at.unit();
            po[16 * mt + gid + 8] = at.acc[mt][nt][hs + 2] * at.unit();
          }
        }
      }
    __threadfence();
    __syncwarp();
    int is_last = 0;
    if (lane == 0) is_last = atomicAdd(&a.arrive[un], 1) == nc - 1;
    is_last = __shfl_sync(0xffffffffu, is_last, 0);
    if (!is_last) continue;
    if (j == ns - 1) {  // the range ends here: the CTA's warps merge it together below
      if (lane == 0) {
        pend_s[warp] = un;
        a.arrive[un] = 0;
      }
      __threadfence();
      continue;
    }
    __threadfence();
    // merge (nc <= 32): lane r holds partial r's (m, l) of each head; lanes then sweep the
    // heads' D columns four at a time, weights broadcast by shuffle
    const size_t p0 = (size_t)un * sp.maxc * 8;
    float2 mlv[8];
#pragma unroll
    for (int h = 0; h < 8; ++h)
      mlv[h] = (lane < nc && h < Gh) ? __ldcg(&a.part_ml[p0 + (size_t)lane * 8 + h]) : make_float2(-INFINITY, 0.f);
    float f[8], inv[8];
#pragma unroll
    for (int h = 0; h < 8; ++h) {
      const float M = warp_max(mlv[h].x);
      f[h] = lane < nc ? exp2_rel(mlv[h].x, M) : 0.f;
      const float L = warp_sum(f[h] * mlv[h].y);
      if constexpr (EPI) inv[h] = sa_norm_factor(M, L, h < Gh ? sink_b2(a.sink, g * G + h0 + h) : -INFINITY);
      else inv[h] = L > 0.f ? 1.f / L : 0.f;
    }
    float4 o4[8];
#pragma unroll
    for (int h = 0; h < 8; ++h) o4[h] = make_float4(0.f, 0.f, 0.f, 0.f);
    const float* pob = a.part_o + p0 * D + 4 * lane;
#pragma unroll 2
    for (int r = 0; r < nc; ++r) {
#pragma unroll
      for (int h = 0; h < 8; ++h) {
        const float fr = __shfl_sync(0xffffffffu, f[h], r);
        if (h < Gh && 4 * lane < D) {
          const float4 v = __ldcg(reinterpret_cast<const float4*>(pob + ((size_t)r * 8 + h) * D));
          o4[h].x += fr * v.x;
          o4[h].y += fr * v.y;
          o4[h].z += fr * v.z;
          o4[h].w += fr * v.w;
        }
      }
    }
#pragma unroll
    for (int h = 0; h < 8; ++h)
      if (h < Gh && 4 * lane < D) {
        float4 r4 = make_float4(o4[h].x * inv[h], o4[h].y * inv[h], o4[h].z * inv[h], o4[h].w * inv[h]);
        if (EPI && a.gate) {
          const float4 g4 = __ldg(reinterpret_cast<const float4*>(a.gate + ((size_t)qi * a.Hq + g * G + h0 + h) * D) + lane);
          r4.x *= sa_gate(g4.x);
          r4.y *= sa_gate(g4.y);
          r4.z *= sa_gate(g4.z);
          r4.w *= sa_gate(g4.w);
        }
        *reinterpret_cast<float4*>(out + h * D + 4 * lane) = r4;
      }
    if (lane == 0) a.arrive[un] = 0;
  }
  cp_async_wait<0>();

  // ---- 4. the merges recorded at range ends finish the kernel: the CTA's active warps take
  // them together, two heads per warp and pass, loading eight partials per head at once
  const int cta_warps = min(4, sp.nwarps - (int)blockIdx.x * 4);
  named_barrier_sync(1, 32 * cta_warps);
  __threadfence();
  for (int e = warp;; e += cta_warps) {
    int want = e >> 2, un = -1;  // item e: pending pair e / 4 (in warp order), heads 2 (e % 4) + {0, 1}
    for (int w2 = 0; w2 < cta_warps; ++w2)
      if (pend_s[w2] >= 0) {
        if (want == 0) {
          un = pend_s[w2];
          break;
        }
        --want;
      }
    if (un < 0) break;
    const int p = un / HG, h0 = (un % HG) * 8, Gh = min(8, G - h0);
    const int ha = 2 * (e & 3);
    if (ha >= Gh) continue;
    const int qi = p / a.Hkv, g = p % a.Hkv;
    const int first = warp_of_step((long long)un * ms, total, sp.nwarps);
    const int last = warp_of_step((long long)(un + 1) * ms - 1, total, sp.nwarps);
    const int nc = last - first + 1;
    const size_t p0 = (size_t)un * sp.maxc * 8;
    float f[2], inv[2];
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      const int h = ha + hh;
      const float2 ml = (lane < nc && h < Gh) ? __ldcg(&a.part_ml[p0 + (size_t)lane * 8 + h]) : make_float2(-INFINITY, 0.f);
      const float M = warp_max(ml.x);
      f[hh] = lane < nc ? exp2_rel(ml.x, M) : 0.f;
      const float L = warp_sum(f[hh] * ml.y);
      if constexpr (EPI) inv[hh] = sa_norm_factor(M, L, h < Gh ? sink_b2(a.sink, g * G + h0 + h) : -INFINITY);
      else inv[hh] = L > 0.f ? 1.f / L : 0.f;
    }
    float4 o4[2] = {make_float4(0.f, 0.f, 0.f, 0.f), make_float4(0.f, 0.f, 0.f, 0.f)};
    const float* pob = a.part_o + p0 * D + 4 * lane;
    for (int r0 = 0; r0 < nc; r0 += 8) {
      float4 v[8][2];
#pragma unroll
      for (int q = 0; q < 8; ++q)
#pragma unroll
        for (int hh = 0; hh < 2; ++hh)
          v[q][hh] = (r0 + q < nc && ha + hh < Gh && 4 * lane < D)
                         ? __ldcg(reinterpret_cast<const float4*>(pob + ((size_t)(r0 + q) * 8 + ha + hh) * D))
                         : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int q = 0; q < 8; ++q)
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const float fr = __shfl_sync(0xffffffffu, f[hh], (r0 + q) & 31);
          o4[hh].x += fr * v[q][hh].x;
          o4[hh].y += fr * v[q][hh].y;
          o4[hh].z += fr * v[q][hh].z;
          o4[hh].w += fr * v[q][hh].w;
        }
    }
    float* out = a.out_o + ((size_t)qi * a.Hq + (size_t)g * G + h0) * D;
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      const int h = ha + hh;
      if (h < Gh && 4 * lane < D) {
        float4 r4 = make_float4(o4[hh].x * inv[hh], o4[hh].y * inv[hh], o4[hh].z * inv[hh], o4[hh].w * inv[hh]);
        if (EPI && a.gate) {
          const float4 g4 = __ldg(reinterpret_cast<const float4*>(a.gate + ((size_t)qi * a.Hq + g * G + h0 + h) * D) + lane);
          r4.x *= sa_gate(g4.x);
          r4.y *= sa_gate(g4.y);
          r4.z *= sa_gate(g4.z);
          r4.w *= sa_gate(g4.w);
        }
        *reinterpret_cast<float4*>(out + h * D + 4 * lane) = r4;
      }
    }
  }
}

template <int D, int FMT>
static bool stream_plan_t(int G, int w, int k, int Bq, int Hkv, SaStreamArgs* sp, int* grid) {
  int dev = 0, sms = 0, per_sm = 0, per_sm2 = 0;
  const size_t sm = str_smem_bytes<D, FMT>();
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
      cudaFuncSetAttribute(sa_stream_kernel<D, FMT, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm) !=
          cudaSuccess ||
      cudaFuncSetAttribute(sa_stream_kernel<D, FMT, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm) !=
          cudaSuccess ||
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, sa_stream_kernel<D, FMT, true>, 128, sm) != cudaSuccess ||
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm2, sa_stream_kernel<D, FMT, false>, 128, sm) != cudaSuccess ||
      std::min(per_sm, per_sm2) < 1) {
    (void)cudaGetLastError();
    return false;
  }
  per_sm = std::min(per_sm, per_sm2);  // the grid is sized for the variant with fewer resident CTAs
  const int hg = (G + 7) / 8;  // units of 8 query heads per (row, KV head)
  const int ms = (w + k + 15) / 16;
  const long long total = (long long)Bq * Hkv * hg * ms;
  if (total < 1) return false;
  const long long resident = 4LL * sms * per_sm;  // every warp of the grid resident at once
  long long nw = std::min(resident, total);
  long long per = total / nw;  // >= 1; ranges hold per or per + 1 steps
  // at most 32 warps share a unit (the merge holds one partial per lane), and at least 4
  // steps per warp: on small problems (few units) a unit split over many short warps ends
  // in a long merge of many partials, which is the critical path
  const long long per_min = std::max<long long>((ms + 30) / 31, std::min<long long>(4, ms));
  if (per < per_min) {
    per = per_min;
    nw = std::max(1LL, total / per);
    per = total / nw;
  }
  if ((total + nw - 1) / nw > kStrMaxSteps) return false;
  sp->nwarps = (int)nw;
  sp->hg = hg;
  sp->ms = ms;
  sp->total = total;
  sp->maxc = (int)((ms + per - 1) / per + 1);
  *grid = (int)((nw + 3) / 4);
  return true;
}

template <int FMT>
static bool stream_plan_f(int G, int D, int w, int k, int Bq, int Hkv, SaStreamArgs* sp, int* grid) {
  return D == 128 ? stream_plan_t<128, FMT>(G, w, k, Bq, Hkv, sp, grid)
                  : stream_plan_t<64, FMT>(G, w, k, Bq, Hkv, sp, grid);
}

// kv_dtype: 1 bf16, 2 FP8 E4M3, 3 FP4 E2M1 (others: not this kernel)
bool sa_stream_plan(int G, int D, int kv_dtype, int w, int k, int Bq, int Hkv, SaStreamArgs* sp, int* grid) {
  if (kv_dtype < 1 || kv_dtype > 3 || (D != 64 && D != 128) || G < 1 || G > 32) return false;
  if (kv_dtype == 2) return stream_plan_f<kFmtFp8>(G, D, w, k, Bq, Hkv, sp, grid);
  if (kv_dtype == 3) return stream_plan_f<kFmtFp4>(G, D, w, k, Bq, Hkv, sp, grid);
  return stream_plan_f<kFmtBf16>(G, D, w, k, Bq, Hkv, sp, grid);
}

template <int D, int FMT>
static cudaError_t launch_stream_t(const AttnArgs& a, const SaStreamArgs& sp, int grid, cudaStream_t s) {
  const size_t sm = str_smem_bytes<D, FMT>();
  auto kern = (a.sink || a.gate) ? sa_stream_kernel<D, FMT, true> : sa_stream_kernel<D, FMT, false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
  if (e != cudaSuccess) return e;
  return launch_pdl(kern, dim3(grid), dim3(128), sm, s, a, sp);
}

template <int FMT>
static cudaError_t launch_stream_f(const AttnArgs& a, const SaStreamArgs& sp, int grid, cudaStream_t s) {
  if (a.D == 128) return launch_stream_t<128, FMT>(a, sp, grid, s);
  if (a.D == 64) return launch_stream_t<64, FMT>(a, sp, grid, s);
  return cudaErrorInvalidValue;
}

cudaError_t launch_sa_stream(const AttnArgs& a, const SaStreamArgs& sp, int grid, cudaStream_t s) {
  if (a.k_sf) return launch_stream_f<kFmtFp4>(a, sp, grid, s);
  if (a.k_scale) return launch_stream_f<kFmtFp8>(a, sp, grid, s);
  return launch_stream_f<kFmtBf16>(a, sp, grid, s);
}
}  // namespace hs2

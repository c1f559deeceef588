// fa_decode.cu — bf16 / FP8 / FP4 split-KV scan of the FA layer (decode and causal rows).
//
// The FA layer of a HySparse2 Cross group attends to every visible key of the group's
// shared paged KV ("HySparse2：整体架构、KV 生命周期与 PD 分离", §5; §16.1: the FA layers
// still scan the whole history at decode). This kernel streams K and V pages straight
// from HBM into registers with 128-bit loads; the head-sharing contraction (the query
// heads of one KV head) runs on mma.sync with the keys as the M dimension, so no MMA
// row is padding. It writes per-split softmax partials and the base-2 logits that the
// selection (combine.cu) needs once the per-head normaliser is known.
#include <algorithm>

#include "common.cuh"
#include "kernels.h"
#include "mma_attn.cuh"

namespace hs2 {

// ============================================================================ bf16 split-KV FA
// Per CTA: one (query, KV head, split of `pps` pages); 4 warps take the split's pages
// round-robin; per warp step: 16 keys (see mma_attn.cuh for the register mappings).
// FMT = kFaFp8: the cache holds E4M3 codes with one scale per (page, KV head); rows load at
// half the bytes and convert to f16 (exact), the page's K scale multiplies the logits and its
// V scale the weights entering P.V (mma_attn.cuh, F16 mode). FMT = kFaFp4: E2M1 codes (a
// quarter of the bytes) with an E4M3 scale per 16 channels of a row, each value times its
// group scale in f16 (exact), the slab scales as FP8's.
constexpr int kFaBf16 = 0, kFaFp8 = 1, kFaFp4 = 2;
constexpr int kRing8 = 3;  // low-precision chunk slots per warp
// one low-precision slot: 16 K rows, 16 V rows, (FP4) their group scales, then k scale,
// v scale, key0 (padded to 16 bytes)
template <int D, int FMT>
constexpr int fa8_slot_bytes() { return FMT == kFaFp4 ? 2 * 8 * D + 2 * D + 16 : 2 * 16 * D + 16; }

template <int D, int NT, int FMT>
__global__ void __launch_bounds__(128, (FMT != kFaBf16 && NT == 1) ? 4 : 0) fa_decode_mma_kernel(const AttnArgs a) {
  constexpr bool FP8 = FMT != kFaBf16;  // a low-precision cache (the f16 MMA path)
  using Attn = MmaAttn<D, NT, FP8>;
  constexpr int KC = Attn::KC, VC = Attn::VC;
  const int qi = blockIdx.z, g = blockIdx.y, split = blockIdx.x;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int gid = lane >> 2, tig = lane & 3;
  const QueryGeom qg = query_geom(qi, a.prefill, a.seq_len);
  const int t = qg.t;
  const int npages = (t + kPage - 1) / kPage;
  const int page0 = split * a.pps;
  if (t < 1 || t > a.max_t || npages > a.max_pages || page0 >= npages) return;  // flagged by the combine
  const int page1 = min(npages, page0 + a.pps);
  const int G = a.G;

  extern __shared__ float smem[];
  float* sm_m = smem;                  // [4][NT*8]
  float* sm_l = sm_m + 4 * NT * 8;     // [4][NT*8]
  float* sm_o = sm_l + 4 * NT * 8;     // [4][NT*8][D]

  Attn at;
  at.init(reinterpret_cast<const __nv_bfloat16*>(a.q) + ((size_t)qi * a.Hq + (size_t)g * G) * D, G);

  const int32_t* bt = a.bt + (size_t)qg.b * a.max_pages;
  const size_t head_stride = (size_t)kPage * D;  // elements per (page, KV head)
  const size_t lrow = (size_t)qi * a.Hq + (size_t)g * G;  // the pair's first head row
  uint16_t* code_base = a.lcode ? a.lcode + lrow * a.ld_logits : nullptr;
  float* max_base = a.lcode ? a.lmax + lrow * (a.ld_logits / kLogitGroup) : nullptr;

  // The K/V stream is read once: evict it first. The logit codes are read by the selection
  // right after this kernel: keep them.
  const uint64_t pol_stream = l2_first_policy(), pol_keep = l2_keep_policy();
  // one 16-key group's logits for the selection: codes below the group's per-head max
  // (logit_code), and the max itself (lanes 0-3, two heads each)
  auto write_logits = [&](const float (&x)[NT][4], const float (&gm)[NT][2], int key0, bool okA, bool okB) {
    if (!code_base) return;
    const int keyA = key0 + gid, keyB = keyA + 8;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
      for (int hs = 0; hs < 2; ++hs) {
        const int h = nt * 8 + 2 * tig + hs;
        if (h < G) {
          uint16_t* row = code_base + (size_t)h * a.ld_logits;
          if (okA) stg_u16_pol(row + keyA, logit_code(x[nt][hs], gm[nt][hs]), pol_keep);
          if (okB) stg_u16_pol(row + keyB, logit_code(x[nt][hs + 2], gm[nt][hs]), pol_keep);
          if (gid == 0) stg_f32_pol(max_base + (size_t)h * (a.ld_logits / kLogitGroup) + key0 / kLogitGroup,
                                    gm[nt][hs], pol_keep);
        }
      }
    }
  };

  if constexpr (!FP8) {
    const bool append = a.k_new != nullptr;  // decode only (the host refuses it for prefill)
    const size_t row_new = ((size_t)qi * a.Hkv + g) * D;
    const __nv_bfloat16* k_new_row = append ? reinterpret_cast<const __nv_bfloat16*>(a.k_new) + row_new : nullptr;
    const __nv_bfloat16* v_new_row = append ? reinterpret_cast<const __nv_bfloat16*>(a.v_new) + row_new : nullptr;
    for (int page = page0 + warp; page < page1; page += 4) {
      const int phys = bt[page];
      if (phys < 0 || phys >= a.num_pages) {
        if (lane == 0) flag_error(a.dev_err, HS2_DEV_BAD_PAGE);
        continue;
      }
      const __nv_bfloat16* kp = reinterpret_cast<const __nv_bfloat16*>(a.k) + ((size_t)phys * a.Hkv + g) * head_stride;
      const __nv_bfloat16* vp = reinterpret_cast<const __nv_bfloat16*>(a.v) + ((size_t)phys * a.Hkv + g) * head_stride;
#pragma unroll 1
      for (int ch = 0; ch < 4; ++ch) {
        const int key0 = page * kPage + ch * 16;
        if (key0 >= t) break;
        const int r0 = ch * 16 + gid;  // row within the page
        // fused append: the chunk holding key t-1 takes that row from k_new / v_new instead
        // of the pool (which this kernel then writes; no lane reads it from the pool)
        const bool tail = append && key0 + 16 >= t;
        const __nv_bfloat16* kA = kp + (size_t)r0 * D;
        const __nv_bfloat16* kB = kp + (size_t)(r0 + 8) * D;
        if (tail) {
          if (key0 + gid == t - 1) kA = k_new_row;
          if (key0 + gid + 8 == t - 1) kB = k_new_row;
        }
        uint4 kr0[KC], kr1[KC], vr[4][VC];
#pragma unroll
        for (int j = 0; j < KC; ++j) {
          kr0[j] = ldg_nc_v4_keep(kA + 32 * j + 8 * tig, pol_stream);
          kr1[j] = ldg_nc_v4_keep(kB + 32 * j + 8 * tig, pol_stream);
        }
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int vrow = ch * 16 + 2 * tig + (e & 1) + 8 * (e >> 1);
          const __nv_bfloat16* vsrc = (tail && page * kPage + vrow == t - 1) ? v_new_row : vp + (size_t)vrow * D;
#pragma unroll
          for (int j = 0; j < VC; ++j) vr[e][j] = ldg_nc_v4_keep(vsrc + (D / 8) * gid + 8 * j, pol_stream);
        }
        if (tail) {  // write-through of the new rows (each element by exactly one lane)
          __nv_bfloat16* kw = const_cast<__nv_bfloat16*>(kp) + (size_t)((t - 1) % kPage) * D;
          if (key0 + gid == t - 1)
#pragma unroll
            for (int j = 0; j < KC; ++j) *reinterpret_cast<uint4*>(kw + 32 * j + 8 * tig) = kr0[j];
          if (key0 + gid + 8 == t - 1)
#pragma unroll
            for (int j = 0; j < KC; ++j) *reinterpret_cast<uint4*>(kw + 32 * j + 8 * tig) = kr1[j];
          __nv_bfloat16* vw = const_cast<__nv_bfloat16*>(vp) + (size_t)((t - 1) % kPage) * D;
#pragma unroll
          for (int e = 0; e < 4; ++e)
            if (page * kPage + ch * 16 + 2 * tig + (e & 1) + 8 * (e >> 1) == t - 1)
#pragma unroll
              for (int j = 0; j < VC; ++j) *reinterpret_cast<uint4*>(vw + (D / 8) * gid + 8 * j) = vr[e][j];
        }
        if (key0 + 16 > t) {  // rows past t: never read their values
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int key = key0 + 2 * tig + (e & 1) + 8 * (e >> 1);
            if (key >= t)
#pragma unroll
              for (int j = 0; j < VC; ++j) vr[e][j] = make_uint4(0, 0, 0, 0);
          }
        }
        const int keyA = key0 + gid, keyB = key0 + gid + 8;
        const bool okA = keyA < t, okB = keyB < t;
        float x[NT][4];
        at.step(kr0, kr1, vr, okA, okB, a.scale_log2, x);
        write_logits(x, at.gmax, key0, okA, okB);
      }
    }
  } else {
    // FP8: each warp streams its 16-key chunks through a ring of kRing8 shared-memory slots
    // filled by 16-byte cp.async copies, so kRing8 - 1 chunks (12 KB at d = 128) are in
    // flight per warp without holding registers. The 16-byte units of a row are stored
    // XOR-swizzled by the row, which keeps the fragment reads below free of bank conflicts.
    constexpr bool FP4 = FMT == kFaFp4;
    constexpr int RB = FP4 ? D / 2 : D;  // bytes per row of codes
    constexpr int CB = 16 * RB;          // bytes of K (or V) codes in one chunk
    constexpr int SFB = FP4 ? D : 0;     // bytes of K (or V) group scales in one chunk (16 rows x D/16)
    constexpr int FT = 2 * CB + 2 * SFB; // the footer: k scale, v scale, key0
    constexpr int UPR = RB / 16;         // 16-byte units per row
    constexpr int SLOT = fa8_slot_bytes<D, FMT>();
    const uint32_t ring = (uint32_t)__cvta_generic_to_shared(smem) + (uint32_t)(warp * kRing8 * SLOT);
    const uint8_t* ring_p = reinterpret_cast<const uint8_t*>(smem) + warp * kRing8 * SLOT;
    // 16-byte units XOR-swizzled by row: 8 consecutive rows hit 8 distinct bank groups
    auto swz = [](int row) {
      if constexpr (FP4) return D == 128 ? ((row >> 1) & 3) : ((row >> 2) & 1);
      else return D == 128 ? (row & 7) : ((row >> 1) & 3);
    };
    auto unit_off = [&](int row, int c) { return row * RB + ((c ^ swz(row)) << 4); };
    float v_unit = 1.f;  // acc holds P.V in units of this V scale

    // first page >= pg of this warp with a valid block-table entry (bad ones are flagged)
    auto good_page = [&](int pg, int& phys) {
      for (; pg < page1; pg += 4) {
        phys = bt[pg];
        if (phys >= 0 && phys < a.num_pages) break;
        if (lane == 0) flag_error(a.dev_err, HS2_DEV_BAD_PAGE);
      }
      return pg;
    };
    // copies of chunk (pg, ch) into a slot: K, V, then the page's two scales and key0
    auto issue = [&](int pg, int phys, int ch, int slot) {
      const uint32_t sl = ring + slot * SLOT;
      const size_t ph = (size_t)phys * a.Hkv + g;
      const uint8_t* kp = reinterpret_cast<const uint8_t*>(a.k) + ph * kPage * RB + (size_t)ch * CB;
      const uint8_t* vp = reinterpret_cast<const uint8_t*>(a.v) + ph * kPage * RB + (size_t)ch * CB;
#pragma unroll
      for (int i = 0; i < CB / 512; ++i) {
        const int u = lane + 32 * i, off = unit_off(u / UPR, u % UPR);
        cp_async16_keep(sl + off, kp + 16 * u, true, pol_stream);
        cp_async16_keep(sl + CB + off, vp + 16 * u, true, pol_stream);
      }
      if constexpr (FP4) {  // the chunk's 16 rows of group scales: D/16 16-byte units each for K and V
        const size_t so = (ph * kPage + (size_t)ch * 16) * (D / 16);
        if (lane < D / 16) cp_async16(sl + 2 * CB + 16 * lane, a.k_sf + so + 16 * lane, true);
        else if (lane >= 16 && lane < 16 + D / 16)
          cp_async16(sl + 2 * CB + SFB + 16 * (lane - 16), a.v_sf + so + 16 * (lane - 16), true);
      }
      if (lane == 0) cp_async4(sl + FT, a.k_scale + ph, true);
      if (lane == 1) cp_async4(sl + FT + 4, a.v_scale + ph, true);
      if (lane == 2) st_shared_s32(sl + FT + 8, pg * kPage + ch * 16);
    };
    auto compute = [&](int slot) {
      const uint8_t* sl = ring_p + slot * SLOT;
      const float ks = *reinterpret_cast<const float*>(sl + FT);
      const float vs = *reinterpret_cast<const float*>(sl + FT + 4);
      const int key0 = *reinterpret_cast<const int*>(sl + FT + 8);
      if (vs != v_unit && vs != 0.f) {  // acc moves to this page's V scale as its unit
        at.scale_acc(v_unit / vs);
        v_unit = vs;
      }
      uint4 kr0[KC], kr1[KC];
      if constexpr (FP4) {
        // 8 values (4 bytes) of rows gid and gid + 8 at channel 32j + 8tig, i.e. unit j,
        // byte 4tig; times the E4M3 scale of group 2j + tig/2 of that row
        const uint8_t* ksf = sl + 2 * CB;
#pragma unroll
        for (int j = 0; j < KC; ++j) {
          const int grp = 2 * j + (tig >> 1);
          const uint32_t sA = e4m3_pair(ksf[gid * (D / 16) + grp], ksf[gid * (D / 16) + grp]);
          const uint32_t sB = e4m3_pair(ksf[(gid + 8) * (D / 16) + grp], ksf[(gid + 8) * (D / 16) + grp]);
          uint32_t h0, h1, h2, h3;
          fp4x8_to_f16x8(*reinterpret_cast<const uint32_t*>(sl + unit_off(gid, j) + 4 * tig), h0, h1, h2, h3);
          kr0[j] = make_uint4(hmul2(h0, sA), hmul2(h1, sA), hmul2(h2, sA), hmul2(h3, sA));
          fp4x8_to_f16x8(*reinterpret_cast<const uint32_t*>(sl + unit_off(gid + 8, j) + 4 * tig), h0, h1, h2, h3);
          kr1[j] = make_uint4(hmul2(h0, sB), hmul2(h1, sB), hmul2(h2, sB), hmul2(h3, sB));
        }
      } else {
#pragma unroll
        for (int j = 0; j < KC; ++j) {  // 8 bytes of rows gid and gid + 8 at byte 32j + 8tig
          const int c = 2 * j + (tig >> 1), h = 8 * (tig & 1);
          kr0[j] = fp8x8_to_f16x8(*reinterpret_cast<const uint2*>(sl + unit_off(gid, c) + h));
          kr1[j] = fp8x8_to_f16x8(*reinterpret_cast<const uint2*>(sl + unit_off(gid + 8, c) + h));
        }
      }
      uint32_t va[Attn::KS][4];
      if constexpr (FP4) {
        // V: the lane's D/8 channels (d = (D/8) * gid ...) of keys 2tig, 2tig+1, 2tig+8,
        // 2tig+9 as D/64 words of 8 codes per key, inside one group of 16 channels
        constexpr int VW4 = D / 64;
        const uint8_t* vsf = sl + 2 * CB + SFB;
        const int grp = (D / 8) * gid / 16;
        uint32_t vw[4][VW4], vsc[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int vrow = 2 * tig + (e & 1) + 8 * (e >> 1);
          const bool live = key0 + vrow < t && vs != 0.f;  // rows past t: never read their values
          const int b = (D / 16) * gid;  // byte of the row
          const uint8_t* src = sl + CB + unit_off(vrow, b >> 4) + (b & 15);
          if constexpr (VW4 == 2) {
            const uint2 w = *reinterpret_cast<const uint2*>(src);
            vw[e][0] = live ? w.x : 0u, vw[e][1] = live ? w.y : 0u;
          } else {
            const uint32_t w = *reinterpret_cast<const uint32_t*>(src);
            vw[e][0] = live ? w : 0u;
          }
          vsc[e] = live ? vsf[vrow * (D / 16) + grp] : 0u;
        }
        // interleave two keys' codes: byte i of LO = (key e0, key e1) codes of channel 2i,
        // of HI the same of channel 2i+1; each byte converts to the (e0, e1) f16 pair
        const uint32_t s01 = e4m3_pair(vsc[0], vsc[1]), s23 = e4m3_pair(vsc[2], vsc[3]);
#pragma unroll
        for (int r = 0; r < VW4; ++r) {
          const uint32_t lo01 = (vw[0][r] & 0x0F0F0F0Fu) | ((vw[1][r] & 0x0F0F0F0Fu) << 4);
          const uint32_t hi01 = ((vw[0][r] >> 4) & 0x0F0F0F0Fu) | (vw[1][r] & 0xF0F0F0F0u);
          const uint32_t lo23 = (vw[2][r] & 0x0F0F0F0Fu) | ((vw[3][r] & 0x0F0F0F0Fu) << 4);
          const uint32_t hi23 = ((vw[2][r] >> 4) & 0x0F0F0F0Fu) | (vw[3][r] & 0xF0F0F0F0u);
          uint32_t a0[4], a1[4], a2[4], a3[4];
          fp4x8_to_f16x8(lo01, a0[0], a0[1], a0[2], a0[3]);
          fp4x8_to_f16x8(hi01, a1[0], a1[1], a1[2], a1[3]);
          fp4x8_to_f16x8(lo23, a2[0], a2[1], a2[2], a2[3]);
          fp4x8_to_f16x8(hi23, a3[0], a3[1], a3[2], a3[3]);
#pragma unroll
          for (int i = 0; i < 4; ++i) {  // m-tile 4r + i: channels 8r + 2i, 8r + 2i + 1 of the lane
            va[4 * r + i][0] = hmul2(a0[i], s01);
            va[4 * r + i][1] = hmul2(a1[i], s01);
            va[4 * r + i][2] = hmul2(a2[i], s23);
            va[4 * r + i][3] = hmul2(a3[i], s23);
          }
        }
      } else {
      // V: the lane's D/8 bytes (d = (D/8) * gid ...) of keys 2tig, 2tig+1, 2tig+8, 2tig+9,
      // as D/32 words per key; rows past t (and a zero V scale) read as zero
      constexpr int VW = D / 32;
      uint32_t vw[4][VW];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int vrow = 2 * tig + (e & 1) + 8 * (e >> 1);
        const bool live = key0 + vrow < t && vs != 0.f;
        const int b = (D / 8) * gid;
        const uint8_t* src = sl + CB + unit_off(vrow, b >> 4) + (b & 15);
        if constexpr (VW == 4) {
          const uint4 w = *reinterpret_cast<const uint4*>(src);
          vw[e][0] = live ? w.x : 0u, vw[e][1] = live ? w.y : 0u, vw[e][2] = live ? w.z : 0u, vw[e][3] = live ? w.w : 0u;
        } else {
          const uint2 w = *reinterpret_cast<const uint2*>(src);
          vw[e][0] = live ? w.x : 0u, vw[e][1] = live ? w.y : 0u;
        }
      }
      // V^T A-fragments straight from the bytes: interleave two keys' bytes, then each
      // byte pair converts to the (key, key + 1) f16 pair of one d
#pragma unroll
      for (int mt = 0; mt < Attn::KS; ++mt) {
        const int r = mt >> 1;
        const uint32_t sel = (mt & 1) ? 0x7362u : 0x5140u;
        fp8x4_to_f16x4(__byte_perm(vw[0][r], vw[1][r], sel), va[mt][0], va[mt][1]);
        fp8x4_to_f16x4(__byte_perm(vw[2][r], vw[3][r], sel), va[mt][2], va[mt][3]);
      }
      }
      const int keyA = key0 + gid, keyB = key0 + gid + 8;
      const bool okA = keyA < t, okB = keyB < t;
      float x[NT][4];
      at.step(kr0, kr1, va, okA, okB, a.scale_log2 * ks, x);
      write_logits(x, at.gmax, key0, okA, okB);
    };
    // issue cursor (pg, ch) over the warp's chunks: 4 per page, fewer on the last page of t
    int phys = 0;
    int pg = good_page(page0 + warp, phys), ch = 0;
    int issued = 0;
    auto issue_next = [&]() {
      if (pg < page1) {
        issue(pg, phys, ch, issued % kRing8);
        ++issued;
        if (ch + 1 < 4 && pg * kPage + (ch + 1) * 16 < t) {
          ++ch;
        } else {
          pg = good_page(pg + 4, phys);
          ch = 0;
        }
      }
      cp_async_commit();  // one group per call, empty or not, so the wait count below holds
    };
#pragma unroll
    for (int i = 0; i < kRing8 - 1; ++i) issue_next();
#pragma unroll 1
    for (int done = 0; done < issued; ++done) {
      issue_next();
      cp_async_wait<kRing8 - 1>();  // this lane's copies of chunk `done` have landed
      __syncwarp();                 // ... and every lane's
      compute(done % kRing8);
      __syncwarp();  // the slot is refilled by the next issue
    }
    __syncthreads();  // the merge buffers below alias the rings
    at.store(warp, sm_m, sm_l, sm_o, v_unit);
  }
  if constexpr (!FP8) at.store(warp, sm_m, sm_l, sm_o);
  __syncthreads();
  // ---- merge the 4 warps and write this split's partial
  for (int e = threadIdx.x; e < G * D; e += blockDim.x) {
    const int hl = e / D, dd = e % D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < 4; ++w) M = fmaxf(M, sm_m[w * NT * 8 + hl]);
    float L = 0.f, Ov = 0.f;
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      const float f = exp2_rel(sm_m[w * NT * 8 + hl], M);
      L += f * sm_l[w * NT * 8 + hl];
      Ov += f * sm_o[((size_t)w * NT * 8 + hl) * D + dd];
    }
    const size_t ph = ((size_t)qi * a.Hq + (size_t)g * G + hl) * a.nsplit + split;
    a.part_o[ph * D + dd] = Ov;
    if (dd == 0) a.part_ml[ph] = make_float2(M, L);
  }
}

// ============================================================================ launcher
template <int D, int NT>
static cudaError_t launch_mma(const AttnArgs& a, int Bq, cudaStream_t s) {
  dim3 grid(a.nsplit, a.Hkv, Bq);
  const size_t merge = (size_t)(64 * NT + 32 * NT * D) * sizeof(float);
  const int fmt = a.k_sf ? kFaFp4 : a.k_scale ? kFaFp8 : kFaBf16;
  const size_t ring = (size_t)4 * kRing8 * (fmt == kFaFp4 ? fa8_slot_bytes<D, kFaFp4>() : fa8_slot_bytes<D, kFaFp8>());
  const size_t sm = fmt != kFaBf16 ? std::max(merge, ring) : merge;
  auto kern = fmt == kFaFp4   ? fa_decode_mma_kernel<D, NT, kFaFp4>
              : fmt == kFaFp8 ? fa_decode_mma_kernel<D, NT, kFaFp8>
                              : fa_decode_mma_kernel<D, NT, kFaBf16>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
  if (e != cudaSuccess) return e;
  kern<<<grid, 128, sm, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_fa_decode_mma(const AttnArgs& a, int Bq, cudaStream_t s) {
  const int NTl = (a.G + 7) / 8;
  if (a.D == 128) {
    switch (NTl) {
      case 1: return launch_mma<128, 1>(a, Bq, s);
      case 2: return launch_mma<128, 2>(a, Bq, s);
      case 4: return launch_mma<128, 4>(a, Bq, s);
    }
  } else if (a.D == 64) {
    switch (NTl) {
      case 1: return launch_mma<64, 1>(a, Bq, s);
      case 2: return launch_mma<64, 2>(a, Bq, s);
      case 4: return launch_mma<64, 4>(a, Bq, s);
    }
  }
  return cudaErrorInvalidValue;
}

}  // namespace hs2

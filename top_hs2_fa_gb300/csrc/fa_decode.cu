// fa_decode.cu — bf16 split-KV scan of the FA layer (decode and causal rows).
//
// The FA layer of a HySparse2 Cross group attends to every visible key of the group's
// shared paged KV ("HySparse2：整体架构、KV 生命周期与 PD 分离", §5; §16.1: the FA layers
// still scan the whole history at decode). This kernel streams K and V pages straight
// from HBM into registers with 128-bit loads; the head-sharing contraction (the query
// heads of one KV head) runs on mma.sync with the keys as the M dimension, so no MMA
// row is padding. It writes per-split softmax partials and the base-2 logits that the
// selection (combine.cu) needs once the per-head normaliser is known.
#include "common.cuh"
#include "kernels.h"
#include "mma_attn.cuh"

namespace hs2 {

// ============================================================================ bf16 split-KV FA
// Per CTA: one (query, KV head, split of `pps` pages); 4 warps take the split's pages
// round-robin; per warp step: 16 keys (see mma_attn.cuh for the register mappings).
// FP8 = true: the cache holds E4M3 codes with one scale per (page, KV head); rows load at half
// the bytes and convert to f16 (exact), the page's K scale multiplies the logits and its V
// scale the weights entering P.V (mma_attn.cuh, F16 mode).
template <int D, int NT, bool FP8>
__global__ void __launch_bounds__(128) fa_decode_mma_kernel(const AttnArgs a) {
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
  float* logit_base = a.logits ? a.logits + ((size_t)qi * a.Hq + (size_t)g * G) * a.ld_logits : nullptr;

  for (int page = page0 + warp; page < page1; page += 4) {
    const int phys = bt[page];
    if (phys < 0 || phys >= a.num_pages) {
      if (lane == 0) flag_error(a.dev_err, HS2_DEV_BAD_PAGE);
      continue;
    }
    constexpr int EB = FP8 ? 1 : 2;  // bytes per element
    const uint8_t* kp = reinterpret_cast<const uint8_t*>(a.k) + ((size_t)phys * a.Hkv + g) * head_stride * EB;
    const uint8_t* vp = reinterpret_cast<const uint8_t*>(a.v) + ((size_t)phys * a.Hkv + g) * head_stride * EB;
    // 8 consecutive elements of a row as 8 bf16 / f16 in a uint4
    auto ld8 = [&](const uint8_t* base, size_t el) -> uint4 {
      if (FP8) return fp8x8_to_f16x8(ldg_nc_v2(base + el));
      return ldg_nc_v4(base + 2 * el);
    };
    const float ks = FP8 ? a.k_scale[(size_t)phys * a.Hkv + g] : 1.f;
    const float vs = FP8 ? a.v_scale[(size_t)phys * a.Hkv + g] : 1.f;
#pragma unroll 1
    for (int ch = 0; ch < 4; ++ch) {
      const int key0 = page * kPage + ch * 16;
      if (key0 >= t) break;
      const int r0 = ch * 16 + gid;  // row within the page
      uint4 kr0[KC], kr1[KC], vr[4][VC];
#pragma unroll
      for (int j = 0; j < KC; ++j) {
        kr0[j] = ld8(kp, (size_t)r0 * D + 32 * j + 8 * tig);
        kr1[j] = ld8(kp, (size_t)(r0 + 8) * D + 32 * j + 8 * tig);
      }
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int vrow = ch * 16 + 2 * tig + (e & 1) + 8 * (e >> 1);
#pragma unroll
        for (int j = 0; j < VC; ++j) vr[e][j] = ld8(vp, (size_t)vrow * D + (D / 8) * gid + 8 * j);
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
      at.step(kr0, kr1, vr, okA, okB, a.scale_log2 * ks, x, vs);
      if (logit_base) {  // base-2 logits for the selection
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          const int h0 = nt * 8 + 2 * tig;
          if (h0 < G) {
            if (okA) logit_base[(size_t)h0 * a.ld_logits + keyA] = x[nt][0];
            if (okB) logit_base[(size_t)h0 * a.ld_logits + keyB] = x[nt][2];
          }
          if (h0 + 1 < G) {
            if (okA) logit_base[(size_t)(h0 + 1) * a.ld_logits + keyA] = x[nt][1];
            if (okB) logit_base[(size_t)(h0 + 1) * a.ld_logits + keyB] = x[nt][3];
          }
        }
      }
    }
  }
  at.store(warp, sm_m, sm_l, sm_o);
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
  const size_t sm = (size_t)(64 * NT + 32 * NT * D) * sizeof(float);
  auto kern = a.k_scale ? fa_decode_mma_kernel<D, NT, true> : fa_decode_mma_kernel<D, NT, false>;
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

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

namespace hs2 {

// ============================================================================ bf16 split-KV FA
// Per CTA: one (query, KV head, split of `pps` pages); 4 warps take the split's pages
// round-robin; per warp step: 16 keys.
//
// Register mappings (m16n8k16, groupID = lane/4, tig = lane%4):
//  S^T[16 keys x 8 heads] = K[16 keys x 16 d] * Q^T[16 d x 8 heads]
//    K rows lane/4 and lane/4+8 are loaded as D/32 chunks of 8 bf16 at
//    d = 32j + 8*tig; k-step s = 2j+u uses words 2u (a0/a1) and 2u+1 (a2/a3), i.e.
//    the contraction index is permuted identically for K and Q (sum is unchanged).
//  O^T[16 d x 8 heads] += V^T[16 d x 16 keys] * P^T[16 keys x 8 heads]
//    thread loads keys {2tig, 2tig+1, 2tig+8, 2tig+9} at d in
//    [(D/8)*groupID, (D/8)*(groupID+1)); m-tile mt row hi <-> d = (D/8)*groupID + 2mt + hi.
//    P^T fragments come from the S^T accumulators by an 8x8 movmatrix transpose.
template <int D, int NT>
__global__ void __launch_bounds__(128) fa_decode_mma_kernel(const AttnArgs a) {
  constexpr int KS = D / 16;  // k-steps of QK^T and m-tiles of PV
  constexpr int KC = D / 32;  // 16-byte chunks per K row per thread
  constexpr int VC = D / 64;  // 16-byte chunks per V row per thread
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

  // ---- Q^T B-fragments (bf16): head nt*8+gid, contraction slots per k-step
  uint32_t qb[KS][NT][2];
  const __nv_bfloat16* q = reinterpret_cast<const __nv_bfloat16*>(a.q);
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const int hl = nt * 8 + gid;
    const bool hv = hl < G;
    const uint32_t* qrow =
        reinterpret_cast<const uint32_t*>(q + ((size_t)qi * a.Hq + (size_t)g * G + (hv ? hl : 0)) * D);
#pragma unroll
    for (int s = 0; s < KS; ++s) {
      const int base = 32 * (s >> 1) + 8 * tig + 4 * (s & 1);
      qb[s][nt][0] = hv ? qrow[base / 2] : 0u;
      qb[s][nt][1] = hv ? qrow[base / 2 + 1] : 0u;
    }
  }

  float m_run[NT][2], l_run[NT][2];
  float acc[KS][NT][4];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    m_run[nt][0] = m_run[nt][1] = -INFINITY;
    l_run[nt][0] = l_run[nt][1] = 0.f;
#pragma unroll
    for (int mt = 0; mt < KS; ++mt) acc[mt][nt][0] = acc[mt][nt][1] = acc[mt][nt][2] = acc[mt][nt][3] = 0.f;
  }

  const int32_t* bt = a.bt + (size_t)qg.b * a.max_pages;
  const size_t head_stride = (size_t)kPage * D;  // elements per (page, KV head)
  float* logit_base = a.logits ? a.logits + ((size_t)qi * a.Hq + (size_t)g * G) * a.ld_logits : nullptr;

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
      uint4 kr0[KC], kr1[KC], vr[4][VC];
#pragma unroll
      for (int j = 0; j < KC; ++j) {
        kr0[j] = ldg_nc_v4(kp + (size_t)r0 * D + 32 * j + 8 * tig);
        kr1[j] = ldg_nc_v4(kp + (size_t)(r0 + 8) * D + 32 * j + 8 * tig);
      }
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int vrow = ch * 16 + 2 * tig + (e & 1) + 8 * (e >> 1);
#pragma unroll
        for (int j = 0; j < VC; ++j) vr[e][j] = ldg_nc_v4(vp + (size_t)vrow * D + (D / 8) * gid + 8 * j);
      }
      const bool tail = key0 + 16 > t;
      if (tail) {  // rows past t: never read their values
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int key = key0 + 2 * tig + (e & 1) + 8 * (e >> 1);
          if (key >= t)
#pragma unroll
            for (int j = 0; j < VC; ++j) vr[e][j] = make_uint4(0, 0, 0, 0);
        }
      }
      // ---- S^T = K Q^T
      float sc[NT][4];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = 0.f;
#pragma unroll
        for (int s = 0; s < KS; ++s) {
          const int j = s >> 1, u = s & 1;
          const uint32_t a0 = u ? kr0[j].z : kr0[j].x;
          const uint32_t a2 = u ? kr0[j].w : kr0[j].y;
          const uint32_t a1 = u ? kr1[j].z : kr1[j].x;
          const uint32_t a3 = u ? kr1[j].w : kr1[j].y;
          mma_bf16_16816(sc[nt], a0, a1, a2, a3, qb[s][nt][0], qb[s][nt][1]);
        }
      }
      const int keyA = key0 + gid, keyB = key0 + gid + 8;
      const bool okA = keyA < t, okB = keyB < t;
      // ---- online softmax (base 2), logits to scratch
      uint32_t pb[NT][2];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        float x[4];
        x[0] = okA ? sc[nt][0] * a.scale_log2 : -INFINITY;
        x[1] = okA ? sc[nt][1] * a.scale_log2 : -INFINITY;
        x[2] = okB ? sc[nt][2] * a.scale_log2 : -INFINITY;
        x[3] = okB ? sc[nt][3] * a.scale_log2 : -INFINITY;
        if (logit_base) {
          const int h0 = nt * 8 + 2 * tig;
          if (h0 < G) {
            if (okA) logit_base[(size_t)h0 * a.ld_logits + keyA] = x[0];
            if (okB) logit_base[(size_t)h0 * a.ld_logits + keyB] = x[2];
          }
          if (h0 + 1 < G) {
            if (okA) logit_base[(size_t)(h0 + 1) * a.ld_logits + keyA] = x[1];
            if (okB) logit_base[(size_t)(h0 + 1) * a.ld_logits + keyB] = x[3];
          }
        }
        float p[4];
#pragma unroll
        for (int hs = 0; hs < 2; ++hs) {
          float cm = fmaxf(x[hs], x[hs + 2]);
          cm = fmaxf(cm, __shfl_xor_sync(0xffffffffu, cm, 4));
          cm = fmaxf(cm, __shfl_xor_sync(0xffffffffu, cm, 8));
          cm = fmaxf(cm, __shfl_xor_sync(0xffffffffu, cm, 16));
          const float mn = fmaxf(m_run[nt][hs], cm);
          const float alpha = (mn == -INFINITY) ? 1.f : exp2f(m_run[nt][hs] - mn);
          m_run[nt][hs] = mn;
          p[hs] = exp2_rel(x[hs], mn);
          p[hs + 2] = exp2_rel(x[hs + 2], mn);
          l_run[nt][hs] *= alpha;
#pragma unroll
          for (int mt = 0; mt < KS; ++mt) {
            acc[mt][nt][hs] *= alpha;
            acc[mt][nt][hs + 2] *= alpha;
          }
        }
        const uint32_t pA = pack_bf16(p[0], p[1]);  // key gid,   heads 2tig, 2tig+1
        const uint32_t pB = pack_bf16(p[2], p[3]);  // key gid+8
        // normaliser from the same bf16-rounded weights that enter the PV product
        l_run[nt][0] += bf16_lo(pA) + bf16_lo(pB);
        l_run[nt][1] += bf16_hi(pA) + bf16_hi(pB);
        pb[nt][0] = movmatrix_trans(pA);
        pb[nt][1] = movmatrix_trans(pB);
      }
      // ---- O^T += V^T P^T
#pragma unroll
      for (int mt = 0; mt < KS; ++mt) {
        const int j = mt >> 2, w4 = mt & 3;
        const uint32_t v0 = (&vr[0][j].x)[w4], v1 = (&vr[1][j].x)[w4];
        const uint32_t v2 = (&vr[2][j].x)[w4], v3 = (&vr[3][j].x)[w4];
        const uint32_t a0 = __byte_perm(v0, v1, 0x5410);
        const uint32_t a1 = __byte_perm(v0, v1, 0x7632);
        const uint32_t a2 = __byte_perm(v2, v3, 0x5410);
        const uint32_t a3 = __byte_perm(v2, v3, 0x7632);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) mma_bf16_16816(acc[mt][nt], a0, a1, a2, a3, pb[nt][0], pb[nt][1]);
      }
    }
  }

  // ---- warp partials -> shared memory
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
    for (int hs = 0; hs < 2; ++hs) {
      float l = l_run[nt][hs];
      l += __shfl_xor_sync(0xffffffffu, l, 4);
      l += __shfl_xor_sync(0xffffffffu, l, 8);
      l += __shfl_xor_sync(0xffffffffu, l, 16);
      const int hl = nt * 8 + 2 * tig + hs;
      if (gid == 0) {
        sm_m[warp * NT * 8 + hl] = m_run[nt][hs];
        sm_l[warp * NT * 8 + hl] = l;
      }
#pragma unroll
      for (int mt = 0; mt < KS; ++mt) {
        const int d0 = (D / 8) * gid + 2 * mt;
        sm_o[((size_t)warp * NT * 8 + hl) * D + d0] = acc[mt][nt][hs];
        sm_o[((size_t)warp * NT * 8 + hl) * D + d0 + 1] = acc[mt][nt][hs + 2];
      }
    }
  }
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
  auto kern = fa_decode_mma_kernel<D, NT>;
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

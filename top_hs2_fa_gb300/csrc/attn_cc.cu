// attn_cc.cu — CUDA-core attention partials over a list of rows of one group's paged KV.
//
// Used for fp32 inputs (FA scan over splits of pages, with logits for the selection) and
// for the SA gather when no faster path applies: rows are the window followed by the
// selected far positions, read in place through the block table, all under one softmax
// ("HySparse2：整体架构、KV 生命周期与 PD 分离", §7.2, §7.4).
#include "common.cuh"
#include "kernels.h"

namespace hs2 {

// ============================================================================ CUDA-core partial
// One CTA = one (query, KV head, chunk). Rows of the chunk are either a contiguous range of
// pages (FA, a.gather == 0: split of pps pages) or a slice of U = W(t) ∪ S(t) (SA,
// a.gather == 1: rows [chunk*128, chunk*128+128) of the window-then-indices list).
// Thread r owns row r for the logits (q in shared memory); for PV, thread t owns
// d-pair t % (D/2) and a residue class of rows.
template <typename T, int D, int G>
__global__ void __launch_bounds__(128) attn_partial_kernel(const AttnArgs a) {
  constexpr int ROWS = 128;
  constexpr int DP = D / 2;          // d-pairs
  constexpr int RG = ROWS / DP;      // row groups in PV (2 for D=128, 4 for D=64)
  const int qi = blockIdx.z, g = blockIdx.y, chunk = blockIdx.x;
  const int tid = threadIdx.x;
  const QueryGeom qg = query_geom(qi, a.prefill, a.seq_len);
  const int t = qg.t;
  if (t < 1 || t > a.max_t || (t + kPage - 1) / kPage > a.max_pages) return;  // flagged by the combine

  int row_begin, row_end;  // rows of this CTA in its list
  int nW = 0;
  const int32_t* sel = nullptr;
  if (!a.gather) {
    row_begin = chunk * a.pps * kPage;
    row_end = min(t, row_begin + a.pps * kPage);
  } else {
    nW = min(a.w, t);
    const int nS = max(0, min(a.kcap, a.cnt[(size_t)qi * a.Hkv + g]));
    sel = a.idx + ((size_t)qi * a.Hkv + g) * a.kcap;
    row_begin = chunk * ROWS;
    row_end = min(nW + nS, row_begin + ROWS);
  }
  if (row_begin >= row_end) return;

  // dynamic shared memory: q_s[G][D] | o_red[G][D] | p_s[ROWS][G] | red_s[4][G] | m_s[G] |
  // alpha_s[G] | vrow_s[ROWS]
  extern __shared__ float smem[];
  float (*q_s)[D] = reinterpret_cast<float (*)[D]>(smem);
  float (*o_red)[D] = reinterpret_cast<float (*)[D]>(smem + G * D);
  float (*p_s)[G] = reinterpret_cast<float (*)[G]>(smem + 2 * G * D);
  float (*red_s)[G] = reinterpret_cast<float (*)[G]>(smem + 2 * G * D + ROWS * G);
  float* m_s = smem + 2 * G * D + ROWS * G + 4 * G;
  float* alpha_s = m_s + G;
  const T** vrow_s = reinterpret_cast<const T**>(alpha_s + G);

  const T* q = reinterpret_cast<const T*>(a.q) + ((size_t)qi * a.Hq + (size_t)g * G) * D;
  for (int e = tid; e < G * D; e += ROWS) {
    q_s[e / D][e % D] = Elem<T>::to_f(q[e]);
    o_red[e / D][e % D] = 0.f;
  }
  float l_part[G];
#pragma unroll
  for (int h = 0; h < G; ++h) l_part[h] = 0.f;
  float oacc[G][2];
#pragma unroll
  for (int h = 0; h < G; ++h) oacc[h][0] = oacc[h][1] = 0.f;
  const int dp = tid % DP, rg = tid / DP;
  const int32_t* bt = a.bt + (size_t)qg.b * a.max_pages;
  // selection logits (FA layer, consecutive positions over consecutive threads): codes below
  // each 16-position group's per-head max, and the max (logit_code)
  const size_t lrow = (size_t)qi * a.Hq + (size_t)g * G;
  uint16_t* code_base = a.lcode ? a.lcode + lrow * a.ld_logits : nullptr;
  float* max_base = a.lcode ? a.lmax + lrow * (a.ld_logits / kLogitGroup) : nullptr;
  __syncthreads();

  for (int r0 = row_begin; r0 < row_end; r0 += ROWS) {
    const int r = r0 + tid;
    bool ok = r < row_end;
    int pos = 0;
    if (ok) {
      if (!a.gather) {
        pos = r;
      } else if (r < nW) {
        pos = t - nW + r;
      } else {
        pos = sel[r - nW];
        const int lim = a.w > 0 ? t - a.w : t;
        if (pos < 0 || pos >= lim) {
          flag_error(a.dev_err, HS2_DEV_BAD_INDEX);
          ok = false;
        }
      }
    }
    const T* krow = nullptr;
    const T* vrow = nullptr;
    if (ok) {
      const int phys = bt[pos / kPage];
      if (phys < 0 || phys >= a.num_pages) {
        flag_error(a.dev_err, HS2_DEV_BAD_PAGE);
        ok = false;
      } else {
        const size_t off = (((size_t)phys * a.Hkv + g) * kPage + pos % kPage) * D;
        krow = reinterpret_cast<const T*>(a.k) + off;
        vrow = reinterpret_cast<const T*>(a.v) + off;
      }
    }
    float x[G];
#pragma unroll
    for (int h = 0; h < G; ++h) x[h] = 0.f;
    if (ok) {
#pragma unroll 4
      for (int d0 = 0; d0 < D; d0 += 8) {
        float kv[8];
        if constexpr (sizeof(T) == 2) {
          const uint4 u = *reinterpret_cast<const uint4*>(krow + d0);
          kv[0] = bf16_lo(u.x); kv[1] = bf16_hi(u.x); kv[2] = bf16_lo(u.y); kv[3] = bf16_hi(u.y);
          kv[4] = bf16_lo(u.z); kv[5] = bf16_hi(u.z); kv[6] = bf16_lo(u.w); kv[7] = bf16_hi(u.w);
        } else {
          const float4 u0 = *reinterpret_cast<const float4*>(krow + d0);
          const float4 u1 = *reinterpret_cast<const float4*>(krow + d0 + 4);
          kv[0] = u0.x; kv[1] = u0.y; kv[2] = u0.z; kv[3] = u0.w;
          kv[4] = u1.x; kv[5] = u1.y; kv[6] = u1.z; kv[7] = u1.w;
        }
#pragma unroll
        for (int h = 0; h < G; ++h) {
          const float4 qa = *reinterpret_cast<const float4*>(&q_s[h][d0]);
          const float4 qb = *reinterpret_cast<const float4*>(&q_s[h][d0 + 4]);
          x[h] = fmaf(kv[0], qa.x, x[h]); x[h] = fmaf(kv[1], qa.y, x[h]);
          x[h] = fmaf(kv[2], qa.z, x[h]); x[h] = fmaf(kv[3], qa.w, x[h]);
          x[h] = fmaf(kv[4], qb.x, x[h]); x[h] = fmaf(kv[5], qb.y, x[h]);
          x[h] = fmaf(kv[6], qb.z, x[h]); x[h] = fmaf(kv[7], qb.w, x[h]);
        }
      }
    }
#pragma unroll
    for (int h = 0; h < G; ++h) x[h] = ok ? x[h] * a.scale_log2 : -INFINITY;
    if (code_base) {  // the block's rows start on a multiple of 16 positions (whole pages)
#pragma unroll
      for (int h = 0; h < G; ++h) {
        float gm = x[h];
        gm = fmaxf(gm, __shfl_xor_sync(0xffffffffu, gm, 1));
        gm = fmaxf(gm, __shfl_xor_sync(0xffffffffu, gm, 2));
        gm = fmaxf(gm, __shfl_xor_sync(0xffffffffu, gm, 4));
        gm = fmaxf(gm, __shfl_xor_sync(0xffffffffu, gm, 8));
        if (ok) {
          code_base[(size_t)h * a.ld_logits + pos] = (uint16_t)logit_code(x[h], gm);
          if ((tid & (kLogitGroup - 1)) == 0) max_base[(size_t)h * (a.ld_logits / kLogitGroup) + pos / kLogitGroup] = gm;
        }
      }
    }
    vrow_s[tid] = ok ? vrow : nullptr;
    // chunk max per head (block reduction), running max update
#pragma unroll
    for (int h = 0; h < G; ++h) {
      const float wm = warp_max(x[h]);
      if ((tid & 31) == 0) red_s[tid >> 5][h] = wm;
    }
    __syncthreads();
    if (tid < G) {
      const float cm = fmaxf(fmaxf(red_s[0][tid], red_s[1][tid]), fmaxf(red_s[2][tid], red_s[3][tid]));
      const float mo = m_s[tid];
      const float mn = (r0 == row_begin) ? cm : fmaxf(mo, cm);
      alpha_s[tid] = (r0 == row_begin || mn == -INFINITY) ? (r0 == row_begin ? 0.f : 1.f) : exp2f(mo - mn);
      m_s[tid] = mn;
    }
    __syncthreads();
#pragma unroll
    for (int h = 0; h < G; ++h) {
      const float mn = m_s[h];
      const float p = exp2_rel(x[h], mn);
      p_s[tid][h] = p;
      l_part[h] = l_part[h] * alpha_s[h] + p;
      oacc[h][0] *= alpha_s[h];
      oacc[h][1] *= alpha_s[h];
    }
    __syncthreads();
    // PV: thread (dp, rg) sums rows rg, rg+RG, ...
    const int nrows = min(ROWS, row_end - r0);
    for (int rr = rg; rr < nrows; rr += RG) {
      const T* vr = vrow_s[rr];
      if (!vr) continue;
      float v0, v1;
      if constexpr (sizeof(T) == 2) {
        const uint32_t u = *reinterpret_cast<const uint32_t*>(vr + 2 * dp);
        v0 = bf16_lo(u);
        v1 = bf16_hi(u);
      } else {
        const float2 u = *reinterpret_cast<const float2*>(vr + 2 * dp);
        v0 = u.x;
        v1 = u.y;
      }
#pragma unroll
      for (int h = 0; h < G; ++h) {
        const float p = p_s[rr][h];
        oacc[h][0] = fmaf(p, v0, oacc[h][0]);
        oacc[h][1] = fmaf(p, v1, oacc[h][1]);
      }
    }
    __syncthreads();
  }
  // l: block sum per head; o: reduce row groups
#pragma unroll
  for (int h = 0; h < G; ++h) {
    const float ws = warp_sum(l_part[h]);
    if ((tid & 31) == 0) red_s[tid >> 5][h] = ws;
  }
#pragma unroll
  for (int h = 0; h < G; ++h) {
    atomicAdd(&o_red[h][2 * dp], oacc[h][0]);
    atomicAdd(&o_red[h][2 * dp + 1], oacc[h][1]);
  }
  __syncthreads();
  for (int e = tid; e < G * D; e += ROWS) {
    const int h = e / D, dd = e % D;
    const float s = o_red[h][dd];
    const size_t ph = ((size_t)qi * a.Hq + (size_t)g * G + h) * a.nsplit + chunk;
    a.part_o[ph * D + dd] = s;
    if (dd == 0) {
      const float L = red_s[0][h] + red_s[1][h] + red_s[2][h] + red_s[3][h];
      a.part_ml[ph] = make_float2(m_s[h], L);
    }
  }
}

// ============================================================================ launcher
template <typename T, int D, int G>
static cudaError_t launch_cc3(const AttnArgs& a, int Bq, cudaStream_t s) {
  dim3 grid(a.nsplit, a.Hkv, Bq);
  const size_t sm = (size_t)(2 * G * D + 128 * G + 6 * G) * sizeof(float) + 128 * sizeof(void*);
  auto kern = attn_partial_kernel<T, D, G>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
  if (e != cudaSuccess) return e;
  kern<<<grid, 128, sm, s>>>(a);
  return cudaGetLastError();
}

template <typename T, int D>
static cudaError_t launch_cc2(const AttnArgs& a, int Bq, cudaStream_t s) {
  switch (a.G) {
    case 1: return launch_cc3<T, D, 1>(a, Bq, s);
    case 2: return launch_cc3<T, D, 2>(a, Bq, s);
    case 4: return launch_cc3<T, D, 4>(a, Bq, s);
    case 8: return launch_cc3<T, D, 8>(a, Bq, s);
    case 16: return launch_cc3<T, D, 16>(a, Bq, s);
    case 32: return launch_cc3<T, D, 32>(a, Bq, s);
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_attn_partial(const AttnArgs& a, int Bq, int bf16, cudaStream_t s) {
  if (bf16) {
    if (a.D == 128) return launch_cc2<__nv_bfloat16, 128>(a, Bq, s);
    if (a.D == 64) return launch_cc2<__nv_bfloat16, 64>(a, Bq, s);
  } else {
    if (a.D == 128) return launch_cc2<float, 128>(a, Bq, s);
    if (a.D == 64) return launch_cc2<float, 64>(a, Bq, s);
  }
  return cudaErrorInvalidValue;
}

}  // namespace hs2

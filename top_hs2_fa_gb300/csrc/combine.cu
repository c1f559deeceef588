// combine.cu — merge of split softmax partials, plus the window-excluding top-k.
//
// The selection score of a far position is the FA's own attention probability summed
// over the query heads of a KV head ("HySparse2：整体架构、KV 生命周期与 PD 分离", §5 and
// the appendix on the FA's "oracle" scores); ranking uses the final per-head normaliser,
// so it runs after the merge, from the base-2 logits the scan wrote. Ties go to the lower
// position; the result is sorted ascending (§7.2: the window is excluded from the budget).
#include "common.cuh"
#include "kernels.h"
#include "topk.cuh"

namespace hs2 {

// ============================================================================ combine (+ select)
// One CTA per (query, KV head). Merges the partials of the query's chunks:
//   M = max m_c, L = sum l_c 2^(m_c - M), o = sum o_c 2^(m_c - M) / L, lse2 = M + log2 L.
// With a.select: score(s) = sum_h 2^(x_h(s) - lse2_h) for s in F(t) from the base-2 logits,
// stored as uint32 bit patterns in a.scores, then the block radix top-k.
template <int D>
__global__ void __launch_bounds__(kCombineThreads) combine_kernel(const CombineArgs a) {
  constexpr int NT = kCombineThreads;
  const int qi = blockIdx.x, g = blockIdx.y;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int G = a.G;
  const QueryGeom qg = query_geom(qi, a.prefill, a.seq_len);
  const int t = qg.t;
  __shared__ float lse2_s[32];
  __shared__ float M_s[32], Linv_s[32];
  __shared__ TopkSmem<NT> tk;
  const bool bad_len = (t < 1) || (t > a.max_t) || ((t + kPage - 1) / kPage > a.max_pages);
  if (bad_len) {
    if (tid == 0) flag_error(a.dev_err, HS2_DEV_BAD_LENGTH);
    for (int e = tid; e < G * D; e += NT) a.o[((size_t)qi * a.Hq + (size_t)g * G) * D + e] = 0.f;
    if (a.select) {
      for (int j = tid; j < a.kcap; j += NT) a.idx[((size_t)qi * a.Hkv + g) * a.kcap + j] = -1;
      if (tid == 0) a.cnt[(size_t)qi * a.Hkv + g] = 0;
    }
    return;
  }
  int nchunk;
  if (a.gather) {
    const int c0 = a.sa_cnt[(size_t)qi * a.Hkv + g];
    if (tid == 0 && (c0 < 0 || c0 > a.kcap)) flag_error(a.dev_err, HS2_DEV_BAD_INDEX);
    const int nS = max(0, min(a.kcap, c0));
    nchunk = (min(a.w, t) + nS + 127) / 128;
  } else {
    nchunk = ((t + kPage - 1) / kPage + a.pps - 1) / a.pps;
  }
  // per-head merge statistics (warp h handles head h)
  for (int h = warp; h < G; h += NT / 32) {
    const size_t ph = ((size_t)qi * a.Hq + (size_t)g * G + h) * a.nsplit;
    float M = -INFINITY;
    for (int c = lane; c < nchunk; c += 32) M = fmaxf(M, a.part_ml[ph + c].x);
    M = warp_max(M);
    float L = 0.f;
    for (int c = lane; c < nchunk; c += 32) {
      const float2 ml = a.part_ml[ph + c];
      L += exp2_rel(ml.x, M) * ml.y;
    }
    L = warp_sum(L);
    if (lane == 0) {
      M_s[h] = M;
      Linv_s[h] = L > 0.f ? 1.f / L : 0.f;
      lse2_s[h] = M + log2f(L);
      if (a.lse) a.lse[(size_t)qi * a.Hq + (size_t)g * G + h] = (M + log2f(L)) / kLog2e;
    }
  }
  __syncthreads();
  for (int e = tid; e < G * D; e += NT) {
    const int h = e / D, dd = e % D;
    const size_t ph = ((size_t)qi * a.Hq + (size_t)g * G + h) * a.nsplit;
    const float M = M_s[h];
    float acc = 0.f;
    for (int c = 0; c < nchunk; ++c) acc += exp2_rel(a.part_ml[ph + c].x, M) * a.part_o[(ph + c) * D + dd];
    a.o[((size_t)qi * a.Hq + (size_t)g * G + h) * D + dd] = acc * Linv_s[h];
  }
  if (!a.select) return;

  // ---- selection over the far range F(t) = [0, t-w)
  const int nF = max(0, t - a.w);
  const int kk = min(a.k, nF);
  int32_t* out = a.idx + ((size_t)qi * a.Hkv + g) * a.kcap;
  if (tid == 0) a.cnt[(size_t)qi * a.Hkv + g] = kk;
  for (int j = kk + tid; j < a.kcap; j += NT) out[j] = -1;
  if (kk == 0) return;
  if (kk == nF) {  // the budget covers the whole far range
    for (int j = tid; j < nF; j += NT) out[j] = j;
    return;
  }
  uint32_t* keys = a.scores + ((size_t)qi * a.Hkv + g) * a.ld_logits;
  const float* lg = a.logits + ((size_t)qi * a.Hq + (size_t)g * G) * a.ld_logits;
  for (int s = tid; s < nF; s += NT) {
    float sc = 0.f;
    for (int h = 0; h < G; ++h) sc += exp2f(lg[(size_t)h * a.ld_logits + s] - lse2_s[h]);
    keys[s] = __float_as_uint(sc);
  }
  __syncthreads();
  block_topk<NT>(
      nF, kk, [&](int i) { return keys[i]; }, [&](int j, int i) { out[j] = i; }, tk);
}

// ============================================================================ launcher
cudaError_t launch_combine(const CombineArgs& a, int Bq, cudaStream_t s) {
  dim3 grid(Bq, a.Hkv);
  if (a.D == 128) combine_kernel<128><<<grid, kCombineThreads, 0, s>>>(a);
  else if (a.D == 64) combine_kernel<64><<<grid, kCombineThreads, 0, s>>>(a);
  else return cudaErrorInvalidValue;
  return cudaGetLastError();
}

}  // namespace hs2

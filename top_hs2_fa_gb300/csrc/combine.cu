// combine.cu — merge of split softmax partials, and the window-excluding top-k.
//
// The selection score of a far position is the FA's own attention probability summed
// over the query heads of a KV head ("HySparse2：整体架构、KV 生命周期与 PD 分离", §5 and
// the appendix on the FA's "oracle" scores). Ranking needs the final per-head
// normaliser, so it runs after the scan, from the base-2 logits the scan wrote. Ties go
// to the lower position; the result is sorted ascending; the window is excluded from
// the candidates (§7.2).
//
// merge_score_kernel  grid (score chunks, Hkv, queries), 256 threads. Every CTA derives
//                     lse from the (m, l) partials; chunk 0 also writes o and lse. With
//                     selection on, each CTA scores 2048 far positions (8 per thread,
//                     128-bit logit loads), writes them as uint32 keys and adds the
//                     histogram of their top 12 bits into a per-(query, KV head) global
//                     histogram (zeroed by the host call).
// select_kernel       one CTA (512 threads) per (query, KV head): from that histogram,
//                     the digit holding the k-th key; one coalesced pass over the keys
//                     splits them into "above the digit" (all taken) and "in the digit"
//                     (candidates) lists in shared memory; a radix select over the
//                     candidates alone fixes the k-th key and the ties to take; the two
//                     sorted lists are merged into the ascending output (topk.cuh).
// score_select_kernel decode with at least 152 (query, KV head) pairs: both of the above
//                     for one pair in one CTA (histogram in shared memory, no global one).
#include <cooperative_groups.h>

#include <algorithm>

#include "common.cuh"
#include "kernels.h"
#include "topk.cuh"

namespace cg = cooperative_groups;

namespace hs2 {

constexpr int kScoreChunk = 2048;
constexpr int kMergeThreads = 256;
constexpr int kSelectThreads = 512;

template <int D>
__global__ void __launch_bounds__(kMergeThreads) merge_score_kernel(const CombineArgs a) {
  constexpr int NT = kMergeThreads;
  const int chunk = blockIdx.x, g = blockIdx.y, qi = blockIdx.z;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int G = a.G;
  const QueryGeom qg = query_geom(qi, a.prefill, a.seq_len);
  const int t = qg.t;
  __shared__ float lse2_s[32], M_s[32], Linv_s[32];
  __shared__ uint32_t hist[kRadixBins];
  float* o_out = a.o + ((size_t)qi * a.Hq + (size_t)g * G) * D;
  int32_t* out = a.select ? a.idx + ((size_t)qi * a.Hkv + g) * a.kcap : nullptr;
  if ((t < 1) || (t > a.max_t) || ((t + kPage - 1) / kPage > a.max_pages)) {
    if (chunk == 0) {
      if (tid == 0) flag_error(a.dev_err, HS2_DEV_BAD_LENGTH);
      for (int e = tid; e < G * D; e += NT) o_out[e] = 0.f;
      if (a.select) {
        for (int j = tid; j < a.kcap; j += NT) out[j] = -1;
        if (tid == 0) a.cnt[(size_t)qi * a.Hkv + g] = 0;
      }
    }
    return;
  }
  const int nF = max(0, t - a.w);
  const int kk = min(a.k, nF);
  const bool scoring = a.select && kk > 0 && kk < nF;
  const int s_lo = chunk * kScoreChunk;
  if (chunk > 0 && (!scoring || s_lo >= nF)) return;

  int nchunk;
  if (a.gather) {
    const int c0 = a.sa_cnt[(size_t)qi * a.Hkv + g];
    if (tid == 0 && chunk == 0 && (c0 < 0 || c0 > a.kcap)) flag_error(a.dev_err, HS2_DEV_BAD_INDEX);
    nchunk = (min(a.w, t) + max(0, min(a.kcap, c0)) + 127) / 128;
  } else {
    nchunk = ((t + kPage - 1) / kPage + a.pps - 1) / a.pps;
  }
  // ---- per-head merge statistics (warp w handles heads w, w+8, ...)
  for (int h = warp; h < G; h += NT / 32) {
    const float2* ml = a.part_ml + ((size_t)qi * a.Hq + (size_t)g * G + h) * a.nsplit;
    float M = -INFINITY;
    for (int c = lane; c < nchunk; c += 32) M = fmaxf(M, ml[c].x);
    M = warp_max(M);
    float L = 0.f;
    for (int c = lane; c < nchunk; c += 32) L += exp2_rel(ml[c].x, M) * ml[c].y;
    L = warp_sum(L);
    if (lane == 0) {
      M_s[h] = M;
      Linv_s[h] = sa_norm_factor(M, L, sink_b2(a.sink, g * G + h));  // SA sink bias, if any
      lse2_s[h] = M + log2f(L);
    }
  }
  __syncthreads();
  if (chunk == 0) {
    if (a.lse && tid < G) a.lse[(size_t)qi * a.Hq + (size_t)g * G + tid] = lse2_s[tid] / kLog2e;
    // o = sum_c 2^(m_c - M) o_c / L; thread -> 4 consecutive outputs of one head
    for (int e4 = tid; e4 < G * D / 4; e4 += NT) {
      const int h = (4 * e4) / D, d0 = (4 * e4) % D;
      const size_t ph = ((size_t)qi * a.Hq + (size_t)g * G + h) * a.nsplit;
      const float M = M_s[h];
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
      for (int c = 0; c < nchunk; ++c) {
        const float wgt = exp2_rel(a.part_ml[ph + c].x, M);
        const float4 v = *reinterpret_cast<const float4*>(a.part_o + (ph + c) * D + d0);
        acc.x = fmaf(wgt, v.x, acc.x);
        acc.y = fmaf(wgt, v.y, acc.y);
        acc.z = fmaf(wgt, v.z, acc.z);
        acc.w = fmaf(wgt, v.w, acc.w);
      }
      const float li = Linv_s[h];
      float4 r4 = make_float4(acc.x * li, acc.y * li, acc.z * li, acc.w * li);
      if (a.gate) {  // SA output gate
        const float4 g4 = __ldg(reinterpret_cast<const float4*>(a.gate + ((size_t)qi * a.Hq + (size_t)g * G + h) * D + d0));
        r4.x *= sa_gate(g4.x);
        r4.y *= sa_gate(g4.y);
        r4.z *= sa_gate(g4.z);
        r4.w *= sa_gate(g4.w);
      }
      *reinterpret_cast<float4*>(o_out + (size_t)h * D + d0) = r4;
    }
    if (a.select) {
      for (int j = kk + tid; j < a.kcap; j += NT) out[j] = -1;
      if (tid == 0) a.cnt[(size_t)qi * a.Hkv + g] = kk;
      if (kk == nF)  // the budget covers the whole far range
        for (int j = tid; j < nF; j += NT) out[j] = j;
    }
  }
  if (!scoring || s_lo >= nF) return;

  // ---- score 2048 far positions, 8 per thread
  for (int i = tid; i < kRadixBins; i += NT) hist[i] = 0;
  __syncthreads();
  const int s0 = s_lo + 8 * tid;
  float sc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  if (s0 < nF) {
    // 8 positions of one 16-position group: 8 codes and the group's max per head
    const size_t lrow = (size_t)qi * a.Hq + (size_t)g * G;
    const uint16_t* lc = a.lcode + lrow * a.ld_logits + s0;
    const float* lm = a.lmax + lrow * (a.ld_logits / kLogitGroup) + s0 / kLogitGroup;
    for (int h = 0; h < G; ++h) {
      const uint4 c = __ldcs(reinterpret_cast<const uint4*>(lc + (size_t)h * a.ld_logits));
      const float d = __ldg(lm + (size_t)h * (a.ld_logits / kLogitGroup)) - lse2_s[h];
      sc[0] += logit_term(c.x & 0xffffu, d); sc[1] += logit_term(c.x >> 16, d);
      sc[2] += logit_term(c.y & 0xffffu, d); sc[3] += logit_term(c.y >> 16, d);
      sc[4] += logit_term(c.z & 0xffffu, d); sc[5] += logit_term(c.z >> 16, d);
      sc[6] += logit_term(c.w & 0xffffu, d); sc[7] += logit_term(c.w >> 16, d);
    }
  }
  uint32_t key[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) key[e] = (s0 + e < nF) ? __float_as_uint(sc[e]) : 0u;
  uint32_t* keys = a.scores + ((size_t)qi * a.Hkv + g) * a.ld_logits;
  if (s0 < nF) {
    *reinterpret_cast<uint4*>(keys + s0) = make_uint4(key[0], key[1], key[2], key[3]);
    *reinterpret_cast<uint4*>(keys + s0 + 4) = make_uint4(key[4], key[5], key[6], key[7]);
  }
#pragma unroll
  for (int e = 0; e < 8; ++e) hist_add(hist, s0 + e < nF, key[e] >> 20);
  __syncthreads();
  uint32_t* gh = a.hist + ((size_t)qi * a.Hkv + g) * kRadixBins;
  for (int i = tid; i < kRadixBins; i += NT) {
    const uint32_t c = hist[i];
    if (c) atomicAdd(&gh[i], c);
  }
}

// Shared memory of the selection kernels: A list (kcap), chosen-C list (kcap), C list.
constexpr int kFilterCap = 4096;
static size_t select_smem(int kcap) {
  return (size_t)2 * kcap * sizeof(int) + (size_t)kFilterCap * sizeof(uint2) + 2 * sizeof(int);
}

// The CTAs of one cluster share one row's selection (cluster_filter_topk; a cluster of one
// CTA takes filter_topk); the fallback passes over all keys run on rank 0 alone.
struct ClusterSel {
  int rank, n;
  HS2_DEVI ClusterSel() : rank((int)cg::this_cluster().block_rank()), n((int)cg::this_cluster().num_blocks()) {}
  HS2_DEVI void sync() const { cg::this_cluster().sync(); }
  template <typename T>
  HS2_DEVI T* remote(T* p, int r) const {
    return cg::this_cluster().map_shared_rank(p, r);
  }
};

// Launch `kern` on grid (gx * csize, gy) in clusters of csize CTAs along x.
template <typename Args>
static cudaError_t launch_clustered(void (*kern)(Args), int gx, int gy, size_t smem, int csize, cudaStream_t s,
                                    const Args& args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(gx * csize, gy);
  cfg.blockDim = dim3(kSelectThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = csize;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, args);
}

// CTAs per row selection: one per 8192 keys of the longest row, at most 8 (portable
// clusters), and only while the rows alone leave the GPU idle (a few long CSA2 rows); with
// hundreds of rows (decode) one CTA per row is faster (measured 26.6 vs 76.9 us at 4 CTAs).
static int sel_cluster_size(long long max_keys, long long rows) {
  int c = (int)std::min<long long>(8, std::max<long long>(1, (max_keys + 8191) / 8192));
  while (c > 1 && rows * c > 2 * 152) --c;
  return c;
}

// grid: clusters of CTAs along x (sel_cluster_size), one cluster per (query, KV head)
__global__ void __launch_bounds__(kSelectThreads, 2) select_kernel(const CombineArgs a) {
  constexpr int NT = kSelectThreads;
  const ClusterSel cl;
  const int g = blockIdx.x / cl.n, qi = blockIdx.y;
  const QueryGeom qg = query_geom(qi, a.prefill, a.seq_len);
  const int t = qg.t;
  if ((t < 1) || (t > a.max_t) || ((t + kPage - 1) / kPage > a.max_pages)) return;
  const int nF = max(0, t - a.w);
  const int kk = min(a.k, nF);
  if (kk == 0 || kk >= nF) return;  // written by merge_score_kernel
  __shared__ TopkSmem<NT> sm;
  extern __shared__ int fbuf[];
  int* la = fbuf;
  int* lsel = la + a.kcap;
  uint2* lc = reinterpret_cast<uint2*>(lsel + a.kcap);
  int* meta = reinterpret_cast<int*>(lc + kFilterCap);
  const uint32_t* gkeys = a.scores + ((size_t)qi * a.Hkv + g) * a.ld_logits;
  const uint32_t* gh = a.hist + ((size_t)qi * a.Hkv + g) * kRadixBins;
  int32_t* out = a.idx + ((size_t)qi * a.Hkv + g) * a.kcap;
  auto emit = [&](int j, int i) { out[j] = i; };
  if (cl.n == 1 ? filter_topk<NT, 16>(gkeys, nF, kk, gh, la, a.kcap, lc, kFilterCap, lsel, emit, sm)
                : cluster_filter_topk<NT, 16>(gkeys, nF, kk, gh, la, a.kcap, lc, kFilterCap, lsel, meta, cl.rank, cl.n,
                                              emit, [&] { cl.sync(); },
                                              [&](auto* p, int r) { return cl.remote(p, r); }, sm))
    return;
  // more candidates share the k-th key's top digit than the buffer holds: radix passes
  // over all keys, on rank 0
  if (cl.rank != 0) return;
  auto key = [&](int i) { return __ldcg(gkeys + i); };
  block_topk<NT>(nF, kk, key, emit, sm);
}

// Block-level selection (the first HySparse version: whole blocks of far positions): one
// CTA per (query, KV head); block maxima of the position keys, radix top-k over the blocks,
// then the chosen blocks' far positions in ascending order.
__global__ void __launch_bounds__(kSelectThreads) block_select_kernel(const CombineArgs a) {
  constexpr int NT = kSelectThreads;
  const int g = blockIdx.x, qi = blockIdx.y;
  const QueryGeom qg = query_geom(qi, a.prefill, a.seq_len);
  const int t = qg.t;
  if ((t < 1) || (t > a.max_t) || ((t + kPage - 1) / kPage > a.max_pages)) return;
  const int nF = max(0, t - a.w);
  const int kk = min(a.k, nF);
  if (kk == 0 || kk >= nF) return;  // written by merge_score_kernel (none, or all of F)
  const int blk = a.sel_block;
  const int nb = (nF + blk - 1) / blk, kb = min(a.k / blk, nb);
  __shared__ TopkSmem<NT> sm;
  extern __shared__ uint32_t bkey[];  // [nb] block maxima, then [kb] chosen blocks
  const uint32_t* keys = a.scores + ((size_t)qi * a.Hkv + g) * a.ld_logits;
  for (int b = threadIdx.x; b < nb; b += NT) bkey[b] = 0u;
  __syncthreads();
  // block maxima: 4-key chunks (blk is a multiple of 4, so a chunk lies in one block)
  const int nch = (nF + 3) / 4;  // the key row is readable up to nF rounded up to 4
#pragma unroll 4
  for (int c = threadIdx.x; c < nch; c += NT) {
    const uint4 v = __ldcg(reinterpret_cast<const uint4*>(keys) + c);
    const int s = 4 * c;
    uint32_t m = v.x;
    if (s + 1 < nF) m = max(m, v.y);
    if (s + 2 < nF) m = max(m, v.z);
    if (s + 3 < nF) m = max(m, v.w);
    atomicMax(&bkey[s / blk], m);
  }
  __syncthreads();
  uint32_t* chosen = bkey + nb;
  block_topk<NT>(nb, kb, [&](int i) { return bkey[i]; }, [&](int j, int i) { chosen[j] = (uint32_t)i; }, sm);
  __syncthreads();
  // every chosen block but the last far block is full, so block j's positions start at j*blk
  int32_t* out = a.idx + ((size_t)qi * a.Hkv + g) * a.kcap;
  for (int e = threadIdx.x; e < kb * blk; e += NT) {
    const int j = e / blk, r = e % blk;
    const int s = (int)chosen[j] * blk + r;
    out[e] = s < nF ? s : -1;
  }
  const int tail = (int)chosen[kb - 1] == nb - 1 ? nb * blk - nF : 0;  // missing positions of a partial last block
  for (int j = kb * blk + threadIdx.x; j < a.kcap; j += NT) out[j] = -1;
  if (threadIdx.x == 0) a.cnt[(size_t)qi * a.Hkv + g] = kb * blk - tail;
}

// ============================================================================ generic row top-k
// grid: clusters of CTAs along x (sel_cluster_size), one cluster per sequence; y = the job
// (the Full layer's position and block selections run as two jobs of one launch)
__global__ void __launch_bounds__(kSelectThreads, 2) select_rows_kernel(const SelectJobs jobs) {
  constexpr int NT = kSelectThreads;
  const SelectArgs& a = jobs.job[blockIdx.y];
  const ClusterSel cl;
  const int b = blockIdx.x / cl.n;
  const int tid = threadIdx.x;
  const int t = a.seq_len[b];
  int32_t* out = a.out + (size_t)b * a.kcap;
  const bool bad = t < 1 || t > a.max_t || (t + kPage - 1) / kPage > a.max_pages;
  int n = 0;
  const int32_t* pool = nullptr;
  if (!bad) {
    if (a.mode == 1) {
      n = t;
    } else if (a.mode == 2) {
      n = (t + 7) / 8;
    } else {
      pool = a.pool + (size_t)b * a.max_blocks;
      const int pc = max(0, min(a.max_blocks, a.pool_cnt[b]));
      if (pc > 0) n = (pc - 1) * 8 + max(0, min(8, t - 8 * pool[pc - 1]));
    }
  }
  const int kk = min(a.k, n);
  if (cl.rank == 0) {
    if (tid == 0) a.cnt[b] = kk;
    for (int j = kk + tid; j < a.kcap; j += NT) out[j] = -1;
  }
  auto map = [&](int i) { return a.mode == 3 ? pool[i >> 3] * 8 + (i & 7) : i; };
  if (kk == 0) return;
  if (kk == n) {
    if (cl.rank == 0)
      for (int i = tid; i < n; i += NT) out[i] = map(i);
    return;
  }
  __shared__ TopkSmem<NT> sm;
  extern __shared__ int fbuf[];
  int* la = fbuf;
  int* lsel = la + a.kcap;
  uint2* lc = reinterpret_cast<uint2*>(lsel + a.kcap);
  int* meta = reinterpret_cast<int*>(lc + kFilterCap);
  const uint32_t* gkeys = a.keys + (size_t)b * a.ld_keys;
  const uint32_t* gh = a.hist + (size_t)b * kRadixBins;
  auto emit = [&](int j, int i) { out[j] = map(i); };
  if (cl.n == 1 ? filter_topk<NT, 16>(gkeys, n, kk, gh, la, a.kcap, lc, kFilterCap, lsel, emit, sm)
                : cluster_filter_topk<NT, 16>(gkeys, n, kk, gh, la, a.kcap, lc, kFilterCap, lsel, meta, cl.rank, cl.n,
                                              emit, [&] { cl.sync(); },
                                              [&](auto* p, int r) { return cl.remote(p, r); }, sm))
    return;
  if (cl.rank != 0) return;
  auto key = [&](int i) { return __ldcg(gkeys + i); };
  block_topk<NT>(n, kk, key, emit, sm);
}

cudaError_t launch_select_rows(const SelectJobs& jobs, int B, cudaStream_t s) {
  if (jobs.n < 1 || jobs.n > kMaxSelectJobs) return cudaErrorInvalidValue;
  size_t sm = 0;
  long long n_max = 0;  // the longest row of any job sets the cluster size of all
  for (int j = 0; j < jobs.n; ++j) {
    const SelectArgs& a = jobs.job[j];
    sm = std::max(sm, select_smem(a.kcap));
    n_max = std::max(n_max, a.mode == 1 ? (long long)a.max_t : a.mode == 2 ? (a.max_t + 7) / 8 : 8LL * a.max_blocks);
  }
  cudaError_t e = cudaFuncSetAttribute(select_rows_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
  if (e != cudaSuccess) return e;
  return launch_clustered(select_rows_kernel, B, jobs.n, sm, sel_cluster_size(n_max, (long long)B * jobs.n), s, jobs);
}

// Prefill rows i whose far range F(i+1) = [0, i+1-w) fits the budget take all of it.
__global__ void prefill_trivial_select_kernel(int32_t* idx, int32_t* cnt, int n, int Hkv, int w, int k) {
  const int row = blockIdx.x;  // row * Hkv + g
  const int i = row / Hkv;
  if (i >= n) return;
  const int nF = max(0, i + 1 - w);
  const int kk = min(k, nF);
  if (threadIdx.x == 0) cnt[row] = kk;
  int32_t* out = idx + (size_t)row * k;
  for (int j = threadIdx.x; j < k; j += blockDim.x) out[j] = j < kk ? j : -1;
}

cudaError_t launch_prefill_trivial_select(int32_t* idx, int32_t* cnt, int n, int Hkv, int w, int k, cudaStream_t s) {
  prefill_trivial_select_kernel<<<n * Hkv, 128, 0, s>>>(idx, cnt, n, Hkv, w, k);
  return cudaGetLastError();
}

// Decode, token-level selection, many (query, KV head) pairs: the split merge, the scoring
// and the top-k of one (query, KV head) in one CTA (512 threads; every pair's CTA resident
// at once). The CTA derives lse from the split partials, merges o, then streams the far
// range's base-2 logits of its heads (four positions of up to eight heads per thread in
// flight), writes the scores as keys into the L2-resident scratch row and bins their top 12
// bits in shared memory, and selects from that histogram and the keys it has just written
// (filter_topk; the radix passes over all keys when the candidates overflow). Against
// merge_score_kernel + select_kernel this drops the global histogram (and its zeroing),
// one launch and a re-read of the keys from a second kernel.
constexpr int kFusedMinPairs = 152;  // below this, too few CTAs to stream the logits fast
constexpr int kScoreHeads = 8;       // heads whose logit-code loads a thread has in flight

bool score_select_fused(const CombineArgs& a, int Bq) {
  return a.select && a.sel_block == 1 && !a.prefill && !a.gather && (long long)Bq * a.Hkv >= kFusedMinPairs &&
         (a.D == 64 || a.D == 128);
}

template <int D>
__global__ void __launch_bounds__(kSelectThreads, 2) score_select_kernel(const CombineArgs a) {
  constexpr int NT = kSelectThreads;
  const int g = blockIdx.x, qi = blockIdx.y;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int G = a.G;
  const QueryGeom qg = query_geom(qi, a.prefill, a.seq_len);
  const int t = qg.t;
  __shared__ TopkSmem<NT> sm;
  __shared__ float lse2_s[32], M_s[32], Linv_s[32];
  extern __shared__ int fbuf[];
  float* o_out = a.o + ((size_t)qi * a.Hq + (size_t)g * G) * D;
  int32_t* out = a.idx + ((size_t)qi * a.Hkv + g) * a.kcap;
  if ((t < 1) || (t > a.max_t) || ((t + kPage - 1) / kPage > a.max_pages)) {
    if (tid == 0) flag_error(a.dev_err, HS2_DEV_BAD_LENGTH);
    for (int e = tid; e < G * D; e += NT) o_out[e] = 0.f;
    for (int j = tid; j < a.kcap; j += NT) out[j] = -1;
    if (tid == 0) a.cnt[(size_t)qi * a.Hkv + g] = 0;
    return;
  }
  const int nF = max(0, t - a.w);
  const int kk = min(a.k, nF);
  const int nchunk = ((t + kPage - 1) / kPage + a.pps - 1) / a.pps;
  // ---- per-head merge statistics (warp w handles heads w, w + 16, ...)
  for (int h = warp; h < G; h += NT / 32) {
    const float2* ml = a.part_ml + ((size_t)qi * a.Hq + (size_t)g * G + h) * a.nsplit;
    float M = -INFINITY;
    for (int c = lane; c < nchunk; c += 32) M = fmaxf(M, ml[c].x);
    M = warp_max(M);
    float L = 0.f;
    for (int c = lane; c < nchunk; c += 32) L += exp2_rel(ml[c].x, M) * ml[c].y;
    L = warp_sum(L);
    if (lane == 0) {
      M_s[h] = M;
      Linv_s[h] = L > 0.f ? 1.f / L : 0.f;
      lse2_s[h] = M + log2f(L);
    }
  }
  for (int i = tid; i < kRadixBins; i += NT) sm.hist[i] = 0;
  __syncthreads();
  if (a.lse && tid < G) a.lse[(size_t)qi * a.Hq + (size_t)g * G + tid] = lse2_s[tid] / kLog2e;
  // o = sum_c 2^(m_c - M) o_c / L; thread -> 4 consecutive outputs of one head
  for (int e4 = tid; e4 < G * D / 4; e4 += NT) {
    const int h = (4 * e4) / D, d0 = (4 * e4) % D;
    const size_t ph = ((size_t)qi * a.Hq + (size_t)g * G + h) * a.nsplit;
    const float M = M_s[h];
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
    for (int c = 0; c < nchunk; ++c) {
      const float wgt = exp2_rel(a.part_ml[ph + c].x, M);
      const float4 v = *reinterpret_cast<const float4*>(a.part_o + (ph + c) * D + d0);
      acc.x = fmaf(wgt, v.x, acc.x);
      acc.y = fmaf(wgt, v.y, acc.y);
      acc.z = fmaf(wgt, v.z, acc.z);
      acc.w = fmaf(wgt, v.w, acc.w);
    }
    const float li = Linv_s[h];
    *reinterpret_cast<float4*>(o_out + (size_t)h * D + d0) = make_float4(acc.x * li, acc.y * li, acc.z * li, acc.w * li);
  }
  for (int j = kk + tid; j < a.kcap; j += NT) out[j] = -1;
  if (tid == 0) a.cnt[(size_t)qi * a.Hkv + g] = kk;
  if (kk == 0) return;
  if (kk == nF) {  // the budget covers the whole far range
    for (int j = tid; j < nF; j += NT) out[j] = j;
    return;
  }
  // ---- scores of the far range, 4 positions per thread and pass, kScoreHeads heads' loads in flight
  const size_t lrow = (size_t)qi * a.Hq + (size_t)g * G;
  const uint16_t* lcd = a.lcode + lrow * a.ld_logits;
  const float* lmx = a.lmax + lrow * (a.ld_logits / kLogitGroup);
  uint32_t* keys = a.scores + ((size_t)qi * a.Hkv + g) * a.ld_logits;
  // (one CTA-wide trip count: threads past nF only skip their loads)
  for (int base = 0; base < nF; base += 4 * NT) {
    const int s0 = base + 4 * tid;
    const bool mine = s0 < nF;
    float sc[4] = {0.f, 0.f, 0.f, 0.f};
    for (int h0 = 0; h0 < G; h0 += kScoreHeads) {
      uint2 c[kScoreHeads];  // 4 codes of one 16-position group
      float d[kScoreHeads];  // the group's max minus the head's lse
#pragma unroll
      for (int hh = 0; hh < kScoreHeads; ++hh)
        if (mine && h0 + hh < G) {
          c[hh] = __ldcs(reinterpret_cast<const uint2*>(lcd + (size_t)(h0 + hh) * a.ld_logits + s0));
          d[hh] = __ldg(lmx + (size_t)(h0 + hh) * (a.ld_logits / kLogitGroup) + s0 / kLogitGroup);
        }
#pragma unroll
      for (int hh = 0; hh < kScoreHeads; ++hh)
        if (mine && h0 + hh < G) {
          const float dd = d[hh] - lse2_s[h0 + hh];
          sc[0] += logit_term(c[hh].x & 0xffffu, dd);
          sc[1] += logit_term(c[hh].x >> 16, dd);
          sc[2] += logit_term(c[hh].y & 0xffffu, dd);
          sc[3] += logit_term(c[hh].y >> 16, dd);
        }
    }
    uint32_t key[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) key[e] = (s0 + e < nF) ? __float_as_uint(sc[e]) : 0u;
    if (mine) *reinterpret_cast<uint4*>(keys + s0) = make_uint4(key[0], key[1], key[2], key[3]);
#pragma unroll
    for (int e = 0; e < 4; ++e) hist_add(sm.hist, s0 + e < nF, key[e] >> 20);
  }
  __syncthreads();  // keys (global, read back through L2) and the histogram are complete
  int* la = fbuf;
  int* lsel = la + a.kcap;
  uint2* lc = reinterpret_cast<uint2*>(lsel + a.kcap);
  auto emit = [&](int j, int i) { out[j] = i; };
  if (filter_topk<NT, 8>(keys, nF, kk, nullptr, la, a.kcap, lc, kFilterCap, lsel, emit, sm)) return;
  // more candidates share the k-th key's top digit than the buffer holds: radix passes
  auto key = [&](int i) { return __ldcg(keys + i); };
  block_topk<NT>(nF, kk, key, emit, sm);
}

// ============================================================================ launchers
cudaError_t launch_combine(const CombineArgs& a, int Bq, cudaStream_t s) {
  if (score_select_fused(a, Bq)) {
    const size_t sm = select_smem(a.kcap);
    auto kern = a.D == 128 ? score_select_kernel<128> : score_select_kernel<64>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
    if (e != cudaSuccess) return e;
    kern<<<dim3(a.Hkv, Bq), kSelectThreads, sm, s>>>(a);
    return cudaGetLastError();
  }
  const int nscore = a.select ? (int)((a.ld_logits + kScoreChunk - 1) / kScoreChunk) : 1;
  dim3 grid(nscore, a.Hkv, Bq);
  if (a.D == 128) merge_score_kernel<128><<<grid, kMergeThreads, 0, s>>>(a);
  else if (a.D == 64) merge_score_kernel<64><<<grid, kMergeThreads, 0, s>>>(a);
  else return cudaErrorInvalidValue;
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || !a.select) return e;
  if (a.sel_block > 1) {
    const int nb_max = (int)((a.ld_logits + a.sel_block - 1) / a.sel_block);
    const size_t smb = (size_t)(nb_max + a.k / a.sel_block) * sizeof(uint32_t);
    e = cudaFuncSetAttribute(block_select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smb);
    if (e != cudaSuccess) return e;
    block_select_kernel<<<dim3(a.Hkv, Bq), kSelectThreads, smb, s>>>(a);
    return cudaGetLastError();
  }
  const size_t sm = select_smem(a.kcap);
  e = cudaFuncSetAttribute(select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
  if (e != cudaSuccess) return e;
  return launch_clustered(select_kernel, a.Hkv, Bq, sm, sel_cluster_size(a.ld_logits, (long long)a.Hkv * Bq), s, a);
}

}  // namespace hs2

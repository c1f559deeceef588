// indexer.cu — CSA2 hierarchical sparse indexer: lightning-indexer scan on tcgen05.
//
// "2.3.1 · CSA、HCA 与 CSA2: 压缩序列上的稀疏检索和跨层复用", §3.1-3.2: the first Full
// layer scores every legal position; the same scores give its top-k positions and, per
// 8-position block, a block maximum from which up to 2048 blocks form the candidate
// pool; Reindex layers rescore only the pool's positions with their own query. The
// score is the lightning indexer of "Lecture 10 · 混合架构与稀疏注意力", §5.1:
// I(s) = sum_j w_j * ReLU(q_j . k_s), one indexer key shared by all indexer heads.
//
// lightning_scan_kernel: one batch row per blockIdx.y; each CTA walks a contiguous range
// of 128-candidate tiles. Warp 0 streams K tiles with TMA (128-byte swizzle; Full: two
// 64-row page boxes per d-half; Reindex: sixteen 8-row pool-block boxes per d-half) into
// a 4-stage ring; warp 1 issues tcgen05.mma (M = 128 candidates, N = 64 heads, K = 128)
// into one of two TMEM accumulators; warps 2-5 read the accumulator rows (one candidate
// per thread, 64 head columns), apply ReLU and the head weights, and write uint32 keys,
// 8-block maxima (Full) and the top-12-bit histograms for the selection.
#include <cuda.h>

#include "common.cuh"
#include "kernels.h"
#include "tc.cuh"
#include "topk.cuh"

namespace hs2 {

namespace {

constexpr int kIdxHeads = 64;      // N of the MMA (indexer heads)
constexpr int kIdxDim = 128;       // contraction (indexer head dim)
constexpr int kIdxTile = 128;      // candidates per tile (M of the MMA)
constexpr int kIdxStages = 4;
constexpr int kIdxThreads = 192;   // 6 warps: TMA, MMA, 4 x epilogue
constexpr uint32_t kStageBytes = kIdxTile * kIdxDim * 2;       // 32 KB
constexpr uint32_t kQBytes = kIdxHeads * kIdxDim * 2;          // 16 KB
constexpr uint32_t kTmemCols = 128;                            // 2 accumulators x 64 columns
constexpr int kIdxPoolBatch = 16;  // Reindex tiles whose pool rows the producer warp resolves at once

struct IdxSmem {
  uint8_t q[kQBytes];                       // B operand, 2 K-blocks of [64 rows x 128 B]
  uint8_t k[kIdxStages][kStageBytes];       // A operand, 2 K-blocks of [128 rows x 128 B]
  uint32_t hist[kRadixBins];
  uint32_t bhist[kRadixBins];
  uint64_t full[kIdxStages], empty[kIdxStages], qbar, accf[2], acce[2];
  int prow[kIdxPoolBatch * 16];  // Reindex: pool rows of the next kIdxPoolBatch tiles
  uint32_t tmem_base;
  int abort;
};

}  // namespace

__global__ void __launch_bounds__(kIdxThreads, 1)
    lightning_scan_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_q,
                          const IdxArgs a) {
  extern __shared__ __align__(1024) uint8_t dsmem[];
  IdxSmem& sm = *reinterpret_cast<IdxSmem*>(dsmem + ((1024 - (tc::smem_u32(dsmem) & 1023)) & 1023));
  const int b = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = a.seq_len[b];
  const int npages = (t + kPage - 1) / kPage;
  if (t < 1 || t > a.max_t || npages > a.max_pages) {
    if (threadIdx.x == 0 && blockIdx.x == 0) flag_error(a.dev_err, HS2_DEV_BAD_LENGTH);
    return;
  }
  const int32_t* bt = a.bt + (size_t)b * a.max_pages;
  // candidates of this row
  int n_cand, pc = 0;
  const int32_t* pool = nullptr;
  if (a.mode == 0) {
    n_cand = t;
  } else {
    pool = a.pool + (size_t)b * a.max_blocks;
    pc = max(0, min(a.max_blocks, a.pool_cnt[b]));
    n_cand = 0;
    if (pc > 0) {
      const int last = pool[pc - 1];
      n_cand = (pc - 1) * 8 + max(0, min(8, t - 8 * last));
    }
  }
  const int ntiles = (n_cand + kIdxTile - 1) / kIdxTile;
  const int tile0 = blockIdx.x * a.tiles_per_cta;
  const int tile1 = min(ntiles, tile0 + a.tiles_per_cta);
  if (tile0 >= tile1) return;
  const int ntl = tile1 - tile0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kIdxStages; ++s) {
      tc::mbar_init(&sm.full[s], 1);
      tc::mbar_init(&sm.empty[s], 1);
    }
    tc::mbar_init(&sm.qbar, 1);
    for (int s = 0; s < 2; ++s) {
      tc::mbar_init(&sm.accf[s], 1);
      tc::mbar_init(&sm.acce[s], 128);
    }
    sm.abort = 0;
    tc::fence_mbar_init();
  }
  for (int i = threadIdx.x; i < kRadixBins; i += kIdxThreads) {
    sm.hist[i] = 0;
    sm.bhist[i] = 0;
  }
  if (warp == 1) tc::tmem_alloc(&sm.tmem_base, kTmemCols);
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = sm.tmem_base;

  if (warp == 0) {
    // ---------------------------------------------------------------- TMA producer
    // Lane 0 issues; in Reindex mode the whole warp first resolves the pool blocks of the next
    // kIdxPoolBatch tiles together (pool entries, then the block table: two dependent rounds
    // of loads per batch) into shared memory.
    if (lane == 0) {
      tc::prefetch_tmap(&tm_k);
      tc::mbar_arrive_expect_tx(&sm.qbar, kQBytes);
      tc::tma_load_2d(sm.q, &tm_q, 0, b * kIdxHeads, &sm.qbar);
      tc::tma_load_2d(sm.q + kQBytes / 2, &tm_q, 64, b * kIdxHeads, &sm.qbar);
    }
    int issued = 0;
    for (int li = 0; li < ntl; ++li) {
      if (__shfl_sync(0xffffffffu, *(volatile int*)&sm.abort, 0)) break;
      const int st = li % kIdxStages;
      const int tile = tile0 + li;
      if (a.mode != 0 && li % kIdxPoolBatch == 0) {
        // pool rows of tiles li .. li + kIdxPoolBatch - 1: every load of a round issued before
        // any check (a flagged error is an atomic later loads cannot move across)
        constexpr int PER = kIdxPoolBatch * 16 / 32;
        int bid[PER], prev[PER], phys[PER];
#pragma unroll
        for (int q = 0; q < PER; ++q) {
          const int e = tile * 16 + lane + 32 * q;
          bid[q] = e < pc ? pool[e] : -1;
          prev[q] = (e < pc && e > 0) ? pool[e - 1] : -1;
        }
#pragma unroll
        for (int q = 0; q < PER; ++q) {
          const int e = tile * 16 + lane + 32 * q;
          const bool bad = e < pc && (bid[q] < 0 || bid[q] * 8 >= t || (e > 0 && prev[q] >= bid[q]));
          if (bad) bid[q] = -2;
          phys[q] = (e < pc && !bad) ? bt[bid[q] * 8 / kPage] : 0;
        }
#pragma unroll
        for (int q = 0; q < PER; ++q) {
          const int e = tile * 16 + lane + 32 * q;
          int r = -1;
          if (e < pc) {
            if (bid[q] == -2) flag_error(a.dev_err, HS2_DEV_BAD_INDEX);
            else if (phys[q] < 0 || phys[q] >= a.num_pages) flag_error(a.dev_err, HS2_DEV_BAD_PAGE);
            else r = phys[q] * kPage + (bid[q] * 8) % kPage;
          }
          sm.prow[lane + 32 * q] = r;
        }
        __syncwarp();
      }
      // Reindex: the pool row of block tile * 16 + lane (lanes 0-15)
      const int row = (a.mode != 0 && lane < 16) ? sm.prow[(li % kIdxPoolBatch) * 16 + lane] : -1;
      bool ok = true;
      if (lane == 0) ok = tc::mbar_wait(&sm.empty[st], ((li / kIdxStages) & 1) ^ 1);
      if (!__shfl_sync(0xffffffffu, ok, 0)) {
        if (lane == 0) {
          flag_error(a.dev_err, HS2_DEV_TIMEOUT);
          atomicExch(&sm.abort, 1);
        }
        break;
      }
      uint8_t* dst = sm.k[st];
      if (a.mode == 0) {
        if (lane == 0) {
          int rows[2];
          uint32_t bytes = 0;
          for (int pg = 0; pg < 2; ++pg) {
            const int lp = tile * 2 + pg;
            rows[pg] = -1;
            if (lp < npages) {
              const int phys = bt[lp];
              if (phys < 0 || phys >= a.num_pages) flag_error(a.dev_err, HS2_DEV_BAD_PAGE);
              else { rows[pg] = phys * kPage; bytes += 2 * 8192; }
            }
          }
          tc::mbar_arrive_expect_tx(&sm.full[st], bytes);
          for (int pg = 0; pg < 2; ++pg)
            if (rows[pg] >= 0)
              for (int h = 0; h < 2; ++h) tc::tma_load_2d(dst + h * 16384 + pg * 8192, &tm_k, 64 * h, rows[pg], &sm.full[st]);
        }
      } else {
        const unsigned have = __ballot_sync(0xffffffffu, row >= 0);
        if (lane == 0) tc::mbar_arrive_expect_tx(&sm.full[st], (uint32_t)__popc(have) * 2 * 1024);
        __syncwarp();  // the expected bytes are armed before any copy can complete
        if (row >= 0)
          for (int h = 0; h < 2; ++h) tc::tma_load_2d(dst + h * 16384 + lane * 1024, &tm_k, 64 * h, row, &sm.full[st]);
      }
      issued = li + 1;
    }
    if (lane == 0) {
      // leave no copy in flight: wait (bounded) for the last tiles issued to each stage
      for (int li = max(0, issued - kIdxStages); li < issued; ++li)
        (void)tc::mbar_wait(&sm.full[li % kIdxStages], (li / kIdxStages) & 1);
      (void)tc::mbar_wait(&sm.qbar, 0);
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = tc::idesc_bf16_f32(kIdxTile, kIdxHeads);
      int last = -1;
      if (!tc::mbar_wait(&sm.qbar, 0)) {
        flag_error(a.dev_err, HS2_DEV_TIMEOUT);
        atomicExch(&sm.abort, 1);
      } else {
        for (int li = 0; li < ntl && !*(volatile int*)&sm.abort; ++li) {
          const int st = li % kIdxStages, ac = li & 1;
          if (!tc::mbar_wait(&sm.full[st], (li / kIdxStages) & 1) ||
              !tc::mbar_wait(&sm.acce[ac], ((li >> 1) & 1) ^ 1)) {
            flag_error(a.dev_err, HS2_DEV_TIMEOUT);
            atomicExch(&sm.abort, 1);
            break;
          }
          tc::tc_fence_after();
          const uint32_t abase = tc::smem_u32(sm.k[st]);
          const uint32_t bbase = tc::smem_u32(sm.q);
#pragma unroll
          for (int kk = 0; kk < kIdxDim / 16; ++kk) {
            const uint32_t koff = (kk >> 2) * 16384u + (kk & 3) * 32u;
            const uint32_t qoff = (kk >> 2) * 8192u + (kk & 3) * 32u;
            tc::mma_bf16(tmem + ac * 64, tc::sdesc_sw128(abase + koff), tc::sdesc_sw128(bbase + qoff), idesc,
                         kk > 0 ? 1u : 0u);
          }
          tc::mma_commit(&sm.empty[st]);
          tc::mma_commit(&sm.accf[ac]);
          last = li;
        }
      }
      if (last >= 0) (void)tc::mbar_wait(&sm.accf[last & 1], (last >> 1) & 1);  // no MMA left in flight
    }
  } else {
    // ---------------------------------------------------------------- epilogue (warps 2..5)
    const int qd = warp & 3;  // TMEM lane quadrant this warp may access
    const int r = qd * 32 + lane;
    float wv[kIdxHeads];
#pragma unroll
    for (int j = 0; j < kIdxHeads; ++j) wv[j] = a.w_idx[(size_t)b * kIdxHeads + j];
    uint32_t* keys = a.keys + (size_t)b * a.ld_keys;
    uint32_t* bkeys = a.mode == 0 ? a.bkeys + (size_t)b * a.ld_bkeys : nullptr;
    const int nblk = (t + 7) / 8;
    for (int li = 0; li < ntl; ++li) {
      const int ac = li & 1;
      if (*(volatile int*)&sm.abort || !tc::mbar_wait(&sm.accf[ac], (li >> 1) & 1)) {
        if (!*(volatile int*)&sm.abort) {
          flag_error(a.dev_err, HS2_DEV_TIMEOUT);
          atomicExch(&sm.abort, 1);
        }
        break;
      }
      tc::tc_fence_after();
      float v0[32], v1[32];
      const uint32_t ta = tmem + ((uint32_t)(qd * 32) << 16) + ac * 64;
      tc::tmem_ld32(ta, v0);
      tc::tmem_ld32(ta + 32, v1);
      tc::tc_fence_before();
      tc::mbar_arrive(&sm.acce[ac]);
      float I = 0.f;
#pragma unroll
      for (int j = 0; j < 32; ++j) I = fmaf(wv[j], fmaxf(v0[j], 0.f), I);
#pragma unroll
      for (int j = 0; j < 32; ++j) I = fmaf(wv[32 + j], fmaxf(v1[j], 0.f), I);
      const int c = (tile0 + li) * kIdxTile + r;
      const bool valid = c < n_cand;
      const uint32_t key = valid ? __float_as_uint(I) : 0u;
      if (valid) keys[c] = key;
      hist_add_warp(sm.hist, valid, key >> 20);
      if (a.mode == 0) {
        float bm = valid ? I : 0.f;  // I >= 0, so invisible members never raise a block max
        bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 1));
        bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 2));
        bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 4));
        const bool bv = (lane & 7) == 0 && c / 8 < nblk;
        const uint32_t bk = __float_as_uint(bm);
        if (bv) bkeys[c / 8] = bk;
        hist_add_warp(sm.bhist, bv, bk >> 20);
      }
    }
  }
  __syncthreads();
  // flush the CTA histograms
  uint32_t* gh = a.hist + (size_t)b * kRadixBins;
  uint32_t* gbh = a.mode == 0 ? a.bhist + (size_t)b * kRadixBins : nullptr;
  for (int i = threadIdx.x; i < kRadixBins; i += kIdxThreads) {
    if (sm.hist[i]) atomicAdd(&gh[i], sm.hist[i]);
    if (gbh && sm.bhist[i]) atomicAdd(&gbh[i], sm.bhist[i]);
  }
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 1) tc::tmem_dealloc(tmem, kTmemCols);
}

size_t lightning_scan_smem() { return sizeof(IdxSmem) + 1024; }

cudaError_t launch_lightning_scan(const CUtensorMap& tm_k, const CUtensorMap& tm_q, const IdxArgs& a, int B,
                                  int grid_x, cudaStream_t s) {
  const size_t sm = lightning_scan_smem();
  cudaError_t e = cudaFuncSetAttribute(lightning_scan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
  if (e != cudaSuccess) return e;
  lightning_scan_kernel<<<dim3(grid_x, B), kIdxThreads, sm, s>>>(tm_k, tm_q, a);
  return cudaGetLastError();
}

}  // namespace hs2

// prefill_select.cu — window-excluding top-k for every causal row of a bf16 prefill.
//
// Row i's selection score of a far position s (s < i+1-w) is the FA attention
// probability summed over the query heads of a KV head ("HySparse2：整体架构、KV 生命周期
// 与 PD 分离", §5, §7.2), normalised with the row's final lse (written by the forward
// kernel). The n x n score matrix is never stored: scores are produced tile by tile from
// a tcgen05 recomputation of Q K^T and consumed on the fly.
//
// prefill_scan_kernel — one CTA per (128-row tile, KV head), four scoring threads per row:
//   sweep 0 (sampled): every 8th key position only, 128 of them per tile (1024 positions;
//            a strided tensor map loads just those K rows); each thread bins the sampled
//            scores of its quarter of the row's columns into the row's 256-bin log histogram
//            (1/8 octave per bin, 16-bit counts in shared memory, atomic adds), then the row's
//            first thread picks a threshold tau whose estimated count of keys at or above it
//            is 1.35 times the budget;
//   sweep 1 (exact): every key tile; the scoring threads stage the tile's 128 x 128 scores in
//            shared memory, then each scoring warp takes 8 rows and appends (key, position)
//            of the scores >= tau of a row, in ascending position, into the row's candidate
//            buffer (capacity C) with ballot compaction, so each store is a contiguous run;
//            past capacity it keeps only the largest dropped key.
//   Warp 0 streams K tiles and, per head, the head's Q tile (TMA); warp 1 issues
//   S_h = Q_h K^T (M=128 rows, N=128 keys, K=128) into four TMEM buffers.
// prefill_topk_warp_kernel — one warp per (row, KV head): exact top-k over the row's
//   candidates (radix select with warp-level ballots and shuffles, ties to the lower
//   position, ascending output). The candidates are a superset of the answer when (a) at
//   least k of them are >= tau and (b) no dropped key exceeds the k-th largest kept key
//   (dropped positions come after every kept one, so equal keys lose); otherwise the row
//   goes to a list of rows to complete.
// prefill_complete_kernel — each listed (row, KV head) again, exactly: its scores over the
//   whole far range recomputed (mma.sync, keys as M, the heads of the KV head as N) into a
//   per-CTA key row, then a block-wide radix top-k over all of them. Every row therefore
//   gets its exact top-k, whatever the score distribution.
#include <cuda.h>

#include <algorithm>

#include "common.cuh"
#include "kernels.h"
#include "tc.cuh"
#include "topk.cuh"

namespace hs2 {

namespace {

constexpr int kST = 128;        // rows per tile = keys per key tile
constexpr int kSThreads = 576;  // TMA warp, MMA warp, 16 scoring warps (four per TMEM lane quadrant)
constexpr uint32_t kSTile = kST * 128 * 2;
constexpr int kBins = 256;
constexpr uint32_t kBinBase = 0x410 - (kBins - 1);  // bin 255 holds keys >> 20 == 0x410 (score 8.0)
// The sampled sweep scores every 4th position (position-correlated scores would bias a
// sample of whole tiles); a sampled key tile holds 128 such positions, 1024 apart at most.
constexpr int kSampleStride = kPsSampleStride;
constexpr int kSampSpan = kST * kSampleStride;                // positions covered by a sampled key tile
constexpr int kSampPages = kSampSpan / kPage;                 // pages of a sampled key tile (16)
constexpr uint32_t kSampBoxBytes = kPsSampleRowsPerPage * 128;  // one 64-column half of a page's sampled rows

constexpr int kCompRows = 4;  // rows compacted together by a scoring warp (of its 8)
constexpr int kQStages = 3;  // Q tiles in flight: a head's load overlaps the two MMAs before it

struct PsSmem {
  uint8_t q[kQStages][kSTile];     // A of S (query rows x d), one head per stage
  uint8_t k[2][kSTile];            // B of S (keys x d)
  union {
    struct {
      uint32_t hist[kBins][kST / 2];  // per-row sample histograms, 16-bit counts (rows 2m, 2m+1 share
    } samp;                           // a word), filled with shared-memory atomics
    float tile[kST * kST];         // exact sweep: the key tile's scores, row-major, swizzled (tile_at)
  };
  uint32_t tau[kST];               // each row's threshold, set at the end of the sampled sweep
  uint64_t q_full[kQStages], q_empty[kQStages], k_full[2], k_empty[2], s_full[4], s_empty[4];
  uint64_t h_done;                 // sampled sweep: the other three quarters' counts are in
  uint64_t t_full, t_free;         // exact sweep: tile written by all scoring threads / tile consumed
  uint32_t tmem_base;
  int abort;
};

// element (row r, column c) of the staged score tile; the XOR keeps both the scoring
// threads' 16-byte column writes and the row-wise 32-lane reads free of bank conflicts
HS2_DEVI int tile_at(int r, int c) { return r * kST + (c ^ ((r & 7) << 2)); }

HS2_DEVI bool aborted(PsSmem& sm) { return *(volatile int*)&sm.abort != 0; }
HS2_DEVI void set_abort(PsSmem& sm, int32_t* dev_err) {
  flag_error(dev_err, HS2_DEV_TIMEOUT);
  atomicExch(&sm.abort, 1);
}

}  // namespace

__global__ void __launch_bounds__(kSThreads, 1)
    prefill_scan_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                        const __grid_constant__ CUtensorMap tm_ks, const PsArgs a) {
  extern __shared__ __align__(1024) uint8_t dsmem[];
  PsSmem& sm = *reinterpret_cast<PsSmem*>(dsmem + ((1024 - (tc::smem_u32(dsmem) & 1023)) & 1023));
  const int tiles = (a.row1 - a.row0 + kST - 1) / kST;
  const int tile = tiles - 1 - blockIdx.x;  // heaviest first
  const int g = blockIdx.y, G = a.G;
  const int i0 = a.row0 + tile * kST;
  const int i_last = min(a.row1, i0 + kST) - 1;
  const int keys_needed = max(0, i_last + 1 - a.w);
  const int J = (keys_needed + kST - 1) / kST;  // key tiles of the exact sweep
  const int J0 = (keys_needed + kSampSpan - 1) / kSampSpan;  // sampled sweep: tiles of sampled keys
  const int NKT = J0 + J;                       // key-tile items over both sweeps
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = a.seq_len[0];
  const int npages = (t + kPage - 1) / kPage;
  if (J == 0) return;
  if (t < a.n || npages > a.max_pages) {
    if (threadIdx.x == 0) flag_error(a.dev_err, HS2_DEV_BAD_LENGTH);
    return;
  }
  if (threadIdx.x == 0) {
    for (int s = 0; s < kQStages; ++s) {
      tc::mbar_init(&sm.q_full[s], 1);
      tc::mbar_init(&sm.q_empty[s], 1);
    }
    for (int s = 0; s < 4; ++s) {
      tc::mbar_init(&sm.s_full[s], 1);
      tc::mbar_init(&sm.s_empty[s], 16);
    }
    for (int s = 0; s < 2; ++s) {
      tc::mbar_init(&sm.k_full[s], 1);
      tc::mbar_init(&sm.k_empty[s], 1);
    }
    tc::mbar_init(&sm.h_done, 384);
    tc::mbar_init(&sm.t_full, 512);
    tc::mbar_init(&sm.t_free, 512);
    sm.abort = 0;
    tc::fence_mbar_init();
  }
  for (int e = threadIdx.x; e < kBins * kST / 2; e += kSThreads) (&sm.samp.hist[0][0])[e] = 0u;
  if (warp == 1) tc::tmem_alloc(&sm.tmem_base, 512);
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tS = sm.tmem_base;
  auto jof = [&](int kt) { return kt < J0 ? kt : kt - J0; };

  if (warp == 0) {
    if (lane == 0) {
      // ---------------------------------------------------------------- TMA producer
      int kissued = 0, qissued = 0;
      for (int kt = 0; kt < NKT && !aborted(sm); ++kt) {
        const int ks = kt & 1;
        if (!tc::mbar_wait(&sm.k_empty[ks], ((kt >> 1) & 1) ^ 1)) { set_abort(sm, a.dev_err); break; }
        const int j = jof(kt);
        if (kt < J0) {
          // sampled keys: rows 0, 8, ..., 56 of each of 16 pages, 8 tile rows (one 1 KB swizzle
          // atom) per page
          int rows[kSampPages];
          uint32_t bytes = 0;
          for (int pg = 0; pg < kSampPages; ++pg) {
            const int lp = kSampPages * j + pg;
            rows[pg] = -1;
            if (lp < npages) {
              const int phys = a.bt[lp];
              if (phys < 0 || phys >= a.num_pages) flag_error(a.dev_err, HS2_DEV_BAD_PAGE);
              else { rows[pg] = (phys * a.Hkv + g) * kPsSampleRowsPerPage; bytes += 2 * kSampBoxBytes; }
            }
          }
          tc::mbar_arrive_expect_tx(&sm.k_full[ks], bytes);
          for (int pg = 0; pg < kSampPages; ++pg)
            if (rows[pg] >= 0)
              for (int hh = 0; hh < 2; ++hh)
                tc::tma_load_2d(sm.k[ks] + hh * 16384 + pg * kSampBoxBytes, &tm_ks, 64 * hh, rows[pg],
                                &sm.k_full[ks]);
        } else {
          int rows[2];
          uint32_t bytes = 0;
          for (int pg = 0; pg < 2; ++pg) {
            const int lp = 2 * j + pg;
            rows[pg] = -1;
            if (lp < npages) {
              const int phys = a.bt[lp];
              if (phys < 0 || phys >= a.num_pages) flag_error(a.dev_err, HS2_DEV_BAD_PAGE);
              else { rows[pg] = (phys * a.Hkv + g) * kPage; bytes += 2 * 8192; }
            }
          }
          tc::mbar_arrive_expect_tx(&sm.k_full[ks], bytes);
          for (int pg = 0; pg < 2; ++pg)
            if (rows[pg] >= 0)
              for (int hh = 0; hh < 2; ++hh)
                tc::tma_load_2d(sm.k[ks] + hh * 16384 + pg * 8192, &tm_k, 64 * hh, rows[pg], &sm.k_full[ks]);
        }
        kissued = kt + 1;
        bool ok = true;
        for (int hl = 0; hl < G; ++hl) {
          const int it = kt * G + hl, qs = it % kQStages;
          if (!tc::mbar_wait(&sm.q_empty[qs], ((it / kQStages) & 1) ^ 1)) { ok = false; break; }
          tc::mbar_arrive_expect_tx(&sm.q_full[qs], kSTile);
          tc::tma_load_3d(sm.q[qs], &tm_q, 0, g * G + hl, i0, &sm.q_full[qs]);
          tc::tma_load_3d(sm.q[qs] + kSTile / 2, &tm_q, 64, g * G + hl, i0, &sm.q_full[qs]);
          qissued = it + 1;
        }
        if (!ok) { set_abort(sm, a.dev_err); break; }
      }
      for (int kt = max(0, kissued - 2); kt < kissued; ++kt) (void)tc::mbar_wait(&sm.k_full[kt & 1], (kt >> 1) & 1);
      for (int it = max(0, qissued - kQStages); it < qissued; ++it)
        (void)tc::mbar_wait(&sm.q_full[it % kQStages], (it / kQStages) & 1);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------------------------------------------------------- MMA issuer
      constexpr uint32_t idS = tc::idesc_bf16_f32(kST, kST);
      int last = -1;
      bool ok = true;
      for (int kt = 0; kt < NKT && ok && !aborted(sm); ++kt) {
        const int ks = kt & 1;
        if (!tc::mbar_wait(&sm.k_full[ks], (kt >> 1) & 1)) { ok = false; break; }
        const uint32_t kb = tc::smem_u32(sm.k[ks]);
        for (int hl = 0; hl < G; ++hl) {
          const int it = kt * G + hl, qs = it % kQStages, sb = it & 3;
          if (!tc::mbar_wait(&sm.q_full[qs], (it / kQStages) & 1) || !tc::mbar_wait(&sm.s_empty[sb], ((it >> 2) & 1) ^ 1)) {
            ok = false;
            break;
          }
          tc::tc_fence_after();
          const uint32_t qb = tc::smem_u32(sm.q[qs]);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint32_t off = (kk >> 2) * 16384u + (kk & 3) * 32u;
            tc::mma_bf16(tS + sb * 128, tc::sdesc_sw128(qb + off), tc::sdesc_sw128(kb + off), idS, kk > 0 ? 1u : 0u);
          }
          tc::mma_commit(&sm.s_full[sb]);
          tc::mma_commit(&sm.q_empty[qs]);
          last = it;
        }
        if (ok) tc::mma_commit(&sm.k_empty[ks]);
      }
      if (!ok) set_abort(sm, a.dev_err);
      if (last >= 0) (void)tc::mbar_wait(&sm.s_full[last & 3], (last >> 2) & 1);
    }
  } else {
    // ---------------------------------------------------------------- scoring warps
    // warps 2-5 own rows and columns 0-31 of every S tile; warps 6-9, 10-13 and 14-17 take
    // columns 32-63, 64-95 and 96-127 of the same rows (a warp reaches only its TMEM lane
    // quadrant, warp % 4). In the sampled sweep every warp bins its columns into the rows'
    // shared histograms and the row owner (first quarter) sets the threshold; in the exact
    // sweep all sixteen warps stage the tile's scores, then each compacts 8 rows.
    const int quarter = (warp - 2) >> 2;
    const int qd = warp & 3;
    const int r = qd * 32 + lane;
    const int i = i0 + r;
    const bool row_ok = i < a.row1;
    const int nF = row_ok ? max(0, i + 1 - a.w) : 0;
    const bool ranked = nF > a.k;  // rows whose far range fits the budget need no candidates
    const uint32_t lane_off = (uint32_t)(qd * 32) << 16;
    // the row's lse of each head: G floats, read through L1 one head ahead of their use
    const float* lse2_row = a.lse2 + (size_t)(row_ok ? i : a.row0) * a.Hq + g * G;
    // rows this warp compacts in the exact sweep: lane l < 8 keeps the state of row 8 sw + l
    const int sw = warp - 2;
    const int cr = sw * 8 + (lane & 7);
    const int ci = i0 + cr;
    const bool c_ok = lane < 8 && ci < a.row1;
    const int c_nF = c_ok ? max(0, ci + 1 - a.w) : 0;
    const bool c_ranked = c_nF > a.k;
    uint32_t c_tau = 0xffffffffu;  // read from shared memory once the sampled sweep is over
    int c_cnt = 0;
    uint32_t c_drop = 0;
    uint32_t tau = 0xffffffffu;  // the owner's threshold, from its row's sample histogram
    bool ok = true;
    for (int kt = 0; kt < NKT && ok; ++kt) {
      const bool sample = kt < J0;
      const int j = jof(kt);
      float sc[32];
#pragma unroll
      for (int e = 0; e < 32; ++e) sc[e] = 0.f;
      float l2_next = __ldg(lse2_row);
      for (int hl = 0; hl < G; ++hl) {
        const float l2 = l2_next;
        if (hl + 1 < G) l2_next = __ldg(lse2_row + hl + 1);
        const int it = kt * G + hl, sb = it & 3;
        // votes keep the warp converged for the warp-collective TMEM loads
        if (!__all_sync(0xffffffffu, !aborted(sm) && tc::mbar_wait(&sm.s_full[sb], (it >> 2) & 1))) { ok = false; break; }
        __syncwarp();
        tc::tc_fence_after();
        uint32_t raw[32];
        tc::tmem_ld32_async(tS + lane_off + sb * 128 + quarter * 32, raw);
        tc::tmem_wait_ld(raw);
        tc::tc_fence_before();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(&sm.s_empty[sb]);
#pragma unroll
        for (int e = 0; e < 32; ++e) sc[e] += tc::ex2(fmaf(__uint_as_float(raw[e]), a.scale_log2, -l2));
      }
      if (!ok) break;
      if (sample) {
        if (ranked) {
          // column 32 quarter + e of a sampled tile is position j * kSampSpan + kSampleStride * (32 quarter + e)
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            if (j * kSampSpan + kSampleStride * (quarter * 32 + e) < nF) {
              const int bin = min(kBins - 1, max(0, (int)(__float_as_uint(sc[e]) >> 20) - (int)kBinBase));
              atomicAdd(&sm.samp.hist[bin][r >> 1], 1u << ((r & 1) * 16));
            }
          }
        }
        if (kt == J0 - 1) {
          if (quarter != 0) {
            tc::mbar_arrive(&sm.h_done);  // this thread's counts are in
          } else {
            if (!__all_sync(0xffffffffu, tc::mbar_wait(&sm.h_done, 0))) { ok = false; break; }
            if (ranked) {
              // threshold: the estimated count at or above it (sample count scaled by the row's
              // sampling rate; the sweep saw every position of [0, nF) that is a multiple of the
              // stride) reaches 1.35 times the budget. Fewer candidates mean fewer stores here
              // and a shorter top-k; a row the estimate leaves short of k is completed exactly
              // (prefill_complete_kernel). On the AR(1) workload at n = 32768 (whole call):
              // stride 4 with 1.25 15.43 ms; stride 8 with 1.25 15.33 ms, 7 rows completed;
              // stride 8 with 1.35 15.06 ms, none (stride 4: 1.1 left 221 rows to complete and
              // was slower overall, 2 was 0.74 ms slower).
              const int n_samp = (nF + kSampleStride - 1) / kSampleStride;
              const float scale = (float)nF / (float)n_samp;
              const float target = 1.35f * (float)a.k;
              float cum = 0.f;
              tau = 0u;
              for (int b = kBins - 1; b >= 0; --b) {
                cum += scale * (float)((sm.samp.hist[b][r >> 1] >> ((r & 1) * 16)) & 0xffffu);
                if (cum >= target) {
                  tau = b == 0 ? 0u : (uint32_t)(kBinBase + b) << 20;
                  break;
                }
              }
            }
            sm.tau[r] = tau;
          }
          tc::mbar_arrive(&sm.t_free);  // the histograms are free for the score tile
        }
        continue;
      }
      // exact sweep: stage the tile, then compact rows 8 sw .. 8 sw + 7
      const int x = kt - J0;
      if (!__all_sync(0xffffffffu, tc::mbar_wait(&sm.t_free, x & 1))) { ok = false; break; }
      if (x == 0) c_tau = sm.tau[cr];
#pragma unroll
      for (int q = 0; q < 8; ++q)
        *reinterpret_cast<float4*>(&sm.tile[tile_at(r, quarter * 32 + 4 * q)]) =
            make_float4(sc[4 * q], sc[4 * q + 1], sc[4 * q + 2], sc[4 * q + 3]);
      tc::mbar_arrive(&sm.t_full);
      if (!__all_sync(0xffffffffu, tc::mbar_wait(&sm.t_full, x & 1))) { ok = false; break; }
      const int s0 = j * kST;
      const int c_lim = c_ranked ? c_nF - s0 : 0;  // columns of this tile inside the row's far range
      const uint32_t below = (1u << lane) - 1u;
      // kCompRows rows at a time: their loads, ballots and counts are independent chains
#pragma unroll 1
      for (int l0 = 0; l0 < 8; l0 += kCompRows) {
        int lim[kCompRows], n_r[kCompRows];
        uint32_t t_r[kCompRows], key[kCompRows][4], bal[kCompRows][4];
#pragma unroll
        for (int u = 0; u < kCompRows; ++u) {
          lim[u] = __shfl_sync(0xffffffffu, c_lim, l0 + u);
          t_r[u] = __shfl_sync(0xffffffffu, c_tau, l0 + u);
          n_r[u] = __shfl_sync(0xffffffffu, c_cnt, l0 + u);
        }
#pragma unroll
        for (int u = 0; u < kCompRows; ++u)
#pragma unroll
          for (int m = 0; m < 4; ++m) {
            const int c = m * 32 + lane;
            key[u][m] = __float_as_uint(sm.tile[tile_at(sw * 8 + l0 + u, c)]);
            bal[u][m] = __ballot_sync(0xffffffffu, c < lim[u] && key[u][m] >= t_r[u]);
          }
#pragma unroll
        for (int u = 0; u < kCompRows; ++u) {
          // rows outside the block or the budget have empty ballots: nothing is stored for them
          const size_t slot = ((size_t)(i0 + sw * 8 + l0 + u - a.row0) * a.Hkv + g) * a.cap;
          uint32_t d_r = 0;
#pragma unroll
          for (int m = 0; m < 4; ++m) {
            const bool pass = (bal[u][m] >> lane) & 1u;
            const int at = n_r[u] + __popc(bal[u][m] & below);
            const bool st = pass && at < a.cap;
            if (st) {
              a.cand_key[slot + at] = key[u][m];
              a.cand_pos[slot + at] = s0 + m * 32 + lane;
            }
            d_r = max(d_r, (pass && !st) ? key[u][m] : 0u);
            n_r[u] += __popc(bal[u][m]);
          }
          if (__any_sync(0xffffffffu, d_r != 0))
            for (int o = 16; o > 0; o >>= 1) d_r = max(d_r, __shfl_xor_sync(0xffffffffu, d_r, o));
          if (lane == l0 + u) {
            c_cnt = min(n_r[u], a.cap);
            c_drop = max(c_drop, d_r);
          }
        }
      }
      tc::mbar_arrive(&sm.t_free);
    }
    if (!ok) set_abort(sm, a.dev_err);
    if (c_ok) {
      const size_t rs = (size_t)(ci - a.row0) * a.Hkv + g;
      a.cand_cnt[rs] = c_ranked ? c_cnt : 0;
      a.cand_drop[rs] = c_drop;
      a.cand_tau[rs] = c_tau;
    }
  }
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 1) tc::tmem_dealloc(sm.tmem_base, 512);
}

// prefill_topk_warp_kernel (see the top of the file): no CTA barrier anywhere. Four radix
// passes of 8 bits, each a histogram of the candidates still matching the chosen prefix in
// the warp's own 256 shared-memory bins (keys read from L2 on every pass), the digit holding
// the kk-th key found from the top bin down with a warp scan; then the candidates in index
// order (= ascending position) are compacted with ballots: every key above T and the first
// take_eq keys equal to T.
constexpr int kTopkWarps = 8;

__global__ void __launch_bounds__(kTopkWarps * 32) prefill_topk_warp_kernel(const PsArgs a) {
  __shared__ uint32_t hist[kTopkWarps][256];
  const int lane = threadIdx.x & 31, wl = threadIdx.x >> 5;
  const int rs = blockIdx.x * kTopkWarps + wl;  // (i - row0) * Hkv + g
  const int i = a.row0 + rs / a.Hkv;
  if (i >= a.row1) return;
  const int nF = max(0, i + 1 - a.w);
  const int kk = min(a.k, nF);
  int32_t* out = a.idx + ((size_t)i * a.Hkv + rs % a.Hkv) * a.k;
  int32_t* cnt_out = a.cnt + (size_t)i * a.Hkv + rs % a.Hkv;
  if (kk == nF) {  // trivial rows: all of F
    if (lane == 0) *cnt_out = kk;
    for (int j = lane; j < a.k; j += 32) out[j] = j < kk ? j : -1;
    return;
  }
  const int c = min(a.cand_cnt[rs], a.cap);
  const uint32_t* keys = a.cand_key + (size_t)rs * a.cap;
  const int32_t* pos = a.cand_pos + (size_t)rs * a.cap;
  uint32_t* h = hist[wl];
  bool fail = c < kk;
  uint32_t prefix = 0, mask = 0;
  int remaining = kk;
  if (!fail) {
#pragma unroll 1
    for (int sh = 24; sh >= 0; sh -= 8) {
#pragma unroll
      for (int b = 0; b < 8; ++b) h[lane * 8 + b] = 0;
      __syncwarp();
      for (int j = lane; j < c; j += 32) {
        const uint32_t key = __ldcg(keys + j);
        if ((key & mask) == prefix) atomicAdd(&h[(key >> sh) & 255u], 1u);
      }
      __syncwarp();
      // lane L holds bins 255 - 8L .. 248 - 8L (descending); cumulative counts from the top
      uint32_t cnt8[8], own = 0;
#pragma unroll
      for (int b = 0; b < 8; ++b) {
        cnt8[b] = h[255 - 8 * lane - b];
        own += cnt8[b];
      }
      uint32_t incl = own;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
      }
      const uint32_t excl = incl - own;
      // the lane whose bins reach `remaining`: the first with incl >= remaining
      const unsigned hit = __ballot_sync(0xffffffffu, incl >= (uint32_t)remaining);
      const int src = __ffs(hit) - 1;  // exists: the total is >= remaining (c >= kk)
      int digit = 0, above = 0;
      if (lane == src) {
        uint32_t cum = excl;
#pragma unroll
        for (int b = 0; b < 8; ++b) {
          if (cum + cnt8[b] >= (uint32_t)remaining) {
            digit = 255 - 8 * lane - b;
            above = (int)cum;
            break;
          }
          cum += cnt8[b];
        }
      }
      digit = __shfl_sync(0xffffffffu, digit, src);
      above = __shfl_sync(0xffffffffu, above, src);
      remaining -= above;
      prefix |= (uint32_t)digit << sh;
      mask |= 255u << sh;
      __syncwarp();  // the bins are cleared again by the next pass
    }
    // a larger dropped key would belong in the answer (equal ones come later and lose)
    fail = a.cand_drop[rs] > prefix;
  }
  if (fail) {  // completed exactly by prefill_complete_kernel
    if (lane == 0) {
      *cnt_out = -1;
      a.redo_list[atomicAdd(a.redo_cnt, 1)] = rs;
    }
    for (int j = lane; j < a.k; j += 32) out[j] = -1;
    return;
  }
  const uint32_t T = prefix;  // the kk-th largest key; take the first `remaining` equal to it
  const unsigned lt = (1u << lane) - 1u;
  int o = 0, eq_seen = 0;
  for (int base = 0; base < c; base += 32) {
    const int j = base + lane;
    const uint32_t key = j < c ? __ldcg(keys + j) : 0u;
    const bool eq = j < c && key == T;
    const unsigned eqm = __ballot_sync(0xffffffffu, eq);
    const bool sel = j < c && (key > T || (eq && eq_seen + __popc(eqm & lt) < remaining));
    const unsigned selm = __ballot_sync(0xffffffffu, sel);
    if (sel) out[o + __popc(selm & lt)] = __ldcg(pos + j);
    o += __popc(selm);
    eq_seen += __popc(eqm);
  }
  if (lane == 0) *cnt_out = kk;
  for (int j = kk + lane; j < a.k; j += 32) out[j] = -1;
}

// prefill_complete_kernel (see the top of the file). A CTA takes listed rows in turn; its
// warps take 16-key chunks of the row's far range: lane (gid, tig) loads K rows gid and
// gid + 8 of the chunk as four 16-byte pieces at d = 32j + 8 tig (mma_attn.cuh's layout,
// the contraction index permuted identically for Q), S^T = K Q^T on mma.sync (8 heads per
// N tile, NT tiles), and the four lanes of a key sum its heads' exp2(x scale_log2 - lse2).
// Heads past G have zero queries and an infinite lse2, so they add nothing.
constexpr int kCompleteThreads = 256;

template <int NT>
__global__ void __launch_bounds__(kCompleteThreads) prefill_complete_kernel(const PsArgs a) {
  __shared__ TopkSmem<kCompleteThreads> tsm;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int gid = lane >> 2, tig = lane & 3;
  const int nredo = *(volatile int32_t*)a.redo_cnt;
  uint32_t* keys = a.redo_keys + (size_t)blockIdx.x * a.ld_redo;
  const __nv_bfloat16* qb16 = reinterpret_cast<const __nv_bfloat16*>(a.q);
  const __nv_bfloat16* kp = reinterpret_cast<const __nv_bfloat16*>(a.kpool);
  for (int f = blockIdx.x; f < nredo; f += gridDim.x) {
    const int rs = a.redo_list[f];
    const int i = a.row0 + rs / a.Hkv, g = rs % a.Hkv;
    const int nF = max(0, i + 1 - a.w);
    const int kk = min(a.k, nF);
    uint32_t qf[8][NT][2];
    float l2[NT][2];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const int hl = nt * 8 + gid;
      const bool hv = hl < a.G;
      const uint32_t* qrow = reinterpret_cast<const uint32_t*>(qb16 + ((size_t)i * a.Hq + g * a.G + (hv ? hl : 0)) * 128);
#pragma unroll
      for (int s = 0; s < 8; ++s) {
        const int base = 32 * (s >> 1) + 8 * tig + 4 * (s & 1);
        qf[s][nt][0] = hv ? __ldg(qrow + base / 2) : 0u;
        qf[s][nt][1] = hv ? __ldg(qrow + base / 2 + 1) : 0u;
      }
#pragma unroll
      for (int hs = 0; hs < 2; ++hs) {
        const int h = nt * 8 + 2 * tig + hs;
        l2[nt][hs] = h < a.G ? __ldg(a.lse2 + (size_t)i * a.Hq + g * a.G + h) : INFINITY;
      }
    }
    const int nchunks = (nF + 15) / 16;
    for (int c = warp; c < nchunks; c += kCompleteThreads / 32) {
      const int s0 = 16 * c;
      uint4 kr[2][4];
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        const int s = s0 + gid + 8 * half;
        int phys = -1;
        if (s < nF) {
          phys = a.bt[s / kPage];
          if (phys < 0 || phys >= a.num_pages) {
            flag_error(a.dev_err, HS2_DEV_BAD_PAGE);
            phys = -1;
          }
        }
        const uint4* row = reinterpret_cast<const uint4*>(kp + (((size_t)(phys < 0 ? 0 : phys) * a.Hkv + g) * kPage +
                                                                 s % kPage) * 128);
#pragma unroll
        for (int j = 0; j < 4; ++j) kr[half][j] = phys >= 0 ? __ldg(row + 4 * j + tig) : make_uint4(0, 0, 0, 0);
      }
      float pA = 0.f, pB = 0.f;
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
        for (int s = 0; s < 8; ++s) {
          const int j = s >> 1, u = s & 1;
          const uint32_t a0 = u ? kr[0][j].z : kr[0][j].x, a2 = u ? kr[0][j].w : kr[0][j].y;
          const uint32_t a1 = u ? kr[1][j].z : kr[1][j].x, a3 = u ? kr[1][j].w : kr[1][j].y;
          mma_bf16_16816(acc[u], a0, a1, a2, a3, qf[s][nt][0], qf[s][nt][1]);
        }
        pA += tc::ex2(fmaf(acc[0][0] + acc[1][0], a.scale_log2, -l2[nt][0])) +
              tc::ex2(fmaf(acc[0][1] + acc[1][1], a.scale_log2, -l2[nt][1]));
        pB += tc::ex2(fmaf(acc[0][2] + acc[1][2], a.scale_log2, -l2[nt][0])) +
              tc::ex2(fmaf(acc[0][3] + acc[1][3], a.scale_log2, -l2[nt][1]));
      }
      pA += __shfl_xor_sync(0xffffffffu, pA, 1);
      pA += __shfl_xor_sync(0xffffffffu, pA, 2);
      pB += __shfl_xor_sync(0xffffffffu, pB, 1);
      pB += __shfl_xor_sync(0xffffffffu, pB, 2);
      if (tig == 0) {
        if (s0 + gid < nF) keys[s0 + gid] = __float_as_uint(pA);
        if (s0 + gid + 8 < nF) keys[s0 + gid + 8] = __float_as_uint(pB);
      }
    }
    __syncthreads();  // the key row is complete (global writes visible to the block)
    int32_t* out = a.idx + ((size_t)i * a.Hkv + g) * a.k;
    block_topk<kCompleteThreads>(
        nF, kk, [&](int s) { return __ldcg(keys + s); }, [&](int j, int s) { out[j] = s; }, tsm);
    if (threadIdx.x == 0) a.cnt[(size_t)i * a.Hkv + g] = kk;
    __syncthreads();  // the next listed row overwrites the key row
  }
}

size_t prefill_scan_smem() { return sizeof(PsSmem) + 1024; }

cudaError_t launch_prefill_select(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tks,
                                  const PsArgs& a, cudaStream_t s) {
  const size_t sm = prefill_scan_smem();
  cudaError_t e = cudaFuncSetAttribute(prefill_scan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
  if (e != cudaSuccess) return e;
  const int tiles = (a.row1 - a.row0 + kST - 1) / kST;
  prefill_scan_kernel<<<dim3(tiles, a.Hkv), kSThreads, sm, s>>>(tq, tk, tks, a);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int rows = (a.row1 - a.row0) * a.Hkv;
  prefill_topk_warp_kernel<<<(rows + kTopkWarps - 1) / kTopkWarps, kTopkWarps * 32, 0, s>>>(a);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int grid = std::min(rows, kPsCompleteCtas);
  if (a.G <= 8) prefill_complete_kernel<1><<<grid, kCompleteThreads, 0, s>>>(a);
  else if (a.G <= 16) prefill_complete_kernel<2><<<grid, kCompleteThreads, 0, s>>>(a);
  else if (a.G <= 32) prefill_complete_kernel<4><<<grid, kCompleteThreads, 0, s>>>(a);
  else return cudaErrorInvalidValue;
  return cudaGetLastError();
}

}  // namespace hs2

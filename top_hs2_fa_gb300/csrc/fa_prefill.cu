// fa_prefill.cu — causal FA forward for bf16 prefill on tcgen05 (O and lse per row).
//
// The FA layer of a HySparse2 Cross group attends causally to every earlier key of the
// group's shared KV ("HySparse2：整体架构、KV 生命周期与 PD 分离", §5, §8.1: during prefill
// the FA builds the cache and attends over all positions). Row i sees keys [0, i].
//
// One CTA per (128-row query tile, query head); heaviest tiles are scheduled first.
//   warps 0, 10 TMA producers: Q tile once (3-D map over [n][Hq][d]); K tiles (warp 0) and
//               V tiles (warp 10) of 128 keys (two 64-row pages each, through the block
//               table) into kKV-slot rings, 128-byte swizzle; a K slot frees when its QK
//               is done, a V slot when its PV is done.
//   warp 1      MMA issuer: S_j = Q K_j^T into one of two TMEM buffers (M=128, N=128,
//               K=128), then O += P_j V_j (A = P from tensor memory, B = V MN-major);
//               S_{j+1} is issued before waiting for P_j so the tensor core stays busy.
//   warps 2-9   softmax, two threads per query row (warps w and w+4 share a TMEM lane
//               quadrant, each takes 64 of the tile's 128 columns; the halves swap their
//               row maxima through shared memory): row max, exp2 (base-2 logits), P in
//               bf16 written back over the tile's own S buffer, and a lazy O rescale: the
//               reference max only moves when the row max grows by more than 2^8, which
//               keeps every weight below 256 and needs no approximation; only a rescale
//               waits for the previous PV. The normaliser is not summed here: every V slot
//               carries a third 64-column block of ones, the P.V MMA runs with N = 144, and
//               O's column 128 accumulates the sum of the same bf16 weights on the tensor
//               core.
//   warp 10     TMA producer of the V tiles.
// TMEM: S0 columns [0,128), S1 [128,256), O [256,400) (d, then the normaliser's 16
// columns, 128-143, all equal); P_j occupies the first 64 columns
// of S_j's buffer (two bf16 per column), so it never passes through shared memory. A
// buffer is rewritten by S_{j+2} only after PV_j has read P_j: one thread issues both in
// that order and the tensor pipe executes one thread's MMAs in order. Every mbarrier wait
// is bounded.
#include <cuda.h>

#include "common.cuh"
#include "kernels.h"
#include "tc.cuh"

namespace hs2 {

namespace {

constexpr int kPT = 128;           // query rows per tile = keys per KV tile
constexpr int kPThreads = 352;     // TMA warps (Q and K; V), MMA warp, 8 softmax warps
constexpr int kVWarp = 10;         // the V producer
constexpr uint32_t kTileBytes = kPT * 128 * 2;  // 32 KB: 128 rows x 128 bf16
constexpr uint32_t kVSlotBytes = kTileBytes + 16384;  // a V tile and its block of ones
constexpr int kPVN = 144;          // P.V width: 128 d columns and 16 of the normaliser
constexpr uint32_t kTmemColsPf = 512;
constexpr float kRescaleLog2 = 8.f;
constexpr int kKV = 2;             // K slots and V slots (tile j in slot j % kKV)

struct PfSmem {
  uint8_t q[kTileBytes];      // A of S: K-blocks (d 0-63, d 64-127) x [128 rows x 128 B]
  uint8_t k[kKV][kTileBytes];  // B of S: same layout, rows = keys
  uint8_t v[kKV][kVSlotBytes];  // B of PV (MN-major): d-halves then ones x [128 keys x 128 B]
  float xch[2][kPT];           // [half] a tile's row maxima of the two column halves (then
                               // the row normaliser's halves, at the end)
  uint64_t q_full, k_full[kKV], k_empty[kKV], v_full[kKV], v_empty[kKV], s_full[2], p_full[2], p_empty[2];
  uint64_t x_full[4], x_empty[4];  // per lane quadrant: both halves wrote / read xch
  uint32_t tmem_base;
  int abort;
};

HS2_DEVI bool aborted(PfSmem& sm) { return *(volatile int*)&sm.abort != 0; }
HS2_DEVI void set_abort(PfSmem& sm, int32_t* dev_err) {
  flag_error(dev_err, HS2_DEV_TIMEOUT);
  atomicExch(&sm.abort, 1);
}

}  // namespace

__global__ void __launch_bounds__(kPThreads, 1)
    fa_prefill_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                          const __grid_constant__ CUtensorMap tm_v, const PfArgs a) {
  extern __shared__ __align__(1024) uint8_t dsmem[];
  PfSmem& sm = *reinterpret_cast<PfSmem*>(dsmem + ((1024 - (tc::smem_u32(dsmem) & 1023)) & 1023));
  const int n_tiles = (a.n + kPT - 1) / kPT;
  const int tile_m = n_tiles - 1 - blockIdx.x;  // heaviest (longest causal range) first
  const int h = blockIdx.y, g = h / a.G;
  const int i0 = tile_m * kPT;
  const int J = tile_m + 1;  // key tiles [0, J)
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = a.seq_len[0];
  const int npages = (t + kPage - 1) / kPage;
  if (t < a.n || npages > a.max_pages) {
    if (threadIdx.x == 0 && blockIdx.x == 0 && blockIdx.y == 0) flag_error(a.dev_err, HS2_DEV_BAD_LENGTH);
    return;
  }
  if (threadIdx.x == 0) {
    tc::mbar_init(&sm.q_full, 1);
    for (int s = 0; s < kKV; ++s) {
      tc::mbar_init(&sm.k_full[s], 1);
      tc::mbar_init(&sm.k_empty[s], 1);  // QK of the slot's tile done
      tc::mbar_init(&sm.v_full[s], 1);
      tc::mbar_init(&sm.v_empty[s], 1);  // PV of the slot's tile done
    }
    for (int s = 0; s < 2; ++s) {
      tc::mbar_init(&sm.s_full[s], 1);
      tc::mbar_init(&sm.p_full[s], 256);  // every softmax thread wrote its part of P into TMEM
      tc::mbar_init(&sm.p_empty[s], 1);   // PV of the buffer's tile done (and every MMA before it)
    }
    for (int q = 0; q < 4; ++q) {
      tc::mbar_init(&sm.x_full[q], 64);
      tc::mbar_init(&sm.x_empty[q], 64);
    }
    sm.abort = 0;
    tc::fence_mbar_init();
  }
  // the V slots' third 64-column block: all ones (bf16), written once; the TMA loads fill
  // only the first two
  for (int e = threadIdx.x; e < kKV * 1024; e += kPThreads)
    *reinterpret_cast<uint4*>(sm.v[e >> 10] + kTileBytes + 16 * (e & 1023)) =
        make_uint4(0x3F803F80u, 0x3F803F80u, 0x3F803F80u, 0x3F803F80u);
  tc::fence_async_smem();  // visible to the tensor core's reads
  if (warp == 1) tc::tmem_alloc(&sm.tmem_base, kTmemColsPf);
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = sm.tmem_base;
  const uint32_t tS = tmem, tO = tmem + 256;

  if (warp == 0 || warp == kVWarp) {
    // ------------------------------------------------------------------ TMA producers
    // warp 0: Q once, then K tiles; warp 6: V tiles. K slots free up when a tile's QK is
    // done and V slots when its PV is done, so the K loads run ahead of the V loads.
    if (lane == 0) {
      const bool is_k = warp == 0;
      const int32_t* bt = a.bt;
      if (is_k) {
        tc::mbar_arrive_expect_tx(&sm.q_full, kTileBytes);
        tc::tma_load_3d(sm.q, &tm_q, 0, h, i0, &sm.q_full);
        tc::tma_load_3d(sm.q + kTileBytes / 2, &tm_q, 64, h, i0, &sm.q_full);
      }
      uint64_t* full = is_k ? sm.k_full : sm.v_full;
      uint64_t* empty = is_k ? sm.k_empty : sm.v_empty;
      const CUtensorMap* tm = is_k ? &tm_k : &tm_v;
      int issued = 0;
      for (int j = 0; j < J && !aborted(sm); ++j) {
        const int st = j % kKV;
        if (!tc::mbar_wait(&empty[st], ((j / kKV) & 1) ^ 1)) {
          set_abort(sm, a.dev_err);
          break;
        }
        // a page past the sequence (or a bad table entry, flagged) is loaded from the row just
        // past the pool, which the TMA fills with zeros: the slot never keeps stale or
        // uninitialised rows (a NaN among V's rows would reach every row through P.V, even
        // with its weight 0)
        const int oob = a.num_pages * a.Hkv * kPage;
        int rows[2];
        for (int pg = 0; pg < 2; ++pg) {
          const int lp = 2 * j + pg;
          rows[pg] = oob;
          if (lp < npages) {
            const int phys = bt[lp];
            if (phys < 0 || phys >= a.num_pages) flag_error(a.dev_err, HS2_DEV_BAD_PAGE);
            else rows[pg] = (phys * a.Hkv + g) * kPage;
          }
        }
        tc::mbar_arrive_expect_tx(&full[st], 4 * 8192);
        uint8_t* dst = is_k ? sm.k[st] : sm.v[st];
        for (int pg = 0; pg < 2; ++pg)
          for (int hh = 0; hh < 2; ++hh) tc::tma_load_2d(dst + hh * 16384 + pg * 8192, tm, 64 * hh, rows[pg], &full[st]);
        issued = j + 1;
      }
      for (int j = max(0, issued - kKV); j < issued; ++j) (void)tc::mbar_wait(&full[j % kKV], (j / kKV) & 1);
      if (is_k) (void)tc::mbar_wait(&sm.q_full, 0);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idS = tc::idesc_bf16_f32(kPT, kPT);
      constexpr uint32_t idO = tc::idesc_bf16_f32_bmn(kPT, kPVN);
      const uint32_t qb = tc::smem_u32(sm.q);
      int pv_issued = 0;
      // S_j's buffer held P_{j-2}, read by PV_{j-2}, which this thread issued before S_j
      auto issue_s = [&](int j) -> bool {
        const int st = j & 1, kv = j % kKV;
        if (!tc::mbar_wait(&sm.k_full[kv], (j / kKV) & 1)) return false;
        tc::tc_fence_after();
        const uint32_t kb = tc::smem_u32(sm.k[kv]);
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
          const uint32_t off = (ks >> 2) * 16384u + (ks & 3) * 32u;
          tc::mma_bf16(tS + st * 128, tc::sdesc_sw128(qb + off), tc::sdesc_sw128(kb + off), idS, ks > 0 ? 1u : 0u);
        }
        tc::mma_commit(&sm.s_full[st]);
        tc::mma_commit(&sm.k_empty[kv]);
        return true;
      };
      bool ok = tc::mbar_wait(&sm.q_full, 0) && issue_s(0);
      for (int j = 0; ok && j < J; ++j) {
        if (j + 1 < J && !issue_s(j + 1)) { ok = false; break; }
        const int st = j & 1, kv = j % kKV;
        if (!tc::mbar_wait(&sm.p_full[st], (j >> 1) & 1) || !tc::mbar_wait(&sm.v_full[kv], (j / kKV) & 1)) {
          ok = false;
          break;
        }
        tc::tc_fence_after();
        const uint32_t vb = tc::smem_u32(sm.v[kv]);
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {  // keys 16 ks .. 16 ks + 15 of P_j: columns 8 ks .. 8 ks + 7
          const uint64_t bd = tc::sdesc_sw128_mn(vb + ks * 2048u, 16384u, 1024u);
          tc::mma_bf16_ts(tO, tS + st * 128 + ks * 8, bd, idO, (j > 0 || ks > 0) ? 1u : 0u);
        }
        tc::mma_commit(&sm.v_empty[kv]);
        tc::mma_commit(&sm.p_empty[st]);
        pv_issued = j + 1;
      }
      if (!ok) set_abort(sm, a.dev_err);
      if (pv_issued > 0) (void)tc::mbar_wait(&sm.p_empty[(pv_issued - 1) & 1], ((pv_issued - 1) >> 1) & 1);
    }
  } else {
    // ------------------------------------------------------------------ softmax warps
    const int qd = warp & 3;
    const int half = (warp - 2) >> 2;  // columns [64 half, 64 half + 64) of every tile
    const int r = qd * 32 + lane;
    const int i = i0 + r;
    const uint32_t lane_off = (uint32_t)(qd * 32) << 16;
    float m_used = -INFINITY;
    // hand a value to the other half of the row through xch (round x: bounded mbarrier
    // waits, so a half that stopped cannot leave the other waiting for ever)
    auto swap = [&](float v, int x, float& other) -> bool {
      if (x > 0 && !__all_sync(0xffffffffu, tc::mbar_wait(&sm.x_empty[qd], (x - 1) & 1))) return false;
      sm.xch[half][r] = v;
      tc::mbar_arrive(&sm.x_full[qd]);
      if (!__all_sync(0xffffffffu, tc::mbar_wait(&sm.x_full[qd], x & 1))) return false;
      other = sm.xch[half ^ 1][r];
      tc::mbar_arrive(&sm.x_empty[qd]);
      return true;
    };
    bool ok = true;
    for (int j = 0; j < J; ++j) {
      const int sb = j & 1;
      // votes keep the warp converged for the warp-collective TMEM accesses
      if (!__all_sync(0xffffffffu, !aborted(sm) && tc::mbar_wait(&sm.s_full[sb], (j >> 1) & 1))) { ok = false; break; }
      tc::tc_fence_after();
      float x[2][32];
      {
        uint32_t raw[2][32];
#pragma unroll
        for (int c = 0; c < 2; ++c) tc::tmem_ld32_async(tS + lane_off + sb * 128 + half * 64 + c * 32, raw[c]);
        tc::tmem_wait_ld(raw[1]);
        tc::tmem_regs_ready(raw[0]);
#pragma unroll
        for (int c = 0; c < 2; ++c)
#pragma unroll
          for (int e = 0; e < 32; ++e) x[c][e] = __uint_as_float(raw[c][e]);
      }
      // raw logits: only the diagonal tile crosses the causal boundary; the scale (> 0) is
      // applied to the max and folded into the exponent's FMA below
      if (j == J - 1) {
        const int kbase = j * kPT + half * 64;
#pragma unroll
        for (int c = 0; c < 2; ++c)
#pragma unroll
          for (int e = 0; e < 32; ++e)
            if (kbase + c * 32 + e > i) x[c][e] = -INFINITY;
      }
      float mt = -INFINITY;
#pragma unroll
      for (int c = 0; c < 2; ++c)
#pragma unroll
        for (int e = 0; e < 32; ++e) mt = fmaxf(mt, x[c][e]);
      // the row max over both halves
      float mo;
      if (!swap(mt, j, mo)) {
        ok = false;
        break;
      }
      mt = fmaxf(mt, mo);
      const float m_new = fmaxf(m_used, mt * a.scale_log2);
      const bool need = m_new > m_used + kRescaleLog2 || (m_used == -INFINITY && m_new > -INFINITY);
      const float alpha = (need && m_used > -INFINITY) ? tc::ex2(m_used - m_new) : 1.f;
      if (need) m_used = m_new;
      if (j > 0) {
        if (__any_sync(0xffffffffu, alpha != 1.f)) {
          // O holds every earlier tile once PV_{j-1} is done
          if (!__all_sync(0xffffffffu, tc::mbar_wait(&sm.p_empty[(j - 1) & 1], ((j - 1) >> 1) & 1))) {
            ok = false;
            break;
          }
          tc::tc_fence_after();
          // this half's 64 d columns; half 0 also the normaliser's block (128 onwards)
#pragma unroll 1
          for (int c = 0; c < 2 + (half == 0); ++c) {
            float ov[32];
            const uint32_t col = c < 2 ? half * 64 + c * 32 : 128;
            tc::tmem_ld32(tO + lane_off + col, ov);
#pragma unroll
            for (int e = 0; e < 32; ++e) ov[e] *= alpha;
            tc::tmem_st32(tO + lane_off + col, ov);
          }
        }
      }
      // P row (bf16) back into tensor memory over S_j: this half's keys 64 half + 2c, +1 go to
      // column 32 half + c of the buffer (the other half read its S columns before the max
      // exchange above). p = 2^(x*s - m): one FMA and ex2 (which maps -inf to +0).
      const float neg_m = -m_used;
      uint32_t w[32];
#pragma unroll
      for (int c = 0; c < 32; ++c) {
        const float p0 = tc::ex2(fmaf(x[c >> 4][(2 * c) & 31], a.scale_log2, neg_m));
        const float p1 = tc::ex2(fmaf(x[c >> 4][(2 * c + 1) & 31], a.scale_log2, neg_m));
        w[c] = pack_bf16(p0, p1);
      }
      tc::tmem_st32u(tS + lane_off + sb * 128 + half * 32, w);
      tc::tc_fence_before();
      tc::mbar_arrive(&sm.p_full[sb]);
    }
    if (__all_sync(0xffffffffu, ok && !aborted(sm) && tc::mbar_wait(&sm.p_empty[(J - 1) & 1], ((J - 1) >> 1) & 1))) {
      tc::tc_fence_after();
      float lv[32];
      tc::tmem_ld32(tO + lane_off + 128, lv);  // the row's normaliser (both halves' weights)
      const float l = lv[0];
      const float linv = l > 0.f ? 1.f / l : 0.f;
      float* orow = a.o + ((size_t)i * a.Hq + h) * 128 + half * 64;
#pragma unroll 1
      for (int c = 0; c < 2; ++c) {
        float ov[32];
        tc::tmem_ld32(tO + lane_off + half * 64 + c * 32, ov);
        if (i < a.n) {
#pragma unroll
          for (int e = 0; e < 32; e += 4)
            *reinterpret_cast<float4*>(orow + c * 32 + e) =
                make_float4(ov[e] * linv, ov[e + 1] * linv, ov[e + 2] * linv, ov[e + 3] * linv);
        }
      }
      if (i < a.n && half == 0) {
        a.lse2[(size_t)i * a.Hq + h] = m_used + log2f(l);
        if (a.lse) a.lse[(size_t)i * a.Hq + h] = (m_used + log2f(l)) / kLog2e;
      }
    } else if (!aborted(sm)) {
      set_abort(sm, a.dev_err);
    }
  }
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 1) tc::tmem_dealloc(tmem, kTmemColsPf);
}

size_t fa_prefill_fwd_smem() { return sizeof(PfSmem) + 1024; }

cudaError_t launch_fa_prefill_fwd(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const PfArgs& a,
                                  cudaStream_t s) {
  const size_t sm = fa_prefill_fwd_smem();
  cudaError_t e = cudaFuncSetAttribute(fa_prefill_fwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
  if (e != cudaSuccess) return e;
  const int n_tiles = (a.n + kPT - 1) / kPT;
  fa_prefill_fwd_kernel<<<dim3(n_tiles, a.Hq), kPThreads, sm, s>>>(tq, tk, tv, a);
  return cudaGetLastError();
}

}  // namespace hs2

// fa_prefill.cu — causal FA forward for bf16 prefill on tcgen05 (O and lse per row).
//
// The FA layer of a HySparse2 Cross group attends causally to every earlier key of the
// group's shared KV ("HySparse2：整体架构、KV 生命周期与 PD 分离", §5, §8.1: during prefill
// the FA builds the cache and attends over all positions). Row i sees keys [0, i].
//
// One CTA per (128-row query tile, query head); heaviest tiles are scheduled first.
//   warp 0      TMA producer: Q tile once (3-D map over [n][Hq][d]); K and V tiles of
//               128 keys (two 64-row pages each, through the block table) into a 2-stage
//               ring, 128-byte swizzle.
//   warp 1      MMA issuer: S_j = Q K_j^T into one of two TMEM buffers (M=128, N=128,
//               K=128), then O += P_j V_j (A = P from shared memory, B = V MN-major);
//               S_{j+1} is issued before waiting for P_j so the tensor core stays busy.
//   warps 2-5   softmax, one query row per thread: row max, exp2 (base-2 logits), P in
//               bf16 to shared memory (the normaliser sums the same rounded values), and a
//               lazy O rescale: the reference max only moves when the row max grows by more
//               than 2^8, which keeps every weight below 256 and needs no approximation.
// TMEM: S0 columns [0,128), S1 [128,256), O [256,384). Every mbarrier wait is bounded.
#include <cuda.h>

#include "common.cuh"
#include "kernels.h"
#include "tc.cuh"

namespace hs2 {

namespace {

constexpr int kPT = 128;           // query rows per tile = keys per KV tile
constexpr int kPThreads = 192;     // TMA warp, MMA warp, 4 softmax warps
constexpr uint32_t kTileBytes = kPT * 128 * 2;  // 32 KB: 128 rows x 128 bf16
constexpr uint32_t kTmemColsPf = 512;
constexpr float kRescaleLog2 = 8.f;

struct PfSmem {
  uint8_t q[kTileBytes];      // A of S: K-blocks (d 0-63, d 64-127) x [128 rows x 128 B]
  uint8_t k[2][kTileBytes];   // B of S: same layout, rows = keys
  uint8_t v[2][kTileBytes];   // B of PV (MN-major): d-halves x [128 keys x 128 B]
  uint8_t p[kTileBytes];      // A of PV: K-blocks (keys 0-63, 64-127) x [128 rows x 128 B]
  uint64_t q_full, kv_full[2], kv_empty[2], s_full[2], s_empty[2], p_full, o_done;
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
    for (int s = 0; s < 2; ++s) {
      tc::mbar_init(&sm.kv_full[s], 1);
      tc::mbar_init(&sm.kv_empty[s], 1);
      tc::mbar_init(&sm.s_full[s], 1);
      tc::mbar_init(&sm.s_empty[s], 128);
    }
    tc::mbar_init(&sm.p_full, 128);
    tc::mbar_init(&sm.o_done, 1);
    sm.abort = 0;
    tc::fence_mbar_init();
  }
  if (warp == 1) tc::tmem_alloc(&sm.tmem_base, kTmemColsPf);
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = sm.tmem_base;
  const uint32_t tS = tmem, tO = tmem + 256;

  if (warp == 0) {
    // ------------------------------------------------------------------ TMA producer
    if (lane == 0) {
      const int32_t* bt = a.bt;
      tc::mbar_arrive_expect_tx(&sm.q_full, kTileBytes);
      tc::tma_load_3d(sm.q, &tm_q, 0, h, i0, &sm.q_full);
      tc::tma_load_3d(sm.q + kTileBytes / 2, &tm_q, 64, h, i0, &sm.q_full);
      int issued = 0;
      for (int j = 0; j < J && !aborted(sm); ++j) {
        const int st = j & 1;
        if (!tc::mbar_wait(&sm.kv_empty[st], ((j >> 1) & 1) ^ 1)) {
          set_abort(sm, a.dev_err);
          break;
        }
        int rows[2];
        uint32_t bytes = 0;
        for (int pg = 0; pg < 2; ++pg) {
          const int lp = 2 * j + pg;
          rows[pg] = -1;
          if (lp < npages) {
            const int phys = bt[lp];
            if (phys < 0 || phys >= a.num_pages) flag_error(a.dev_err, HS2_DEV_BAD_PAGE);
            else { rows[pg] = (phys * a.Hkv + g) * kPage; bytes += 4 * 8192; }
          }
        }
        tc::mbar_arrive_expect_tx(&sm.kv_full[st], bytes);
        for (int pg = 0; pg < 2; ++pg) {
          if (rows[pg] < 0) continue;
          for (int hh = 0; hh < 2; ++hh) {
            tc::tma_load_2d(sm.k[st] + hh * 16384 + pg * 8192, &tm_k, 64 * hh, rows[pg], &sm.kv_full[st]);
            tc::tma_load_2d(sm.v[st] + hh * 16384 + pg * 8192, &tm_v, 64 * hh, rows[pg], &sm.kv_full[st]);
          }
        }
        issued = j + 1;
      }
      for (int j = max(0, issued - 2); j < issued; ++j) (void)tc::mbar_wait(&sm.kv_full[j & 1], (j >> 1) & 1);
      (void)tc::mbar_wait(&sm.q_full, 0);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idS = tc::idesc_bf16_f32(kPT, kPT);
      constexpr uint32_t idO = tc::idesc_bf16_f32_bmn(kPT, 128);
      const uint32_t qb = tc::smem_u32(sm.q), pb = tc::smem_u32(sm.p);
      int pv_issued = 0;
      auto issue_s = [&](int j) -> bool {
        const int st = j & 1;
        if (!tc::mbar_wait(&sm.kv_full[st], (j >> 1) & 1) || !tc::mbar_wait(&sm.s_empty[st], ((j >> 1) & 1) ^ 1))
          return false;
        tc::tc_fence_after();
        const uint32_t kb = tc::smem_u32(sm.k[st]);
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
          const uint32_t off = (ks >> 2) * 16384u + (ks & 3) * 32u;
          tc::mma_bf16(tS + st * 128, tc::sdesc_sw128(qb + off), tc::sdesc_sw128(kb + off), idS, ks > 0 ? 1u : 0u);
        }
        tc::mma_commit(&sm.s_full[st]);
        return true;
      };
      bool ok = tc::mbar_wait(&sm.q_full, 0) && issue_s(0);
      for (int j = 0; ok && j < J; ++j) {
        if (j + 1 < J && !issue_s(j + 1)) { ok = false; break; }
        if (!tc::mbar_wait(&sm.p_full, j & 1)) { ok = false; break; }
        tc::tc_fence_after();
        const int st = j & 1;
        const uint32_t vb = tc::smem_u32(sm.v[st]);
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
          const uint64_t ad = tc::sdesc_sw128(pb + (ks >> 2) * 16384u + (ks & 3) * 32u);
          const uint64_t bd = tc::sdesc_sw128_mn(vb + ks * 2048u, 16384u, 1024u);
          tc::mma_bf16(tO, ad, bd, idO, (j > 0 || ks > 0) ? 1u : 0u);
        }
        tc::mma_commit(&sm.kv_empty[st]);
        tc::mma_commit(&sm.o_done);
        pv_issued = j + 1;
      }
      if (!ok) set_abort(sm, a.dev_err);
      if (pv_issued > 0) (void)tc::mbar_wait(&sm.o_done, (pv_issued - 1) & 1);
    }
  } else {
    // ------------------------------------------------------------------ softmax warps
    const int qd = warp & 3;
    const int r = qd * 32 + lane;
    const int i = i0 + r;
    const uint32_t lane_off = (uint32_t)(qd * 32) << 16;
    float m_used = -INFINITY, l = 0.f;
    bool ok = true;
    for (int j = 0; j < J; ++j) {
      const int sb = j & 1;
      // votes keep the warp converged for the warp-collective TMEM accesses
      if (!__all_sync(0xffffffffu, !aborted(sm) && tc::mbar_wait(&sm.s_full[sb], (j >> 1) & 1))) { ok = false; break; }
      tc::tc_fence_after();
      float x[4][32];
      {
        uint32_t raw[4][32];
#pragma unroll
        for (int c = 0; c < 4; ++c) tc::tmem_ld32_async(tS + lane_off + sb * 128 + c * 32, raw[c]);
        tc::tmem_wait_ld(raw[3]);
        tc::tmem_regs_ready(raw[0]);
        tc::tmem_regs_ready(raw[1]);
        tc::tmem_regs_ready(raw[2]);
#pragma unroll
        for (int c = 0; c < 4; ++c)
#pragma unroll
          for (int e = 0; e < 32; ++e) x[c][e] = __uint_as_float(raw[c][e]);
      }
      tc::tc_fence_before();
      tc::mbar_arrive(&sm.s_empty[sb]);
      const int kbase = j * kPT;
      float mt = -INFINITY;
#pragma unroll
      for (int c = 0; c < 4; ++c)
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          const int key = kbase + c * 32 + e;
          x[c][e] = key <= i ? x[c][e] * a.scale_log2 : -INFINITY;
          mt = fmaxf(mt, x[c][e]);
        }
      const float m_new = fmaxf(m_used, mt);
      const bool need = m_new > m_used + kRescaleLog2 || (m_used == -INFINITY && m_new > -INFINITY);
      const float alpha = (need && m_used > -INFINITY) ? tc::ex2(m_used - m_new) : 1.f;
      if (need) m_used = m_new;
      if (j > 0) {
        // P_{j-1} has been consumed and O holds every earlier tile once PV_{j-1} is done
        if (!__all_sync(0xffffffffu, tc::mbar_wait(&sm.o_done, (j - 1) & 1))) { ok = false; break; }
        tc::tc_fence_after();
        if (__any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll 1
          for (int c = 0; c < 4; ++c) {
            float ov[32];
            tc::tmem_ld32(tO + lane_off + c * 32, ov);
#pragma unroll
            for (int e = 0; e < 32; ++e) ov[e] *= alpha;
            tc::tmem_st32(tO + lane_off + c * 32, ov);
          }
        }
        l *= alpha;
      }
      // P row (bf16) into shared memory, 128-byte swizzled K-major layout
      uint8_t* prow = sm.p + (r >> 3) * 1024 + (r & 7) * 128;
#pragma unroll
      for (int cc = 0; cc < 16; ++cc) {
        uint32_t w[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const float p0 = x[cc >> 2][(cc & 3) * 8 + 2 * u] == -INFINITY ? 0.f : tc::ex2(x[cc >> 2][(cc & 3) * 8 + 2 * u] - m_used);
          const float p1 = x[cc >> 2][(cc & 3) * 8 + 2 * u + 1] == -INFINITY ? 0.f : tc::ex2(x[cc >> 2][(cc & 3) * 8 + 2 * u + 1] - m_used);
          w[u] = pack_bf16(p0, p1);
          l += bf16_lo(w[u]) + bf16_hi(w[u]);
        }
        *reinterpret_cast<uint4*>(prow + (cc >> 3) * 16384 + (((cc & 7) ^ (r & 7)) << 4)) = make_uint4(w[0], w[1], w[2], w[3]);
      }
      tc::fence_async_smem();
      tc::mbar_arrive(&sm.p_full);
    }
    if (__all_sync(0xffffffffu, ok && !aborted(sm) && tc::mbar_wait(&sm.o_done, (J - 1) & 1))) {
      tc::tc_fence_after();
      const float linv = l > 0.f ? 1.f / l : 0.f;
      float* orow = a.o + ((size_t)i * a.Hq + h) * 128;
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        float ov[32];
        tc::tmem_ld32(tO + lane_off + c * 32, ov);
        if (i < a.n) {
#pragma unroll
          for (int e = 0; e < 32; e += 4)
            *reinterpret_cast<float4*>(orow + c * 32 + e) =
                make_float4(ov[e] * linv, ov[e + 1] * linv, ov[e + 2] * linv, ov[e + 3] * linv);
        }
      }
      if (i < a.n) {
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

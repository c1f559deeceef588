// staged_attn.cuh — one warp's online-softmax attention over 16 staged entries at a time,
// from shared memory in the 128-byte swizzle layout, on mma.sync (bf16 in, fp32 accumulate).
#pragma once
#include "common.cuh"

namespace hs2 {

HS2_DEVI void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
HS2_DEVI void ldsm_x4_t(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

// Byte offset of (row, 16-byte chunk) inside a 1024-byte aligned block of 128-byte rows in
// the 128-byte swizzle layout: the chunk index is XORed with row % 8, so the eight rows of
// an 8x8 ldmatrix tile fall in distinct banks.
HS2_DEVI uint32_t sw128(int row, int chunk) { return (uint32_t)(row * 128 + ((chunk ^ (row & 7)) << 4)); }

// One warp's online-softmax attention state for the 8*NT query heads of a KV head, fed
// 16 entries at a time from a staged slot. Slot layout (D/64 halves of 64 columns):
//   K half h at h*2048, V half h at (D/64)*2048 + h*2048; 16 rows of 128 bytes each.
// Register mappings (m16n8k16, gid = lane/4, tig = lane%4):
//   S^T[16 entries x 8 heads] = K[16 x 16 d] Q^T[16 d x 8 heads], k-step s covers d 16s..16s+15
//   O^T[16 d x 8 heads] += V^T[16 d x 16 entries] P^T[16 entries x 8 heads];
//   acc[mt][nt][0..1]: d = 16mt + gid, heads nt*8 + 2tig, +1; acc[mt][nt][2..3]: d + 8.
// F16 = true (an FP8 cache converted to f16 when staged): queries become f16 at init, both
// contractions use the f16 MMA, entries carry their own K scale (on the logits) and V scale
// (on the weights entering P.V), and the normaliser sums the unscaled weights. acc is kept
// in units of vu, the largest |V scale| seen so far, so each weight enters P.V as
// f16(p * vs / vu) in [-1, 1]: tiny V scales do not fall into the f16 subnormal range.
// The true P.V is acc * unit().
template <int D, int NT, bool F16 = false>
struct StagedAttn {
  static constexpr int KS = D / 16;
  static constexpr int HALVES = D / 64;
  uint32_t qb[KS][NT][2];
  float m[NT][2], l[NT][2];
  float acc[KS][NT][4];
  float vu, vinv;  // F16: the unit of acc (0 until a nonzero V scale is seen) and 1 / vu (or 0)

  HS2_DEVI float unit() const { return F16 ? vu : 1.f; }

  HS2_DEVI void init(const __nv_bfloat16* q_heads, int G) {
    const int lane = threadIdx.x & 31, gid = lane >> 2, tig = lane & 3;
    vu = vinv = 0.f;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const int hl = nt * 8 + gid;
      const bool hv = hl < G;
      const uint32_t* qrow = reinterpret_cast<const uint32_t*>(q_heads + (size_t)(hv ? hl : 0) * D);
#pragma unroll
      for (int s = 0; s < KS; ++s) {
        qb[s][nt][0] = hv ? qrow[8 * s + tig] : 0u;
        qb[s][nt][1] = hv ? qrow[8 * s + 4 + tig] : 0u;
        if (F16) {
          qb[s][nt][0] = bf16x2_to_f16x2(qb[s][nt][0]);
          qb[s][nt][1] = bf16x2_to_f16x2(qb[s][nt][1]);
        }
      }
      m[nt][0] = m[nt][1] = -INFINITY;
      l[nt][0] = l[nt][1] = 0.f;
#pragma unroll
      for (int mt = 0; mt < KS; ++mt) acc[mt][nt][0] = acc[mt][nt][1] = acc[mt][nt][2] = acc[mt][nt][3] = 0.f;
    }
  }

  // slot: shared address of the staged entries; okA / okB: entries gid / gid+8 are valid.
  // Invalid entries must be staged as zero rows (their weight is zero, and so is V).
  HS2_DEVI static void mma(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                           uint32_t b1) {
    if (F16) mma_f16_16816(c, a0, a1, a2, a3, b0, b1);
    else mma_bf16_16816(c, a0, a1, a2, a3, b0, b1);
  }

  // F16 mode: ksA / ksB scale the logits of entries gid / gid+8, vsA / vsB their weights.
  HS2_DEVI void step(uint32_t slot, bool okA, bool okB, float scale_log2, float ksA = 1.f, float ksB = 1.f,
                     float vsA = 1.f, float vsB = 1.f) {
    const int lane = threadIdx.x & 31;
    const int mi = lane >> 3, rr = lane & 7;
    float sc[NT][4];
    {
      // even and odd k-steps accumulate apart (two independent MMA chains), then add
      float s2[2][NT][4];
#pragma unroll
      for (int u = 0; u < 2; ++u)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) s2[u][nt][0] = s2[u][nt][1] = s2[u][nt][2] = s2[u][nt][3] = 0.f;
      // matrices: (entries 0-7 | 8-15) x (d +0 | +8): a0 = (0-7, +0), a1 = (8-15, +0), a2 = (0-7, +8), a3 = (8-15, +8)
      const int row = rr + 8 * (mi & 1), dsub = 8 * (mi >> 1);
#pragma unroll
      for (int s = 0; s < KS; ++s) {
        const int d0 = 16 * s + dsub;
        uint32_t a[4];
        ldsm_x4(slot + (d0 >> 6) * 2048 + sw128(row, (d0 & 63) >> 3), a);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) mma(s2[s & 1][nt], a[0], a[1], a[2], a[3], qb[s][nt][0], qb[s][nt][1]);
      }
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int i = 0; i < 4; ++i) sc[nt][i] = s2[0][nt][i] + s2[1][nt][i];
    }
    // V^T fragments by transposed loads, issued before the softmax so their latency overlaps
    // it: a0 = (entries 0-7, d +0), a1 = (0-7, d +8), a2 = (8-15, d +0), a3 = (8-15, d +8)
    uint32_t va[KS][4];
    {
      const int row = rr + 8 * (mi >> 1), dsub = 8 * (mi & 1);
      const uint32_t vbase = slot + HALVES * 2048;
#pragma unroll
      for (int mt = 0; mt < KS; ++mt) {
        const int d0 = 16 * mt + dsub;
        ldsm_x4_t(vbase + (d0 >> 6) * 2048 + sw128(row, (d0 & 63) >> 3), va[mt]);
      }
    }
    if (F16) {
      // a step whose largest |V scale| (vsA / vsB depend on gid only) exceeds the unit makes
      // that scale the unit, acc rescaled to it
      float vm = fmaxf(fabsf(vsA), fabsf(vsB));
      if (__any_sync(0xffffffffu, vm > vu)) {
        vm = fmaxf(vm, __shfl_xor_sync(0xffffffffu, vm, 4));
        vm = fmaxf(vm, __shfl_xor_sync(0xffffffffu, vm, 8));
        vm = fmaxf(vm, __shfl_xor_sync(0xffffffffu, vm, 16));
        const float f = vu / vm;
#pragma unroll
        for (int mt = 0; mt < KS; ++mt)
#pragma unroll
          for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int i = 0; i < 4; ++i) acc[mt][nt][i] *= f;
        vu = vm;
        vinv = 1.f / vm;
      }
    }
    uint32_t pb[NT][2];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      float x[4];
      x[0] = okA ? sc[nt][0] * (scale_log2 * ksA) : -INFINITY;
      x[1] = okA ? sc[nt][1] * (scale_log2 * ksA) : -INFINITY;
      x[2] = okB ? sc[nt][2] * (scale_log2 * ksB) : -INFINITY;
      x[3] = okB ? sc[nt][3] * (scale_log2 * ksB) : -INFINITY;
      float p[4];
      // lazy rescale: the running max moves (l and acc rescaled) only when a logit exceeds it
      // by more than kLazyRescale, so weights stay <= 2^8; the final normalisation uses the
      // same max. Each lane checks its own logits; the column maxima are reduced across the
      // warp only when some lane needs a move (after the first step, rarely). The first
      // step with a valid entry moves every head's max off -inf (every head then has a finite
      // logit), so x - m below is never -inf - (-inf).
      const bool grow = x[0] > m[nt][0] + kLazyRescale || x[2] > m[nt][0] + kLazyRescale ||
                        x[1] > m[nt][1] + kLazyRescale || x[3] > m[nt][1] + kLazyRescale;
      if (__any_sync(0xffffffffu, grow)) {
        float cm[2];
#pragma unroll
        for (int hs = 0; hs < 2; ++hs) {
          cm[hs] = fmaxf(x[hs], x[hs + 2]);
          cm[hs] = fmaxf(cm[hs], __shfl_xor_sync(0xffffffffu, cm[hs], 4));
          cm[hs] = fmaxf(cm[hs], __shfl_xor_sync(0xffffffffu, cm[hs], 8));
          cm[hs] = fmaxf(cm[hs], __shfl_xor_sync(0xffffffffu, cm[hs], 16));
        }
#pragma unroll
        for (int hs = 0; hs < 2; ++hs) {
          const float mn = fmaxf(m[nt][hs], cm[hs]);
          const float alpha = (mn == -INFINITY) ? 1.f : exp2f(m[nt][hs] - mn);
          m[nt][hs] = mn;
          l[nt][hs] *= alpha;
#pragma unroll
          for (int mt = 0; mt < KS; ++mt) {
            acc[mt][nt][hs] *= alpha;
            acc[mt][nt][hs + 2] *= alpha;
          }
        }
      }
#pragma unroll
      for (int hs = 0; hs < 2; ++hs) {
        p[hs] = ex2_approx(x[hs] - m[nt][hs]);
        p[hs + 2] = ex2_approx(x[hs + 2] - m[nt][hs]);
      }
      uint32_t pA, pB;  // entry gid / gid+8, heads 2tig, 2tig+1
      if (F16) {
        const float wA = vsA * vinv, wB = vsB * vinv;
        pA = pack_f16(p[0] * wA, p[1] * wA);
        pB = pack_f16(p[2] * wB, p[3] * wB);
        l[nt][0] += p[0] + p[2];
        l[nt][1] += p[1] + p[3];
      } else {
        pA = pack_bf16(p[0], p[1]);
        pB = pack_bf16(p[2], p[3]);
        l[nt][0] += bf16_lo(pA) + bf16_lo(pB);
        l[nt][1] += bf16_hi(pA) + bf16_hi(pB);
      }
      pb[nt][0] = movmatrix_trans(pA);
      pb[nt][1] = movmatrix_trans(pB);
    }
#pragma unroll
    for (int mt = 0; mt < KS; ++mt)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) mma(acc[mt][nt], va[mt][0], va[mt][1], va[mt][2], va[mt][3], pb[nt][0], pb[nt][1]);
  }

  // Write this warp's (m, l, unnormalised o): sm_m / sm_l [warp][NT*8], sm_o [warp][NT*8][D].
  HS2_DEVI void store(int warp, float* sm_m, float* sm_l, float* sm_o) const {
    const int lane = threadIdx.x & 31, gid = lane >> 2, tig = lane & 3;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
      for (int hs = 0; hs < 2; ++hs) {
        float lv = l[nt][hs];
        lv += __shfl_xor_sync(0xffffffffu, lv, 4);
        lv += __shfl_xor_sync(0xffffffffu, lv, 8);
        lv += __shfl_xor_sync(0xffffffffu, lv, 16);
        const int hl = nt * 8 + 2 * tig + hs;
        if (gid == 0) {
          sm_m[warp * NT * 8 + hl] = m[nt][hs];
          sm_l[warp * NT * 8 + hl] = lv;
        }
        float* o = sm_o + ((size_t)warp * NT * 8 + hl) * D;
#pragma unroll
        for (int mt = 0; mt < KS; ++mt) {
          o[16 * mt + gid] = acc[mt][nt][hs] * unit();
          o[16 * mt + gid + 8] = acc[mt][nt][hs + 2] * unit();
        }
      }
    }
  }
};

}  // namespace hs2

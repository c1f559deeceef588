// mma_attn.cuh — one warp's online-softmax attention over 16 keys at a time on mma.sync,
// for a KV head shared by up to 8*NT query heads (bf16 inputs, fp32 accumulation).
//
// Register mappings (m16n8k16, groupID = lane/4, tig = lane%4):
//  S^T[16 keys x 8 heads] = K[16 keys x 16 d] * Q^T[16 d x 8 heads]
//    K rows gid and gid+8 arrive as D/32 chunks of 8 bf16 at d = 32j + 8*tig; k-step
//    s = 2j+u uses words 2u (a0/a1) and 2u+1 (a2/a3): the contraction index is permuted
//    identically for K and Q, so the dot products are unchanged.
//  O^T[16 d x 8 heads] += V^T[16 d x 16 keys] * P^T[16 keys x 8 heads]
//    the lane holds keys {2tig, 2tig+1, 2tig+8, 2tig+9} at d in [(D/8)gid, (D/8)(gid+1));
//    m-tile mt, row hi <-> d = (D/8)*gid + 2mt + hi. P^T fragments come from the S^T
//    accumulators through an 8x8 movmatrix transpose.
// Softmax is base 2 with a lazily moved running max; the normaliser sums the bf16-rounded
// weights that enter P.V.
// F16 = true (an FP8 cache, converted to f16 on load): queries are converted from bf16 to
// f16 once, both contractions run on the f16 MMA on the unscaled E4M3 codes, and P enters
// P.V as f16(p) (p <= 2^8, the codes <= 448: no f16 overflow or underflow of note); the
// normaliser sums p itself (fp32). The caller keeps acc in units of the current page's V
// scale (scale_acc when the page changes) and hands the last unit to store().
#pragma once
#include "common.cuh"

namespace hs2 {

template <int D, int NT, bool F16 = false>
struct MmaAttn {
  static constexpr int KS = D / 16;  // k-steps of QK^T and m-tiles of PV
  static constexpr int KC = D / 32;  // 16-byte K chunks per lane and row
  static constexpr int VC = D / 64;  // 16-byte V chunks per lane and key
  uint32_t qb[KS][NT][2];
  float m[NT][2], l[NT][2];
  float gmax[NT][2];  // the last step's max logit over its 16 keys, heads 2tig and 2tig+1
  float acc[KS][NT][4];

  // Q^T B-fragments of heads nt*8 + gid (heads >= G contribute zeros).
  HS2_DEVI void init(const __nv_bfloat16* q_heads, int G) {
    const int lane = threadIdx.x & 31, gid = lane >> 2, tig = lane & 3;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const int hl = nt * 8 + gid;
      const bool hv = hl < G;
      const uint32_t* qrow = reinterpret_cast<const uint32_t*>(q_heads + (size_t)(hv ? hl : 0) * D);
#pragma unroll
      for (int s = 0; s < KS; ++s) {
        const int base = 32 * (s >> 1) + 8 * tig + 4 * (s & 1);
        qb[s][nt][0] = hv ? qrow[base / 2] : 0u;
        qb[s][nt][1] = hv ? qrow[base / 2 + 1] : 0u;
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

  // K rows gid (kr0) and gid+8 (kr1); V keys 2tig, 2tig+1, 2tig+8, 2tig+9 (vr, zeroed when
  // invalid); okA / okB mask keys gid / gid+8. x receives the scaled base-2 logits
  // (x[nt][0..1]: key gid, heads 2tig, 2tig+1; x[nt][2..3]: key gid+8), -inf when masked.
  HS2_DEVI static void mma(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                           uint32_t b1) {
    if (F16) mma_f16_16816(c, a0, a1, a2, a3, b0, b1);
    else mma_bf16_16816(c, a0, a1, a2, a3, b0, b1);
  }

  // V^T A-fragments of m-tile mt from the per-key rows: va[mt] = {keys (2tig, 2tig+1) at
  // d, at d+1; keys (2tig+8, 2tig+9) at d, at d+1}, d = (D/8)*gid + 2mt.
  HS2_DEVI static void v_frags(const uint4 (&vr)[4][VC], uint32_t (&va)[KS][4]) {
#pragma unroll
    for (int mt = 0; mt < KS; ++mt) {
      const int j = mt >> 2, w4 = mt & 3;
      const uint32_t v0 = (&vr[0][j].x)[w4], v1 = (&vr[1][j].x)[w4];
      const uint32_t v2 = (&vr[2][j].x)[w4], v3 = (&vr[3][j].x)[w4];
      va[mt][0] = __byte_perm(v0, v1, 0x5410);
      va[mt][1] = __byte_perm(v0, v1, 0x7632);
      va[mt][2] = __byte_perm(v2, v3, 0x5410);
      va[mt][3] = __byte_perm(v2, v3, 0x7632);
    }
  }

  HS2_DEVI void step(const uint4 (&kr0)[KC], const uint4 (&kr1)[KC], const uint4 (&vr)[4][VC], bool okA, bool okB,
                     float scale_log2, float (&x)[NT][4]) {
    uint32_t va[KS][4];
    v_frags(vr, va);
    step(kr0, kr1, va, okA, okB, scale_log2, x);
  }

  HS2_DEVI void step(const uint4 (&kr0)[KC], const uint4 (&kr1)[KC], const uint32_t (&va)[KS][4], bool okA,
                     bool okB, float scale_log2, float (&x)[NT][4]) {
    float sc[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      // even and odd k-steps accumulate apart (two independent MMA chains), then add
      float s2[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
      for (int s = 0; s < KS; ++s) {
        const int j = s >> 1, u = s & 1;
        const uint32_t a0 = u ? kr0[j].z : kr0[j].x;
        const uint32_t a2 = u ? kr0[j].w : kr0[j].y;
        const uint32_t a1 = u ? kr1[j].z : kr1[j].x;
        const uint32_t a3 = u ? kr1[j].w : kr1[j].y;
        mma(s2[u], a0, a1, a2, a3, qb[s][nt][0], qb[s][nt][1]);
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) sc[nt][i] = s2[0][i] + s2[1][i];
    }
    uint32_t pb[NT][2];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      x[nt][0] = okA ? sc[nt][0] * scale_log2 : -INFINITY;
      x[nt][1] = okA ? sc[nt][1] * scale_log2 : -INFINITY;
      x[nt][2] = okB ? sc[nt][2] * scale_log2 : -INFINITY;
      x[nt][3] = okB ? sc[nt][3] * scale_log2 : -INFINITY;
      float p[4], cm[2];
      bool grow = false;
#pragma unroll
      for (int hs = 0; hs < 2; ++hs) {
        cm[hs] = fmaxf(x[nt][hs], x[nt][hs + 2]);
        cm[hs] = fmaxf(cm[hs], __shfl_xor_sync(0xffffffffu, cm[hs], 4));
        cm[hs] = fmaxf(cm[hs], __shfl_xor_sync(0xffffffffu, cm[hs], 8));
        cm[hs] = fmaxf(cm[hs], __shfl_xor_sync(0xffffffffu, cm[hs], 16));
        gmax[nt][hs] = cm[hs];
        grow |= cm[hs] > m[nt][hs] + kLazyRescale;
      }
      // Lazy rescale: the running max moves (and l, acc are rescaled) only when a head's
      // chunk max exceeds it by more than kLazyRescale (base 2), so weights stay <= 2^8;
      // the final normalisation divides by the same stale max, so the result is unchanged.
      if (__any_sync(0xffffffffu, grow)) {
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
        p[hs] = exp2_rel(x[nt][hs], m[nt][hs]);
        p[hs + 2] = exp2_rel(x[nt][hs + 2], m[nt][hs]);
      }
      uint32_t pA, pB;  // key gid / gid+8, heads 2tig, 2tig+1
      if (F16) {
        pA = pack_f16(p[0], p[1]);
        pB = pack_f16(p[2], p[3]);
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

  // acc *= f (a change of the unit acc is kept in)
  HS2_DEVI void scale_acc(float f) {
#pragma unroll
    for (int mt = 0; mt < KS; ++mt)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[mt][nt][i] *= f;
  }

  // Write this warp's (m, l, unnormalised o * unit) for its 8*NT heads to shared memory:
  // sm_m / sm_l [warp][NT*8], sm_o [warp][NT*8][D].
  HS2_DEVI void store(int warp, float* sm_m, float* sm_l, float* sm_o, float unit = 1.f) const {
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
#pragma unroll
        for (int mt = 0; mt < KS; ++mt) {
          const int d0 = (D / 8) * gid + 2 * mt;
          sm_o[((size_t)warp * NT * 8 + hl) * D + d0] = acc[mt][nt][hs] * unit;
          sm_o[((size_t)warp * NT * 8 + hl) * D + d0 + 1] = acc[mt][nt][hs + 2] * unit;
        }
      }
    }
  }
};

}  // namespace hs2

// sa_decode.cu — SA gather-attention over window ∪ top-k, staged through shared memory.
//
// An SA layer of a HySparse2 Cross group reuses the group's KV and the FA's index set
// with its own query ("HySparse2：整体架构、KV 生命周期与 PD 分离", §5). Its query
// attends to the forced window W(t) and the selected far positions S(t) under ONE
// softmax (§7.2, §7.4: both kinds of positions join the same normalisation), reading
// entries in place through the block table rather than copying them (§7.2, last
// paragraph; "Lecture 10 · 混合架构与稀疏注意力", §5.5: a second lookup through the table).
//
// One CTA per (query, KV head) walks U = W(t) ++ S(t) in chunks of 64 rows. Every entry
// of U is first resolved through the block table into a pool row id in shared memory
// (one round of dependent loads per CTA); the K and V rows of each chunk are then
// gathered into shared memory with 16-byte cp.async copies, three chunks in flight.
// The query heads of the KV head share every gathered row, which is what makes the
// gather worth its cost.
// Logits: each thread keeps 2 query heads x 32 contraction elements in registers (bf16)
// and the 4 partial sums of a row are combined with shuffles. P.V: each thread
// accumulates 8 output elements of 2 heads over a quarter of the rows. Products are
// bf16 x bf16 with fp32 accumulation (mixed-precision FMA, no widening instructions);
// the softmax weights enter P.V rounded to bf16 and the normaliser sums the same values. The online softmax merges
// chunks inside the CTA, so no partials leave the SM. CUDA cores only (fp32 FMA).
#include "common.cuh"
#include "kernels.h"

namespace hs2 {

namespace {

constexpr int kSaThreads = 256;
constexpr int kSaRows = 64;    // rows per chunk
constexpr int kSaStages = 3;   // chunks in flight (cp.async ring)

HS2_DEVI void cp_async16(void* smem, const void* gmem, bool valid) {
  const uint32_t s = (uint32_t)__cvta_generic_to_shared(smem);
  const int n = valid ? 16 : 0;  // zero-fill when the row is invalid (no global read)
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(s), "l"(gmem), "r"(n) : "memory");
}
HS2_DEVI void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
HS2_DEVI void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// 16-byte chunk c of a staged row r lives at chunk c ^ (4 * (r & 1)): the two rows a warp
// reads together in the logits phase then hit disjoint bank groups.
HS2_DEVI int swz(int r, int c) { return c ^ ((r & 1) << 2); }

}  // namespace

template <int D, int G>
__global__ void __launch_bounds__(kSaThreads) sa_gather_kernel(const AttnArgs a) {
  constexpr int HPT = G >= 2 ? 2 : 1;        // heads per thread (logits and P.V)
  constexpr int NHP = G / HPT;                // head groups
  constexpr int NDS = D / 32;                 // contraction slices of 32 per row
  constexpr int LPR = NDS * NHP;              // lanes per row in the logits phase
  static_assert(32 % LPR == 0, "row task must tile a warp");
  constexpr int RPW = 32 / LPR;               // rows per warp per logits pass
  constexpr int RPP = RPW * (kSaThreads / 32);  // rows per logits pass per CTA
  constexpr int CPR = D / 8;                  // 16-byte chunks per bf16 row
  constexpr int PV_GROUPS = CPR * NHP;        // (chunk, head group) tasks in P.V
  static_assert(kSaThreads % PV_GROUPS == 0, "P.V tasks must tile the CTA");
  constexpr int RQ = kSaThreads / PV_GROUPS;  // row residue classes in P.V

  const int qi = blockIdx.y, g = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const QueryGeom qg = query_geom(qi, a.prefill, a.seq_len);
  const int t = qg.t;
  float* out = a.out_o + ((size_t)qi * a.Hq + (size_t)g * G) * D;
  if (t < 1 || t > a.max_t || (t + kPage - 1) / kPage > a.max_pages) {
    if (tid == 0) flag_error(a.dev_err, HS2_DEV_BAD_LENGTH);
    for (int e = tid; e < G * D; e += kSaThreads) out[e] = 0.f;
    return;
  }
  const int nW = min(a.w, t);
  const int c0 = a.cnt[(size_t)qi * a.Hkv + g];
  if (tid == 0 && (c0 < 0 || c0 > a.kcap)) flag_error(a.dev_err, HS2_DEV_BAD_INDEX);
  const int nS = max(0, min(a.kcap, c0));
  const int nU = nW + nS;
  const int32_t* sel = a.idx + ((size_t)qi * a.Hkv + g) * a.kcap;
  const int32_t* bt = a.bt + (size_t)qg.b * a.max_pages;
  const int lim = a.w > 0 ? t - a.w : t;  // selected positions must lie in F(t)

  extern __shared__ float smem[];
  uint4* kst = reinterpret_cast<uint4*>(smem);                     // [kSaStages][kSaRows][CPR]
  uint4* vst = kst + kSaStages * kSaRows * CPR;                    // [kSaStages][kSaRows][CPR]
  float* p_s = reinterpret_cast<float*>(vst + kSaStages * kSaRows * CPR);  // [kSaRows][G] base-2 logits
  uint16_t* pb_s = reinterpret_cast<uint16_t*>(p_s + kSaRows * G);  // [kSaRows][G] bf16 weights
  float* red = reinterpret_cast<float*>(smem);            // [RQ][G][D], reuses the stage buffers at the end
  static_assert(RQ * G * D * 4 <= 2 * kSaStages * kSaRows * CPR * 16, "reduction buffer must fit the stage buffers");
  float* m_s = p_s + kSaRows * G + kSaRows * G / 2;       // [G]
  float* l_s = m_s + G;                                   // [G]
  float* alpha_s = l_s + G;                               // [G]
  int32_t* rowid = reinterpret_cast<int32_t*>(alpha_s + G);  // [w + kcap] pool row of each U entry, -1 = invalid

  // ---- q in registers: heads (hp*HPT .. +HPT), contraction slice ds, elements
  //      {8*(NDS*i + ds) .. +8} for i < 4 (interleaved so lanes of a row hit distinct banks)
  const int r_in = lane / LPR;            // row within the warp's pass
  const int hp = (lane % LPR) / NDS;      // head group
  const int ds = lane % NDS;              // contraction slice
  uint4 qw[HPT][4];  // bf16 pairs: head (hp*HPT+hh), elements 8*(NDS*i+ds) .. +8
  {
    const __nv_bfloat16* q = reinterpret_cast<const __nv_bfloat16*>(a.q) + ((size_t)qi * a.Hq + (size_t)g * G) * D;
#pragma unroll
    for (int hh = 0; hh < HPT; ++hh)
#pragma unroll
      for (int i = 0; i < 4; ++i)
        qw[hh][i] = *reinterpret_cast<const uint4*>(q + (size_t)(hp * HPT + hh) * D + 8 * (NDS * i + ds));
  }
  // P.V task of this thread
  const int pv_c = tid % CPR;             // 16-byte chunk = 8 output elements
  const int pv_hp = (tid / CPR) % NHP;    // head group
  const int pv_rq = tid / PV_GROUPS;      // row residue class
  float acc[HPT][8];
#pragma unroll
  for (int hh = 0; hh < HPT; ++hh)
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[hh][e] = 0.f;
  if (tid < G) {
    m_s[tid] = -INFINITY;
    l_s[tid] = 0.f;
  }

  // resolve every entry of U through the block table once (one round of dependent loads)
  for (int u = tid; u < nU; u += kSaThreads) {
    int pos, rid = -1;
    bool ok = true;
    if (u < nW) {
      pos = t - nW + u;
    } else {
      pos = sel[u - nW];
      if (pos < 0 || pos >= lim) {
        flag_error(a.dev_err, HS2_DEV_BAD_INDEX);
        ok = false;
      }
    }
    if (ok) {
      const int phys = bt[pos / kPage];
      if (phys < 0 || phys >= a.num_pages) flag_error(a.dev_err, HS2_DEV_BAD_PAGE);
      else rid = (phys * a.Hkv + g) * kPage + pos % kPage;
    }
    rowid[u] = rid;
  }
  __syncthreads();
  const int nchunk = (nU + kSaRows - 1) / kSaRows;
  const __nv_bfloat16* kb = reinterpret_cast<const __nv_bfloat16*>(a.k);
  const __nv_bfloat16* vb = reinterpret_cast<const __nv_bfloat16*>(a.v);
  // gather the rows of chunk c into ring slot `slot` (invalid rows are zero-filled)
  auto stage = [&](int c, int slot) {
    for (int e = tid; e < kSaRows * CPR; e += kSaThreads) {
      const int r = e / CPR, cc = e % CPR;
      const int u = c * kSaRows + r;
      const int rid = u < nU ? rowid[u] : -1;
      const bool ok = rid >= 0;
      const long long off = ok ? (long long)rid * D + 8 * cc : 0;
      cp_async16(&kst[(slot * kSaRows + r) * CPR + swz(r, cc)], kb + off, ok);
      cp_async16(&vst[(slot * kSaRows + r) * CPR + cc], vb + off, ok);
    }
  };
#pragma unroll
  for (int c = 0; c < kSaStages - 1; ++c) {
    if (c < nchunk) stage(c, c);
    cp_async_commit();
  }
  for (int c = 0; c < nchunk; ++c) {
    const int buf = c % kSaStages;
    cp_async_wait<kSaStages - 2>();
    __syncthreads();  // chunk c landed for every thread; the slot refilled below is free
    if (c + kSaStages - 1 < nchunk) stage(c + kSaStages - 1, (c + kSaStages - 1) % kSaStages);
    cp_async_commit();
    const int rows = min(kSaRows, nU - c * kSaRows);
    // ---- logits of this chunk (base 2) into p_s
    for (int r0 = warp * RPW; r0 < kSaRows; r0 += RPP) {
      const int r = r0 + r_in;
      float x[HPT];
#pragma unroll
      for (int hh = 0; hh < HPT; ++hh) x[hh] = 0.f;
      const uint4* krow = &kst[(buf * kSaRows + r) * CPR];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint4 u = krow[swz(r, NDS * i + ds)];
#pragma unroll
        for (int hh = 0; hh < HPT; ++hh) {
          const uint4 qv = qw[hh][i];
          x[hh] = fmab_ll(u.x, qv.x, x[hh]); x[hh] = fmab_hh(u.x, qv.x, x[hh]);
          x[hh] = fmab_ll(u.y, qv.y, x[hh]); x[hh] = fmab_hh(u.y, qv.y, x[hh]);
          x[hh] = fmab_ll(u.z, qv.z, x[hh]); x[hh] = fmab_hh(u.z, qv.z, x[hh]);
          x[hh] = fmab_ll(u.w, qv.w, x[hh]); x[hh] = fmab_hh(u.w, qv.w, x[hh]);
        }
      }
#pragma unroll
      for (int hh = 0; hh < HPT; ++hh) {
#pragma unroll
        for (int o = 1; o < NDS; o <<= 1) x[hh] += __shfl_xor_sync(0xffffffffu, x[hh], o);
      }
      if (ds == 0) {
        const int u = c * kSaRows + r;
        const bool ok = r < rows && rowid[u] >= 0;
#pragma unroll
        for (int hh = 0; hh < HPT; ++hh) p_s[r * G + hp * HPT + hh] = ok ? x[hh] * a.scale_log2 : -INFINITY;
      }
    }
    __syncthreads();
    // ---- chunk max per head, running max, weights (warp h handles head h)
    for (int h = warp; h < G; h += kSaThreads / 32) {
      float mx = -INFINITY;
      for (int r = lane; r < kSaRows; r += 32) mx = fmaxf(mx, p_s[r * G + h]);
      mx = warp_max(mx);
      const float mo = m_s[h];
      const float mn = fmaxf(mo, mx);
      const float al = (mn == -INFINITY) ? 1.f : exp2f(mo - mn);
      float ls = 0.f;
      for (int r = lane; r < kSaRows; r += 32) {
        // weights enter P.V as bf16; the normaliser sums the same rounded values
        const __nv_bfloat16 pb = __float2bfloat16_rn(exp2_rel(p_s[r * G + h], mn));
        pb_s[r * G + h] = __bfloat16_as_ushort(pb);
        ls += __bfloat162float(pb);
      }
      ls = warp_sum(ls);
      if (lane == 0) {
        m_s[h] = mn;
        l_s[h] = l_s[h] * al + ls;
        alpha_s[h] = al;
      }
    }
    __syncthreads();
    // ---- P.V over this chunk
#pragma unroll
    for (int hh = 0; hh < HPT; ++hh) {
      const float al = alpha_s[pv_hp * HPT + hh];
#pragma unroll
      for (int e = 0; e < 8; ++e) acc[hh][e] *= al;
    }
    for (int r = pv_rq; r < rows; r += RQ) {
      const uint4 u = vst[(buf * kSaRows + r) * CPR + pv_c];
      uint32_t pw;  // bf16 weights of this thread's heads: low half head 0, high half head 1
      if constexpr (HPT == 2) pw = *reinterpret_cast<const uint32_t*>(&pb_s[r * G + pv_hp * 2]);
      else pw = (uint32_t)pb_s[r * G + pv_hp];
#pragma unroll
      for (int hh = 0; hh < HPT; ++hh) {
        float* ac = acc[hh];
        if (hh == 0) {
          ac[0] = fmab_ll(pw, u.x, ac[0]); ac[1] = fmab_lh(pw, u.x, ac[1]);
          ac[2] = fmab_ll(pw, u.y, ac[2]); ac[3] = fmab_lh(pw, u.y, ac[3]);
          ac[4] = fmab_ll(pw, u.z, ac[4]); ac[5] = fmab_lh(pw, u.z, ac[5]);
          ac[6] = fmab_ll(pw, u.w, ac[6]); ac[7] = fmab_lh(pw, u.w, ac[7]);
        } else {
          ac[0] = fmab_hl(pw, u.x, ac[0]); ac[1] = fmab_hh(pw, u.x, ac[1]);
          ac[2] = fmab_hl(pw, u.y, ac[2]); ac[3] = fmab_hh(pw, u.y, ac[3]);
          ac[4] = fmab_hl(pw, u.z, ac[4]); ac[5] = fmab_hh(pw, u.z, ac[5]);
          ac[6] = fmab_hl(pw, u.w, ac[6]); ac[7] = fmab_hh(pw, u.w, ac[7]);
        }
      }
    }
    __syncthreads();  // the next iteration refills this chunk's slot only after its barrier
  }
  cp_async_wait<0>();
  __syncthreads();
  // ---- reduce the row residue classes and normalise
#pragma unroll
  for (int hh = 0; hh < HPT; ++hh)
#pragma unroll
    for (int e = 0; e < 8; ++e) red[(pv_rq * G + pv_hp * HPT + hh) * D + 8 * pv_c + e] = acc[hh][e];
  __syncthreads();
  for (int e = tid; e < G * D; e += kSaThreads) {
    float s = 0.f;
#pragma unroll
    for (int q2 = 0; q2 < RQ; ++q2) s += red[q2 * G * D + e];
    const float L = l_s[e / D];
    out[e] = L > 0.f ? s / L : 0.f;
  }
}

template <int D, int G>
static cudaError_t launch_sa(const AttnArgs& a, int Bq, cudaStream_t s) {
  const size_t sm = (size_t)2 * kSaStages * kSaRows * (D / 8) * 16 +
                    (size_t)(kSaRows * G + kSaRows * G / 2 + 3 * G) * 4 + (size_t)(a.w + a.kcap) * sizeof(int32_t);
  auto kern = sa_gather_kernel<D, G>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
  if (e != cudaSuccess) return e;
  kern<<<dim3(a.Hkv, Bq), kSaThreads, sm, s>>>(a);
  return cudaGetLastError();
}

bool sa_gather_supported(int G, int D, int bf16) {
  return bf16 && (D == 64 || D == 128) && (G == 2 || G == 4 || G == 8 || G == 16);
}

cudaError_t launch_sa_gather(const AttnArgs& a, int Bq, cudaStream_t s) {
  if (a.D == 128) {
    switch (a.G) {
      case 2: return launch_sa<128, 2>(a, Bq, s);
      case 4: return launch_sa<128, 4>(a, Bq, s);
      case 8: return launch_sa<128, 8>(a, Bq, s);
      case 16: return launch_sa<128, 16>(a, Bq, s);
    }
  } else if (a.D == 64) {
    switch (a.G) {
      case 2: return launch_sa<64, 2>(a, Bq, s);
      case 4: return launch_sa<64, 4>(a, Bq, s);
      case 8: return launch_sa<64, 8>(a, Bq, s);
      case 16: return launch_sa<64, 16>(a, Bq, s);
    }
  }
  return cudaErrorInvalidValue;
}

}  // namespace hs2

// sa_prefill.cu — SA gather-attention for every row of a bf16 prefill, on tensor cores.
//
// Each row's SA query attends to its forced window and its FA-selected far positions
// under one softmax ("HySparse2：整体架构、KV 生命周期与 PD 分离", §5, §7.2, §7.4), entries
// read in place through the block table. In prefill the gathered Q.K and P.V per row are
// dense contractions over the row's |W ∪ S| keys and the query heads sharing a KV head,
// so they run on mma.sync (keys as M, heads as N; see mma_attn.cuh).
//
// One CTA (4 warps) per (row, KV head, split). The CTA first resolves its share of the
// row's positions — window then selected — through the block table into pool row ids in
// shared memory (one round of dependent loads), then each warp walks 16-key steps
// (steps w, w+4, ...), loading K and V rows straight into MMA fragments with 128-bit
// loads, and the four warps' online-softmax states are merged at the end.
//
// Decode has one row per sequence, so (row, KV head) pairs alone leave most SMs of the
// GPU with one or two CTAs. There the row's |W ∪ S| entries are split across the CTAs of
// a thread-block cluster (grid z = cluster z = split count); each CTA merges its warps,
// and CTA rank 0 merges the cluster's partial states through distributed shared memory.
#include <cooperative_groups.h>

#include <algorithm>

#include "common.cuh"
#include "kernels.h"
#include "mma_attn.cuh"
#include "staged_attn.cuh"

namespace cg = cooperative_groups;

namespace hs2 {

constexpr int kSaMaxSplit = 8;  // portable cluster size

template <int D, int NT>
__global__ void __launch_bounds__(128, NT == 1 ? 4 : 0) sa_mma_kernel(const AttnArgs a) {
  using Attn = MmaAttn<D, NT>;
  constexpr int KC = Attn::KC, VC = Attn::VC;
  const int qi = blockIdx.y, g = blockIdx.x;
  const int split = blockIdx.z, nsplit = gridDim.z;  // cluster rank and size along z
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int gid = lane >> 2, tig = lane & 3;
  const int G = a.G;
  const QueryGeom qg = query_geom(qi, a.prefill, a.seq_len);
  const int t = qg.t;
  float* out = a.out_o + ((size_t)qi * a.Hq + (size_t)g * G) * D;
  // every CTA of a cluster shares (qi, g), so all of them take this exit or none does
  if (t < 1 || t > a.max_t || (t + kPage - 1) / kPage > a.max_pages) {
    if (split == 0) {
      if (tid == 0) flag_error(a.dev_err, HS2_DEV_BAD_LENGTH);
      for (int e = tid; e < G * D; e += 128) out[e] = 0.f;
    }
    return;
  }
  const int nW = min(a.w, t);
  const int c0 = a.cnt[(size_t)qi * a.Hkv + g];
  if (tid == 0 && split == 0 && (c0 < 0 || c0 > a.kcap)) flag_error(a.dev_err, HS2_DEV_BAD_INDEX);
  const int nS = max(0, min(a.kcap, c0));
  const int nUall = nW + nS;
  // this CTA's share: whole 16-entry steps [st0, st1) of W ∪ S
  const int nst_all = (nUall + 15) / 16;
  const int st0 = (int)((long long)nst_all * split / nsplit), st1 = (int)((long long)nst_all * (split + 1) / nsplit);
  const int u_lo = st0 * 16, nU = min(nUall, st1 * 16) - u_lo;  // entries u_lo .. u_lo + nU - 1
  const int32_t* sel = a.idx + ((size_t)qi * a.Hkv + g) * a.kcap;
  const int32_t* bt = a.bt + (size_t)qg.b * a.max_pages;
  const int lim = a.w > 0 ? t - a.w : t;

  extern __shared__ float smem[];
  float* sm_m = smem;                  // [4][NT*8]
  float* sm_l = sm_m + 4 * NT * 8;     // [4][NT*8]
  float* sm_o = sm_l + 4 * NT * 8;     // [4][NT*8][D]
  float* cta_m = sm_o + 4 * NT * 8 * D;  // [NT*8]     this CTA's merged state
  float* cta_l = cta_m + NT * 8;         // [NT*8]
  float* cta_o = cta_l + NT * 8;         // [NT*8][D]  (unnormalised, relative to cta_m)
  int32_t* rowid = reinterpret_cast<int32_t*>(cta_o + NT * 8 * D);  // [nU] pool row, -1 invalid

  for (int ul = tid; ul < nU; ul += 128) {
    const int u = u_lo + ul;
    int pos, r = -1;
    bool ok = true;
    if (u < nW) {
      pos = t - nW + u;
    } else {
      pos = __ldcs(&sel[u - nW]);  // read once: do not keep in L2
      if (pos < 0 || pos >= lim) {
        flag_error(a.dev_err, HS2_DEV_BAD_INDEX);
        ok = false;
      }
    }
    if (ok) {
      const int phys = bt[pos / kPage];
      if (phys < 0 || phys >= a.num_pages) flag_error(a.dev_err, HS2_DEV_BAD_PAGE);
      else r = (phys * a.Hkv + g) * kPage + pos % kPage;
    }
    rowid[ul] = r;
  }
  Attn at;
  at.init(reinterpret_cast<const __nv_bfloat16*>(a.q) + ((size_t)qi * a.Hq + (size_t)g * G) * D, G);
  __syncthreads();

  const __nv_bfloat16* kb = reinterpret_cast<const __nv_bfloat16*>(a.k);
  const __nv_bfloat16* vb = reinterpret_cast<const __nv_bfloat16*>(a.v);
  const uint64_t keep = l2_keep_policy();  // rows are re-read by other rows' CTAs
  const int nsteps = (nU + 15) / 16;
  for (int st = warp; st < nsteps; st += 4) {
    const int u0 = st * 16;
    const int ua = u0 + gid, ub = u0 + gid + 8;
    const int ra = ua < nU ? rowid[ua] : -1;
    const int rb = ub < nU ? rowid[ub] : -1;
    uint4 kr0[KC], kr1[KC], vr[4][VC];
#pragma unroll
    for (int j = 0; j < KC; ++j) {
      kr0[j] = ra >= 0 ? ldg_nc_v4_keep(kb + (size_t)ra * D + 32 * j + 8 * tig, keep) : make_uint4(0, 0, 0, 0);
      kr1[j] = rb >= 0 ? ldg_nc_v4_keep(kb + (size_t)rb * D + 32 * j + 8 * tig, keep) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int uv = u0 + 2 * tig + (e & 1) + 8 * (e >> 1);
      const int rv = uv < nU ? rowid[uv] : -1;
#pragma unroll
      for (int j = 0; j < VC; ++j)
        vr[e][j] = rv >= 0 ? ldg_nc_v4_keep(vb + (size_t)rv * D + (D / 8) * gid + 8 * j, keep) : make_uint4(0, 0, 0, 0);
    }
    float x[NT][4];
    at.step(kr0, kr1, vr, ra >= 0, rb >= 0, a.scale_log2, x);
  }
  at.store(warp, sm_m, sm_l, sm_o);
  __syncthreads();
  for (int e = tid; e < G * D; e += 128) {
    const int hl = e / D, dd = e % D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < 4; ++w) M = fmaxf(M, sm_m[w * NT * 8 + hl]);
    float L = 0.f, Ov = 0.f;
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      const float f = exp2_rel(sm_m[w * NT * 8 + hl], M);
      L += f * sm_l[w * NT * 8 + hl];
      Ov += f * sm_o[((size_t)w * NT * 8 + hl) * D + dd];
    }
    if (nsplit == 1) {
      const int hq = g * G + hl;
      float v = Ov * sa_norm_factor(M, L, sink_b2(a.sink, hq));
      if (a.gate) v *= sa_gate(__ldcs(&a.gate[((size_t)qi * a.Hq + hq) * D + dd]));
      __stcs(&out[e], v);  // streaming store: keep L2 for the K/V rows
    } else {
      cta_o[e] = Ov;
      if (dd == 0) {
        cta_m[hl] = M;
        cta_l[hl] = L;
      }
    }
  }
  if (nsplit == 1) return;
  // cluster merge: rank 0 reads every CTA's (m, l, o) through distributed shared memory;
  // the second barrier keeps the peers' shared memory alive until it has done so
  cg::cluster_group cluster = cg::this_cluster();
  cluster.sync();
  if (split == 0) {
    for (int e = tid; e < G * D; e += 128) {
      const int hl = e / D;
      float M = -INFINITY;
      for (int r = 0; r < nsplit; ++r) M = fmaxf(M, cluster.map_shared_rank(cta_m, r)[hl]);
      float L = 0.f, Ov = 0.f;
      for (int r = 0; r < nsplit; ++r) {
        const float f = exp2_rel(cluster.map_shared_rank(cta_m, r)[hl], M);
        L += f * cluster.map_shared_rank(cta_l, r)[hl];
        Ov += f * cluster.map_shared_rank(cta_o, r)[e];
      }
      const int hq = g * G + hl;
      float v = Ov * sa_norm_factor(M, L, sink_b2(a.sink, hq));
      if (a.gate) v *= sa_gate(a.gate[((size_t)qi * a.Hq + hq) * D + e % D]);
      out[e] = v;
    }
  }
  cluster.sync();
}

// ============================================================================ staged variant
// Prefill with at most 8 query heads per KV head: the same CTA per (row, KV head) and steps
// per warp, but each warp streams its steps through a 2-slot shared-memory ring (cp.async,
// zero rows for invalid entries, 128-byte swizzle), so the next step's rows are in flight
// from L2 while the current one is contracted from shared memory (ldmatrix + mma.sync,
// staged_attn.cuh). The warps' merge buffers reuse the rings once the stream is done.
constexpr int kStgSlots = 2;
template <int D>
constexpr uint32_t stg_slot_bytes() {  // 16 K rows and 16 V rows
  return 2u * (D / 64) * 2048u;
}

template <int D>
__global__ void __launch_bounds__(128, 3) sa_staged_kernel(const AttnArgs a) {
  constexpr int HALVES = D / 64;
  constexpr int CPR = D / 8;  // 16-byte chunks per row
  constexpr uint32_t kSlot = stg_slot_bytes<D>();
  const int qi = blockIdx.y, g = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int gid = lane >> 2;
  const int G = a.G;  // <= 8
  const QueryGeom qg = query_geom(qi, a.prefill, a.seq_len);
  const int t = qg.t;
  float* out = a.out_o + ((size_t)qi * a.Hq + (size_t)g * G) * D;
  if (t < 1 || t > a.max_t || (t + kPage - 1) / kPage > a.max_pages) {
    if (tid == 0) flag_error(a.dev_err, HS2_DEV_BAD_LENGTH);
    for (int e = tid; e < G * D; e += 128) out[e] = 0.f;
    return;
  }
  const int nW = min(a.w, t);
  const int c0 = a.cnt[(size_t)qi * a.Hkv + g];
  if (tid == 0 && (c0 < 0 || c0 > a.kcap)) flag_error(a.dev_err, HS2_DEV_BAD_INDEX);
  const int nS = max(0, min(a.kcap, c0));
  const int nU = nW + nS;
  const int32_t* sel = a.idx + ((size_t)qi * a.Hkv + g) * a.kcap;
  const int32_t* bt = a.bt + (size_t)qg.b * a.max_pages;
  const int lim = a.w > 0 ? t - a.w : t;

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = (uint32_t)__cvta_generic_to_shared(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;  // the swizzled slots want 1024-byte alignment
  uint8_t* basep = smem_raw + (base - raw);
  int32_t* rowid = reinterpret_cast<int32_t*>(basep + 4 * kStgSlots * kSlot);  // [nU] pool row, -1 invalid

  for (int u = tid; u < nU; u += 128) {
    int pos, r = -1;
    bool ok = true;
    if (u < nW) {
      pos = t - nW + u;
    } else {
      pos = __ldcs(&sel[u - nW]);  // read once: do not keep in L2
      if (pos < 0 || pos >= lim) {
        flag_error(a.dev_err, HS2_DEV_BAD_INDEX);
        ok = false;
      }
    }
    if (ok) {
      const int phys = bt[pos / kPage];
      if (phys < 0 || phys >= a.num_pages) flag_error(a.dev_err, HS2_DEV_BAD_PAGE);
      else r = (phys * a.Hkv + g) * kPage + pos % kPage;
    }
    rowid[u] = r;
  }
  // the last step's tail: no rows
  for (int u = nU + tid; u < (nU + 15) / 16 * 16; u += 128) rowid[u] = -1;
  StagedAttn<D, 1> at;
  at.init(reinterpret_cast<const __nv_bfloat16*>(a.q) + ((size_t)qi * a.Hq + (size_t)g * G) * D, G);
  __syncthreads();

  const __nv_bfloat16* kb = reinterpret_cast<const __nv_bfloat16*>(a.k);
  const __nv_bfloat16* vb = reinterpret_cast<const __nv_bfloat16*>(a.v);
  const uint64_t keep = l2_keep_policy();  // rows are re-read by other rows' CTAs
  const uint32_t ring = base + (uint32_t)warp * kStgSlots * kSlot;
  // A warp instruction copies 16-byte chunk cc = lane % CPR of rows r0 + RSTEP m, r0 =
  // lane / CPR < RSTEP. Everything but the row id is fixed per lane: the source is the row's
  // base plus this lane's chunk, and the swizzled destination of row r0 + RSTEP m is this
  // lane's row-r0 offset with bits 4-6 flipped by (RSTEP m) & 7 (r0 and RSTEP m share no bit).
  constexpr int RSTEP = 32 / CPR;
  const int cc = lane % CPR, r0 = lane / CPR;
  const __nv_bfloat16* kl = kb + 8 * cc;
  const __nv_bfloat16* vl = vb + 8 * cc;
  const uint32_t so0 = (uint32_t)(cc >> 3) * 2048u + sw128(r0, cc & 7);
  auto issue = [&](int st, int slot) {
    const uint32_t dst = ring + (uint32_t)slot * kSlot;
    const int32_t* rid_st = rowid + st * 16 + r0;  // padded with -1 to a whole step
#pragma unroll
    for (int m = 0; m < 16 / RSTEP; ++m) {
      const int rid = rid_st[RSTEP * m];
      const size_t off = (size_t)max(rid, 0) * D;
      const uint32_t so = (so0 ^ ((uint32_t)((RSTEP * m) & 7) << 4)) + (uint32_t)(RSTEP * m) * 128u;
      cp_async16_keep(dst + so, kl + off, rid >= 0, keep);
      cp_async16_keep(dst + HALVES * 2048u + so, vl + off, rid >= 0, keep);
    }
  };
  const int nsteps = (nU + 15) / 16;
  if (warp < nsteps) issue(warp, 0);
  cp_async_commit();
  int li = 0;
  for (int st = warp; st < nsteps; st += 4, ++li) {
    if (st + 4 < nsteps) issue(st + 4, (li + 1) & 1);
    cp_async_commit();
    cp_async_wait<1>();  // this step's copies (issued one step earlier) have landed
    __syncwarp();
    const int ua = st * 16 + gid, ub = ua + 8;
    const bool okA = ua < nU && rowid[ua] >= 0, okB = ub < nU && rowid[ub] >= 0;
    if (__any_sync(0xffffffffu, okA || okB)) at.step(ring + (uint32_t)(li & 1) * kSlot, okA, okB, a.scale_log2);
    __syncwarp();  // the slot is refilled by the next issue
  }
  cp_async_wait<0>();
  __syncthreads();  // the merge buffers below reuse the rings
  float* sm_m = reinterpret_cast<float*>(basep);  // [4][8]
  float* sm_l = sm_m + 4 * 8;                      // [4][8]
  float* sm_o = sm_l + 4 * 8;                      // [4][8][D]
  at.store(warp, sm_m, sm_l, sm_o);
  __syncthreads();
  for (int e = tid; e < G * D; e += 128) {
    const int hl = e / D, dd = e % D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < 4; ++w) M = fmaxf(M, sm_m[w * 8 + hl]);
    float L = 0.f, Ov = 0.f;
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      const float f = exp2_rel(sm_m[w * 8 + hl], M);
      L += f * sm_l[w * 8 + hl];
      Ov += f * sm_o[((size_t)w * 8 + hl) * D + dd];
    }
    const int hq = g * G + hl;
    float v = Ov * sa_norm_factor(M, L, sink_b2(a.sink, hq));
    if (a.gate) v *= sa_gate(__ldcs(&a.gate[((size_t)qi * a.Hq + hq) * D + dd]));
    __stcs(&out[e], v);  // streaming store: keep L2 for the K/V rows
  }
}

static size_t sa_staged_smem(int D, long long w, long long k) {  // rings, then the row ids of whole steps
  return 1024 + 4 * kStgSlots * (size_t)(D == 128 ? stg_slot_bytes<128>() : stg_slot_bytes<64>()) +
         (size_t)((w + k + 15) / 16 * 16) * 4;
}

template <int D>
static cudaError_t launch_sa_staged_t(const AttnArgs& a, int Bq, cudaStream_t s) {
  const size_t sm = sa_staged_smem(D, a.w, a.kcap);
  cudaError_t e = cudaFuncSetAttribute(sa_staged_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
  if (e != cudaSuccess) return e;
  sa_staged_kernel<D><<<dim3(a.Hkv, Bq), 128, sm, s>>>(a);
  return cudaGetLastError();
}

static long long sa_mma_smem(int NT, int D, long long w, long long k) {
  return (64LL * NT + 32LL * NT * D + 16LL * NT + 8LL * NT * D) * 4 + (w + k) * 4;
}

template <int D, int NT>
static cudaError_t launch_sa_mma_t(const AttnArgs& a, int Bq, cudaStream_t s) {
  const size_t sm = (size_t)sa_mma_smem(NT, D, a.w, a.kcap);
  auto kern = sa_mma_kernel<D, NT>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
  if (e != cudaSuccess) return e;
  // split each (row, KV head) over a cluster when the pairs alone cannot fill the GPU
  int dev = 0, sms = 0, per_sm = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, 128, sm)) != cudaSuccess) return e;
  const long long pairs = (long long)a.Hkv * Bq, slots = (long long)sms * std::max(per_sm, 1);
  const int max_steps = (a.w + a.kcap + 15) / 16;
  int nsplit = 1;
  if (pairs < slots) nsplit = (int)std::min<long long>(kSaMaxSplit, (slots + pairs - 1) / pairs);
  nsplit = std::max(1, std::min(nsplit, max_steps / 4));  // at least ~4 steps of 16 per CTA
  if (nsplit == 1) {
    kern<<<dim3(a.Hkv, Bq), 128, sm, s>>>(a);
    return cudaGetLastError();
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.Hkv, Bq, nsplit);
  cfg.blockDim = dim3(128);
  cfg.dynamicSmemBytes = sm;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 1;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = nsplit;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, a);
}

bool sa_mma_supported(int G, int D, int bf16, int w, int k) {
  if (!bf16 || (D != 64 && D != 128) || G > 32 || (G > 8 && G != 16 && G != 32)) return false;
  return sa_mma_smem((G + 7) / 8, D, w, k) <= 227LL * 1024;
}

cudaError_t launch_sa_mma(const AttnArgs& a, int Bq, cudaStream_t s) {
  const int NTl = (a.G + 7) / 8;
  // prefill rows fill the GPU on their own: the staged stream for up to 8 heads per KV head
  if (a.prefill && NTl == 1 && sa_staged_smem(a.D, a.w, a.kcap) <= 227u * 1024u)
    return a.D == 128 ? launch_sa_staged_t<128>(a, Bq, s) : launch_sa_staged_t<64>(a, Bq, s);
  if (a.D == 128) {
    switch (NTl) {
      case 1: return launch_sa_mma_t<128, 1>(a, Bq, s);
      case 2: return launch_sa_mma_t<128, 2>(a, Bq, s);
      case 4: return launch_sa_mma_t<128, 4>(a, Bq, s);
    }
  } else if (a.D == 64) {
    switch (NTl) {
      case 1: return launch_sa_mma_t<64, 1>(a, Bq, s);
      case 2: return launch_sa_mma_t<64, 2>(a, Bq, s);
      case 4: return launch_sa_mma_t<64, 4>(a, Bq, s);
    }
  }
  return cudaErrorInvalidValue;
}

}  // namespace hs2

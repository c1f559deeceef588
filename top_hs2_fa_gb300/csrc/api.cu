// api.cu — the extern "C" boundary of libhs2: argument validation, workspace layout,
// launches. No allocation, no synchronisation; every call is asynchronous on `stream`.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>
#include <cmath>

#include "../../include/hs2.h"
#include "kernels.h"

namespace {

thread_local int g_last_cuda_error = 0;
thread_local void* g_prof[3][2] = {{nullptr, nullptr}, {nullptr, nullptr}, {nullptr, nullptr}};

// Records the one-shot profiling events of `stage` around `launch` (a callable returning cudaError_t).
template <typename F>
cudaError_t profiled(int stage, cudaStream_t s, F launch) {
  void* ev0 = g_prof[stage][0];
  void* ev1 = g_prof[stage][1];
  g_prof[stage][0] = g_prof[stage][1] = nullptr;
  if (ev0) {
    cudaError_t e = cudaEventRecord((cudaEvent_t)ev0, s);
    if (e != cudaSuccess) return e;
  }
  cudaError_t e = launch();
  if (e == cudaSuccess && ev1) e = cudaEventRecord((cudaEvent_t)ev1, s);
  return e;
}

hs2_status cuda_fail(cudaError_t e) {
  g_last_cuda_error = (int)e;
  (void)cudaGetLastError();  // clear the sticky-free error state of the calling thread
  return HS2_ERR_CUDA;
}

inline size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }
inline bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }
inline int cdiv(long long a, long long b) { return (int)((a + b - 1) / b); }

bool valid_kv(const hs2_kv* kv, bool need_v) {
  if (!kv || !kv->k || !kv->block_table || !kv->seq_len) return false;
  if (need_v && !kv->v) return false;
  if (kv->batch < 1 || kv->num_pages < 1 || kv->max_pages < 1 || kv->Hkv < 1) return false;
  if (kv->page_size != 64) return false;
  if (kv->d != 64 && kv->d != 128) return false;
  if (kv->dtype != HS2_F32 && kv->dtype != HS2_BF16 && kv->dtype != HS2_FP8_E4M3 && kv->dtype != HS2_FP4_E2M1)
    return false;
  if ((kv->dtype == HS2_FP8_E4M3 || kv->dtype == HS2_FP4_E2M1) && (!kv->k_scale || (need_v && !kv->v_scale)))
    return false;
  if (kv->dtype == HS2_FP4_E2M1 && (!kv->k_sf || !aligned16(kv->k_sf) || (need_v && (!kv->v_sf || !aligned16(kv->v_sf)))))
    return false;
  if (!aligned16(kv->k) || (need_v && !aligned16(kv->v))) return false;
  return true;
}

// FP8 / FP4 caches (quantised codes with scales): decode only
bool low_precision(const hs2_kv* kv) { return kv->dtype == HS2_FP8_E4M3 || kv->dtype == HS2_FP4_E2M1; }

bool pow2_le32(int g) { return g == 1 || g == 2 || g == 4 || g == 8 || g == 16 || g == 32; }

// ---------------------------------------------------------------------------- FA layout
struct FaPlan {
  bool mma;   // bf16 tensor-core scan (else CUDA-core)
  int pps;    // pages per split
  int nsplit;
  long long ld;  // logits row length
  size_t off_ml, off_o, off_lcode, off_lmax, off_scores, off_hist, total;
};

FaPlan fa_plan(int Bq, int Hq, const hs2_kv* kv, int max_t) {
  FaPlan p{};
  const int G = Hq / kv->Hkv;
  p.mma = (kv->dtype == HS2_BF16 || low_precision(kv)) && G <= 32 && (G <= 8 || G == 16 || G == 32);
  const int maxpg = cdiv(max_t, 64);
  if (p.mma) {
    // enough CTAs to fill 152 SMs several times over, splits of at most 32 pages (2048 keys:
    // 16 wrote and merged twice the partials, 6.6 us more per decode step; 64 left too few CTAs)
    p.pps = 32;
    while (p.pps > 1 && (long long)Bq * kv->Hkv * cdiv(maxpg, p.pps) < 152LL * 8) p.pps >>= 1;
  } else {
    p.pps = 2;
  }
  p.nsplit = cdiv(maxpg, p.pps);
  p.ld = (long long)maxpg * 64;
  size_t off = 0;
  p.off_ml = off;
  off = align256(off + (size_t)Bq * Hq * p.nsplit * sizeof(float) * 2);
  p.off_o = off;
  off = align256(off + (size_t)Bq * Hq * p.nsplit * kv->d * sizeof(float));
  p.off_lcode = off;
  off = align256(off + (size_t)Bq * Hq * p.ld * sizeof(uint16_t));
  p.off_lmax = off;
  off = align256(off + (size_t)Bq * Hq * (p.ld / 16) * sizeof(float));
  p.off_scores = off;
  off = align256(off + (size_t)Bq * kv->Hkv * p.ld * sizeof(uint32_t));
  p.off_hist = off;
  off = align256(off + (size_t)Bq * kv->Hkv * 4096 * sizeof(uint32_t));
  p.total = off;
  return p;
}

struct SaPlan {
  bool stream;  // decode (bf16, FP8, FP4): persistent warp stream
  int nsplit;   // CUDA-core path: chunks of 128 entries of W ∪ S
  hs2::SaStreamArgs sp;
  int grid;
  size_t off_ml, off_o, off_arrive, total;
};

SaPlan sa_plan(int Bq, int Hq, const hs2_kv* kv, int w, int k, int prefill) {
  SaPlan p{};
  const int G = Hq / kv->Hkv;
  const bool bf16 = kv->dtype == HS2_BF16;
  size_t off = 0;
  const int kvt = bf16 ? 1 : kv->dtype == HS2_FP8_E4M3 ? 2 : kv->dtype == HS2_FP4_E2M1 ? 3 : 0;
  if (!prefill && hs2::sa_stream_plan(G, kv->d, kvt, w, k, Bq, kv->Hkv, &p.sp, &p.grid)) {
    p.stream = true;
    const size_t units = (size_t)Bq * kv->Hkv * p.sp.hg;
    const size_t slots = units * p.sp.maxc * 8;
    p.off_ml = off;
    off = align256(off + slots * sizeof(float) * 2);
    p.off_o = off;
    off = align256(off + slots * kv->d * sizeof(float));
    p.off_arrive = off;
    off = align256(off + units * sizeof(int32_t));
    p.total = off;
    return p;
  }
  if (hs2::sa_mma_supported(G, kv->d, bf16, w, k)) {  // no partials
    p.nsplit = 1;
    p.total = 256;
    return p;
  }
  p.nsplit = std::max(1, cdiv((long long)w + k, 128));
  p.off_ml = off;
  off = align256(off + (size_t)Bq * Hq * p.nsplit * sizeof(float) * 2);
  p.off_o = off;
  off = align256(off + (size_t)Bq * Hq * p.nsplit * kv->d * sizeof(float));
  p.total = off;
  return p;
}

// ---------------------------------------------------------------------------- CSA2 indexer layout
struct IdxPlan {
  long long ld_keys, ld_bkeys;
  size_t off_keys, off_bkeys, off_hist, total;
};

IdxPlan idx_plan(hs2_idx_mode mode, int B, int max_t, int max_blocks) {
  IdxPlan p{};
  p.ld_keys = mode == HS2_FULL ? ((long long)max_t + 63) / 64 * 64 : (long long)max_blocks * 8;
  p.ld_bkeys = ((long long)(max_t + 7) / 8 + 63) / 64 * 64;
  size_t off = 0;
  p.off_keys = off;
  off = align256(off + (size_t)B * p.ld_keys * 4);
  p.off_bkeys = off;
  off = align256(off + (size_t)B * p.ld_bkeys * 4);
  p.off_hist = off;
  off = align256(off + 2 * (size_t)B * 4096 * 4);
  p.total = off;
  return p;
}

// 2-D bf16 tensor map: rows x cols (cols contiguous), box of 64 columns x box_rows rows,
// 128-byte swizzle. cuTensorMapEncodeTiled is fetched from the driver at run time so the
// library has no link-time dependency on libcuda.
// rows x cols bf16, tiles of box_rows x 64 in the 128-byte swizzle. row_step > 1: a view of
// every row_step-th row (rows / row_step view rows, row stride row_step * cols * 2 bytes).
bool encode_2d_bf16(CUtensorMap* map, const void* base, uint64_t cols, uint64_t rows, uint32_t box_rows,
                    uint32_t row_step = 1) {
  static PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
  if (!encode) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !fn) {
      (void)cudaGetLastError();
      return false;
    }
    encode = (PFN_cuTensorMapEncodeTiled_v12000)fn;
  }
  const cuuint64_t dims[2] = {cols, rows / row_step};
  const cuuint64_t strides[1] = {cols * 2 * row_step};
  const cuuint32_t box[2] = {64, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_3d_bf16(CUtensorMap* map, const void* base, uint64_t d0, uint64_t d1, uint64_t d2, uint32_t b1,
                    uint32_t b2) {
  static PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
  if (!encode) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !fn) {
      (void)cudaGetLastError();
      return false;
    }
    encode = (PFN_cuTensorMapEncodeTiled_v12000)fn;
  }
  const cuuint64_t dims[3] = {d0, d1, d2};
  const cuuint64_t strides[2] = {d0 * 2, d0 * d1 * 2};
  const cuuint32_t box[3] = {64, b1, b2};
  const cuuint32_t estr[3] = {1, 1, 1};
  return encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// ---------------------------------------------------------------------------- bf16 prefill layout
bool use_prefill_tc(const hs2_kv* kv, int prefill) { return prefill && kv->dtype == HS2_BF16 && kv->d == 128; }

// Rows are ranked in chunks of kPrefillChunk rows (one scan launch per chunk; a single
// chunk keeps the heaviest-first schedule balanced); each chunk's candidate buffers hold
// cap entries per (row, KV head), cap = max(256, 4k).
constexpr int kPrefillChunk = 32768;

struct PrefillPlan {
  int chunk, cap;
  size_t off_lse2, off_ckey, off_cpos, off_ccnt, off_cdrop, off_ctau, off_redo_list, off_redo_cnt, off_redo_keys,
      total;
};

PrefillPlan prefill_plan(int n, int Hq, const hs2_kv* kv, int k) {
  PrefillPlan p{};
  p.chunk = std::max(1, std::min(n, kPrefillChunk));
  p.cap = std::max(256, 4 * k);
  const size_t rows = (size_t)p.chunk * kv->Hkv;
  size_t off = 0;
  p.off_lse2 = off;
  off = align256(off + (size_t)n * Hq * sizeof(float));
  p.off_ckey = off;
  off = align256(off + rows * p.cap * 4);
  p.off_cpos = off;
  off = align256(off + rows * p.cap * 4);
  p.off_ccnt = off;
  off = align256(off + rows * 4);
  p.off_cdrop = off;
  off = align256(off + rows * 4);
  p.off_ctau = off;
  off = align256(off + rows * 4);
  p.off_redo_list = off;  // rows the candidates cannot prove, completed exactly
  off = align256(off + rows * 4);
  p.off_redo_cnt = off;
  off = align256(off + 4);
  p.off_redo_keys = off;  // one key row of up to n far positions per completion CTA
  off = align256(off + (size_t)hs2::kPsCompleteCtas * n * 4);
  p.total = off;
  return p;
}

hs2_status common_checks(const void* q, int Bq, int Hq, const hs2_kv* kv, int prefill, bool need_v) {
  if (!valid_kv(kv, need_v)) return HS2_ERR_ARG;
  if (!q || !aligned16(q) || Bq < 0 || Hq < 1) return HS2_ERR_ARG;
  if (Hq % kv->Hkv != 0) return HS2_ERR_ARG;
  if (!pow2_le32(Hq / kv->Hkv)) return HS2_ERR_UNSUPPORTED;
  if (prefill) {
    if (kv->batch != 1) return HS2_ERR_ARG;
    if ((long long)Bq > (long long)kv->max_pages * 64) return HS2_ERR_ARG;
  } else if (Bq != kv->batch) {
    return HS2_ERR_ARG;
  }
  return HS2_OK;
}

}  // namespace

extern "C" {

int hs2_abi_version(void) { return HS2_ABI_VERSION; }

void hs2_profile_next(hs2_stage stage, void* start, void* stop) {
  if ((int)stage < 0 || (int)stage > 2) return;
  g_prof[stage][0] = start;
  g_prof[stage][1] = stop;
}

int hs2_last_cuda_error(void) { return g_last_cuda_error; }

const char* hs2_strerror(hs2_status st) {
  switch (st) {
    case HS2_OK: return "ok";
    case HS2_ERR_ARG: return "invalid argument";
    case HS2_ERR_UNSUPPORTED: return "unsupported configuration";
    case HS2_ERR_CUDA: return "CUDA launch or runtime error";
    case HS2_ERR_DEVICE: return "device-side error flag set";
    case HS2_ERR_SCRATCH_LIMIT: return "problem needs more scratch than the no-allocation entry point holds";
  }
  return "unknown status";
}

size_t hs2_fa_select_workspace(int B_or_n, int Hq, const hs2_kv* kv, int max_t, int k, int prefill) {
  if (!kv || kv->Hkv < 1 || Hq < 1 || max_t < 1 || B_or_n < 0 || (kv->d != 64 && kv->d != 128)) return 0;
  if (use_prefill_tc(kv, prefill)) return prefill_plan(B_or_n, Hq, kv, k).total;
  return fa_plan(B_or_n, Hq, kv, max_t).total;
}

static hs2_status fa_select_prefill_tc(const void* q, int n, int Hq, const hs2_kv* kv, int w, int k, float scale,
                                       float* o, float* lse, int32_t* idx, int32_t* idx_cnt, void* workspace,
                                       size_t ws_bytes, int32_t* dev_err, cudaStream_t s) {
  const PrefillPlan p = prefill_plan(n, Hq, kv, k);
  if (!workspace || ws_bytes < p.total || ((uintptr_t)workspace & 255u)) return HS2_ERR_ARG;
  const bool ranked = k > 0 && n - w > k;  // some row's far range exceeds the budget
  char* ws = (char*)workspace;
  CUtensorMap tq, tk, tv;
  const uint64_t rows = (uint64_t)kv->num_pages * kv->Hkv * 64;
  if (!encode_3d_bf16(&tq, q, 128, (uint64_t)Hq, (uint64_t)n, 1, 128) || !encode_2d_bf16(&tk, kv->k, 128, rows, 64) ||
      !encode_2d_bf16(&tv, kv->v, 128, rows, 64))
    return HS2_ERR_ARG;
  hs2::PfArgs a{};
  a.n = n;
  a.Hq = Hq;
  a.Hkv = kv->Hkv;
  a.G = Hq / kv->Hkv;
  a.bt = kv->block_table;
  a.max_pages = kv->max_pages;
  a.num_pages = kv->num_pages;
  a.seq_len = kv->seq_len;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.o = o;
  a.lse = lse;
  a.lse2 = (float*)(ws + p.off_lse2);
  a.dev_err = dev_err;
  cudaError_t e = profiled(HS2_STAGE_FA_SCAN, s, [&] { return hs2::launch_fa_prefill_fwd(tq, tk, tv, a, s); });
  if (e != cudaSuccess) return cuda_fail(e);
  if (!ranked) {
    // every row's far range is empty or fits the budget: each row takes all of it
    e = hs2::launch_prefill_trivial_select(idx, idx_cnt, n, kv->Hkv, w, k, s);
    if (e != cudaSuccess) return cuda_fail(e);
    return HS2_OK;
  }
  hs2::PsArgs b{};
  b.n = n;
  b.Hq = Hq;
  b.Hkv = kv->Hkv;
  b.G = Hq / kv->Hkv;
  b.w = w;
  b.k = k;
  b.cap = p.cap;
  b.bt = kv->block_table;
  b.max_pages = kv->max_pages;
  b.num_pages = kv->num_pages;
  b.seq_len = kv->seq_len;
  b.scale_log2 = a.scale_log2;
  b.lse2 = a.lse2;
  b.cand_key = (uint32_t*)(ws + p.off_ckey);
  b.cand_pos = (int32_t*)(ws + p.off_cpos);
  b.cand_cnt = (int32_t*)(ws + p.off_ccnt);
  b.cand_drop = (uint32_t*)(ws + p.off_cdrop);
  b.cand_tau = (uint32_t*)(ws + p.off_ctau);
  b.idx = idx;
  b.cnt = idx_cnt;
  b.q = q;
  b.kpool = kv->k;
  b.redo_list = (int32_t*)(ws + p.off_redo_list);
  b.redo_cnt = (int32_t*)(ws + p.off_redo_cnt);
  b.redo_keys = (uint32_t*)(ws + p.off_redo_keys);
  b.ld_redo = n;
  b.dev_err = dev_err;
  for (int r0 = 0; r0 < n; r0 += p.chunk) {
    e = cudaMemsetAsync(b.redo_cnt, 0, sizeof(int32_t), s);
    if (e != cudaSuccess) return cuda_fail(e);
    b.row0 = r0;
    b.row1 = std::min(n, r0 + p.chunk);
    // the sampled sweep of the selection scan reads every kPsSampleStride-th key only
    CUtensorMap tks;
    if (!encode_2d_bf16(&tks, kv->k, 128, rows, hs2::kPsSampleRowsPerPage, hs2::kPsSampleStride)) return HS2_ERR_ARG;
    e = hs2::launch_prefill_select(tq, tk, tks, b, s);
    if (e != cudaSuccess) return cuda_fail(e);
  }
  return HS2_OK;
}

int hs2_fa_select_launches(int B_or_n, int Hq, const hs2_kv* kv, int max_t, int w, int k, int prefill, int sel_block,
                           int append) {
  if (!kv || !valid_kv(kv, true) || Hq < 1 || Hq % kv->Hkv != 0 || !pow2_le32(Hq / kv->Hkv) || B_or_n < 0 || w < 0 ||
      k < 0 || max_t < 1 || sel_block < 1 || (append && prefill))
    return -1;
  if (B_or_n == 0) return 0;
  if (use_prefill_tc(kv, prefill)) {
    if (!(k > 0 && B_or_n - w > k)) return 2;  // forward + the all-of-F select
    const int chunks = cdiv(B_or_n, prefill_plan(B_or_n, Hq, kv, k).chunk);
    return 1 + 3 * chunks;  // forward; per chunk: candidate scan, top-k, completion
  }
  const FaPlan p = fa_plan(B_or_n, Hq, kv, max_t);
  int n = 1;  // the scan (tensor-core or CUDA-core)
  if (append && !(p.mma && kv->dtype == HS2_BF16)) n += 1;  // a separate append kernel
  hs2::CombineArgs c{};
  c.select = 1;
  c.sel_block = sel_block;
  c.prefill = prefill ? 1 : 0;
  c.gather = 0;
  c.Hkv = kv->Hkv;
  c.D = kv->d;
  return n + (hs2::score_select_fused(c, B_or_n) ? 1 : 2);  // fused, else merge + select
}

int hs2_sa_reuse_launches(int B_or_n, int Hq, const hs2_kv* kv, int w, int k, int prefill) {
  if (!kv || !valid_kv(kv, true) || Hq < 1 || Hq % kv->Hkv != 0 || !pow2_le32(Hq / kv->Hkv) || B_or_n < 0 || w < 0 ||
      k < 0)
    return -1;
  if (B_or_n == 0) return 0;
  const SaPlan p = sa_plan(B_or_n, Hq, kv, w, k, prefill);
  if (p.stream || hs2::sa_mma_supported(Hq / kv->Hkv, kv->d, kv->dtype == HS2_BF16, w, k)) return 1;
  return 2;  // partial attention + merge
}

hs2_status hs2_selftest_wait_timeout(int timeout_us, int32_t* dev_err, void* stream) {
  if (timeout_us < 1 || timeout_us > 2000000 || !dev_err) return HS2_ERR_ARG;
  cudaError_t e = hs2::launch_wait_selftest(dev_err, 1000ull * (unsigned long long)timeout_us, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e);
  return HS2_OK;
}

hs2_status hs2_fa_select(const void* q, int B_or_n, int Hq, const hs2_kv* kv, int max_t, int w, int k,
                         float scale, int prefill, float* o, float* lse, int32_t* idx, int32_t* idx_cnt,
                         void* workspace, size_t ws_bytes, int32_t* dev_err, void* stream) {
  return hs2_fa_select_ex(q, B_or_n, Hq, kv, max_t, w, k, scale, prefill, 1, o, lse, idx, idx_cnt, workspace,
                          ws_bytes, dev_err, stream);
}

static bool append_rows_ok(const hs2_kv* kv, const void* k_new, const void* v_new) {
  if (!valid_kv(kv, false) || !k_new || !aligned16(k_new)) return false;
  return !kv->v || (v_new && aligned16(v_new));
}

static hs2::AppendCache append_cache(const hs2_kv* kv, const void* k_new, const void* v_new) {
  hs2::AppendCache c{};
  c.k = const_cast<void*>(kv->k);  // the caller owns the pool; an append writes into it
  c.v = const_cast<void*>(kv->v);
  c.bt = kv->block_table;
  c.seq_len = kv->seq_len;
  c.k_new = k_new;
  c.v_new = kv->v ? v_new : nullptr;
  c.num_pages = kv->num_pages;
  c.max_pages = kv->max_pages;
  c.Hkv = kv->Hkv;
  c.row_bytes = kv->d * (kv->dtype == HS2_F32 ? 4 : 2);
  c.B = kv->batch;
  return c;
}

hs2_status hs2_kv_append(int n_caches, const hs2_kv* kvs, const void* const* k_new, const void* const* v_new,
                         int32_t* dev_err, void* stream) {
  if (n_caches < 1 || n_caches > hs2::kMaxAppendCaches || !kvs || !k_new) return HS2_ERR_ARG;
  hs2::AppendArgs a{};
  a.n = n_caches;
  a.dev_err = dev_err;
  for (int c = 0; c < n_caches; ++c) {
    const hs2_kv* kv = &kvs[c];
    const void* vn = v_new ? v_new[c] : nullptr;
    if (!append_rows_ok(kv, k_new[c], vn)) return HS2_ERR_ARG;
    if (low_precision(kv)) return HS2_ERR_UNSUPPORTED;
    a.c[c] = append_cache(kv, k_new[c], vn);
    a.B = std::max(a.B, (int)kv->batch);
  }
  cudaError_t e = hs2::launch_kv_append(a, (cudaStream_t)stream);
  return e == cudaSuccess ? HS2_OK : cuda_fail(e);
}

static hs2_status fa_select_impl(const void* q, int B_or_n, int Hq, const hs2_kv* kv, int max_t, int w, int k,
                                 float scale, int prefill, int sel_block, const void* k_new, const void* v_new,
                                 float* o, float* lse, int32_t* idx, int32_t* idx_cnt, void* workspace,
                                 size_t ws_bytes, int32_t* dev_err, void* stream) {
  hs2_status st = common_checks(q, B_or_n, Hq, kv, prefill, true);
  if (st != HS2_OK) return st;
  if (w < 0 || k < 0 || max_t < 1 || !std::isfinite(scale)) return HS2_ERR_ARG;
  if (sel_block < 1 || sel_block > 4096 || (sel_block > 1 && (sel_block % 4 != 0 || k % sel_block != 0)))
    return HS2_ERR_ARG;
  if (sel_block > 1 && prefill) return HS2_ERR_UNSUPPORTED;
  if (low_precision(kv) && prefill) return HS2_ERR_UNSUPPORTED;  // FP8 / FP4 caches: decode only
  if ((long long)max_t > (long long)kv->max_pages * 64) return HS2_ERR_ARG;
  if (prefill && B_or_n > max_t) return HS2_ERR_ARG;
  if (!o || !idx_cnt || (k > 0 && !idx)) return HS2_ERR_ARG;
  if (B_or_n == 0) return HS2_OK;
  if (use_prefill_tc(kv, prefill))
    return fa_select_prefill_tc(q, B_or_n, Hq, kv, w, k, scale, o, lse, idx, idx_cnt, workspace, ws_bytes, dev_err,
                                (cudaStream_t)stream);
  const FaPlan p = fa_plan(B_or_n, Hq, kv, max_t);
  if (!workspace || ws_bytes < p.total || ((uintptr_t)workspace & 255u)) return HS2_ERR_ARG;
  cudaStream_t s = (cudaStream_t)stream;
  char* ws = (char*)workspace;
  // the current token's rows: fused into the bf16 tensor-core scan, else appended first
  const bool fused_append = k_new && p.mma && kv->dtype == HS2_BF16;
  if (k_new && !fused_append) {
    hs2::AppendArgs ap{};
    ap.n = 1;
    ap.B = B_or_n;
    ap.dev_err = dev_err;
    ap.c[0] = append_cache(kv, k_new, v_new);
    cudaError_t e = hs2::launch_kv_append(ap, s);
    if (e != cudaSuccess) return cuda_fail(e);
  }

  hs2::AttnArgs a{};
  a.q = q;
  if (fused_append) {
    a.k_new = k_new;
    a.v_new = v_new;
  }
  a.Hq = Hq;
  a.G = Hq / kv->Hkv;
  a.D = kv->d;
  a.k = kv->k;
  a.v = kv->v;
  a.bt = kv->block_table;
  a.seq_len = kv->seq_len;
  a.max_pages = kv->max_pages;
  a.num_pages = kv->num_pages;
  a.Hkv = kv->Hkv;
  a.max_t = max_t;
  a.prefill = prefill ? 1 : 0;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.gather = 0;
  a.pps = p.pps;
  a.nsplit = p.nsplit;
  a.part_ml = (float2*)(ws + p.off_ml);
  a.part_o = (float*)(ws + p.off_o);
  a.lcode = (uint16_t*)(ws + p.off_lcode);
  a.lmax = (float*)(ws + p.off_lmax);
  a.ld_logits = p.ld;
  if (low_precision(kv)) {
    if (!p.mma) return HS2_ERR_UNSUPPORTED;
    a.k_scale = kv->k_scale;
    a.v_scale = kv->v_scale;
    a.k_sf = kv->k_sf;
    a.v_sf = kv->v_sf;
  }
  a.dev_err = dev_err;
  cudaError_t e = profiled(HS2_STAGE_FA_SCAN, s, [&] {
    return p.mma ? hs2::launch_fa_decode_mma(a, B_or_n, s)
                 : hs2::launch_attn_partial(a, B_or_n, kv->dtype == HS2_BF16, s);
  });
  if (e != cudaSuccess) return cuda_fail(e);

  hs2::CombineArgs c{};
  c.part_ml = a.part_ml;
  c.part_o = a.part_o;
  c.nsplit = p.nsplit;
  c.G = a.G;
  c.Hq = Hq;
  c.Hkv = kv->Hkv;
  c.D = kv->d;
  c.prefill = a.prefill;
  c.seq_len = kv->seq_len;
  c.max_pages = kv->max_pages;
  c.max_t = max_t;
  c.gather = 0;
  c.w = w;
  c.pps = p.pps;
  c.o = o;
  c.lse = lse;
  c.select = 1;
  c.sel_block = sel_block;
  c.k = k;
  c.kcap = k;
  c.idx = idx;
  c.cnt = idx_cnt;
  c.lcode = a.lcode;
  c.lmax = a.lmax;
  c.scores = (uint32_t*)(ws + p.off_scores);
  c.hist = (uint32_t*)(ws + p.off_hist);
  c.ld_logits = p.ld;
  c.dev_err = dev_err;
  if (!hs2::score_select_fused(c, B_or_n)) {  // the fused kernel keeps its histogram in shared memory
    e = cudaMemsetAsync(c.hist, 0, (size_t)B_or_n * kv->Hkv * 4096 * sizeof(uint32_t), s);
    if (e != cudaSuccess) return cuda_fail(e);
  }
  e = hs2::launch_combine(c, B_or_n, s);
  if (e != cudaSuccess) return cuda_fail(e);
  return HS2_OK;
}

hs2_status hs2_fa_select_ex(const void* q, int B_or_n, int Hq, const hs2_kv* kv, int max_t, int w, int k,
                            float scale, int prefill, int sel_block, float* o, float* lse, int32_t* idx,
                            int32_t* idx_cnt, void* workspace, size_t ws_bytes, int32_t* dev_err, void* stream) {
  return fa_select_impl(q, B_or_n, Hq, kv, max_t, w, k, scale, prefill, sel_block, nullptr, nullptr, o, lse, idx,
                        idx_cnt, workspace, ws_bytes, dev_err, stream);
}

hs2_status hs2_fa_select_append(const void* q, int B, int Hq, const hs2_kv* kv, int max_t, int w, int k, float scale,
                                int sel_block, const void* k_new, const void* v_new, float* o, float* lse,
                                int32_t* idx, int32_t* idx_cnt, void* workspace, size_t ws_bytes, int32_t* dev_err,
                                void* stream) {
  if (!kv || !append_rows_ok(kv, k_new, v_new) || !kv->v) return HS2_ERR_ARG;
  if (low_precision(kv)) return HS2_ERR_UNSUPPORTED;
  return fa_select_impl(q, B, Hq, kv, max_t, w, k, scale, 0, sel_block, k_new, v_new, o, lse, idx, idx_cnt, workspace,
                        ws_bytes, dev_err, stream);
}

size_t hs2_sa_reuse_workspace(int B_or_n, int Hq, const hs2_kv* kv, int w, int k, int prefill) {
  if (!kv || kv->Hkv < 1 || Hq < 1 || B_or_n < 0 || w < 0 || k < 0 || (kv->d != 64 && kv->d != 128)) return 0;
  return sa_plan(B_or_n, Hq, kv, w, k, prefill).total;
}

hs2_status hs2_sa_reuse(const void* q, int B_or_n, int Hq, const hs2_kv* kv, int w, const int32_t* idx,
                        const int32_t* idx_cnt, int k, float scale, int prefill, float* o, void* workspace,
                        size_t ws_bytes, int32_t* dev_err, void* stream) {
  return hs2_sa_reuse_ex(q, B_or_n, Hq, kv, w, idx, idx_cnt, k, scale, prefill, nullptr, nullptr, 0, o, workspace,
                         ws_bytes, dev_err, stream);
}

hs2_status hs2_sa_reuse_ex(const void* q, int B_or_n, int Hq, const hs2_kv* kv, int w, const int32_t* idx,
                           const int32_t* idx_cnt, int k, float scale, int prefill, const float* sink,
                           const float* gate, int flags, float* o, void* workspace, size_t ws_bytes,
                           int32_t* dev_err, void* stream) {
  hs2_status st = common_checks(q, B_or_n, Hq, kv, prefill, true);
  if (st != HS2_OK) return st;
  if (w < 0 || k < 0 || !std::isfinite(scale) || !o || !idx_cnt || (k > 0 && !idx)) return HS2_ERR_ARG;
  if (flags & ~HS2_SA_OVERLAP) return HS2_ERR_ARG;
  if (B_or_n == 0) return HS2_OK;
  const SaPlan p = sa_plan(B_or_n, Hq, kv, w, k, prefill);
  if (low_precision(kv) && !p.stream) return HS2_ERR_UNSUPPORTED;  // FP8 / FP4: the decode stream only
  if (!workspace || ws_bytes < p.total || ((uintptr_t)workspace & 255u)) return HS2_ERR_ARG;
  cudaStream_t s = (cudaStream_t)stream;
  char* ws = (char*)workspace;

  hs2::AttnArgs a{};
  a.q = q;
  a.Hq = Hq;
  a.G = Hq / kv->Hkv;
  a.D = kv->d;
  a.k = kv->k;
  a.v = kv->v;
  a.bt = kv->block_table;
  a.seq_len = kv->seq_len;
  a.max_pages = kv->max_pages;
  a.num_pages = kv->num_pages;
  a.Hkv = kv->Hkv;
  a.max_t = prefill ? B_or_n : kv->max_pages * 64;
  a.prefill = prefill ? 1 : 0;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.gather = 1;
  a.pps = 1;
  a.nsplit = p.nsplit;
  a.w = w;
  a.idx = idx;
  a.cnt = idx_cnt;
  a.kcap = k;
  a.part_ml = (float2*)(ws + p.off_ml);
  a.part_o = (float*)(ws + p.off_o);
  a.lcode = nullptr;
  a.lmax = nullptr;
  a.out_o = o;
  a.sink = sink;
  a.gate = gate;
  if (low_precision(kv)) {
    a.k_scale = kv->k_scale;
    a.v_scale = kv->v_scale;
    a.k_sf = kv->k_sf;
    a.v_sf = kv->v_sf;
  }
  a.dev_err = dev_err;
  if (p.stream) {
    // decode (bf16, FP8, FP4): one persistent warp stream over all (query, KV head) pairs' entries
    // the counters start at zero; an HS2_SA_OVERLAP call takes them as the SA call before it
    // on this workspace left them (zero), so it is a single launch whose row resolve can
    // overlap the end of that call's kernel
    a.arrive = (int32_t*)(ws + p.off_arrive);
    hs2::SaStreamArgs sp = p.sp;
    sp.early = (flags & HS2_SA_OVERLAP) ? 1 : 0;
    if (!sp.early) {
      cudaError_t e = cudaMemsetAsync(a.arrive, 0, (size_t)B_or_n * kv->Hkv * p.sp.hg * sizeof(int32_t), s);
      if (e != cudaSuccess) return cuda_fail(e);
    }
    cudaError_t e = profiled(HS2_STAGE_SA_GATHER, s, [&] { return hs2::launch_sa_stream(a, sp, p.grid, s); });
    if (e != cudaSuccess) return cuda_fail(e);
    return HS2_OK;
  }
  if (hs2::sa_mma_supported(a.G, a.D, kv->dtype == HS2_BF16, w, k)) {
    // bf16: per-row gathered Q.K and P.V over the heads sharing a KV head are small dense
    // contractions -> mma.sync; decode splits each row over a thread-block cluster
    cudaError_t e = profiled(HS2_STAGE_SA_GATHER, s, [&] { return hs2::launch_sa_mma(a, B_or_n, s); });
    if (e != cudaSuccess) return cuda_fail(e);
    return HS2_OK;
  }
  cudaError_t e = profiled(HS2_STAGE_SA_GATHER, s,
                           [&] { return hs2::launch_attn_partial(a, B_or_n, kv->dtype == HS2_BF16, s); });
  if (e != cudaSuccess) return cuda_fail(e);

  hs2::CombineArgs c{};
  c.part_ml = a.part_ml;
  c.part_o = a.part_o;
  c.nsplit = p.nsplit;
  c.G = a.G;
  c.Hq = Hq;
  c.Hkv = kv->Hkv;
  c.D = kv->d;
  c.prefill = a.prefill;
  c.seq_len = kv->seq_len;
  c.max_pages = kv->max_pages;
  c.max_t = a.max_t;
  c.gather = 1;
  c.w = w;
  c.sa_cnt = idx_cnt;
  c.kcap = k;
  c.o = o;
  c.sink = sink;
  c.gate = gate;
  c.select = 0;
  c.dev_err = dev_err;
  e = hs2::launch_combine(c, B_or_n, s);
  if (e != cudaSuccess) return cuda_fail(e);
  return HS2_OK;
}

size_t hs2_hier_reindex_workspace(hs2_idx_mode mode, int Hi, const hs2_kv* k_idx, int max_t, int k_top,
                                  int blk, int max_blocks) {
  (void)Hi;
  (void)k_top;
  (void)blk;
  if (!k_idx || k_idx->batch < 1 || max_t < 1 || max_blocks < 1) return 0;
  return idx_plan(mode, k_idx->batch, max_t, max_blocks).total;
}

hs2_status hs2_hier_reindex(hs2_idx_mode mode, const void* q_idx, const float* w_idx, int Hi,
                            const hs2_kv* k_idx, int max_t, int k_top, int blk, int max_blocks,
                            int32_t* pool_blocks, int32_t* pool_cnt, int32_t* idx, int32_t* idx_cnt,
                            void* workspace, size_t ws_bytes, int32_t* dev_err, void* stream) {
  if (mode != HS2_FULL && mode != HS2_REINDEX) return HS2_ERR_ARG;
  if (!valid_kv(k_idx, false) || !q_idx || !aligned16(q_idx) || !w_idx) return HS2_ERR_ARG;
  if (max_t < 1 || (long long)max_t > (long long)k_idx->max_pages * 64 || k_top < 0 || max_blocks < 1) return HS2_ERR_ARG;
  if (!pool_blocks || !pool_cnt || !idx_cnt || (k_top > 0 && !idx)) return HS2_ERR_ARG;
  if (Hi != 64 || k_idx->d != 128 || k_idx->Hkv != 1 || k_idx->dtype != HS2_BF16 || blk != 8) return HS2_ERR_UNSUPPORTED;
  const IdxPlan p = idx_plan(mode, k_idx->batch, max_t, max_blocks);
  if (!workspace || ws_bytes < p.total || ((uintptr_t)workspace & 255u)) return HS2_ERR_ARG;
  cudaStream_t s = (cudaStream_t)stream;
  char* ws = (char*)workspace;
  const int B = k_idx->batch;

  CUtensorMap tm_k, tm_q;
  const int box_rows = mode == HS2_FULL ? 64 : 8;
  if (!encode_2d_bf16(&tm_k, k_idx->k, 128, (uint64_t)k_idx->num_pages * 64, box_rows) ||
      !encode_2d_bf16(&tm_q, q_idx, 128, (uint64_t)B * 64, 64))
    return HS2_ERR_ARG;
  cudaError_t e = cudaMemsetAsync(ws + p.off_hist, 0, 2 * (size_t)B * 4096 * sizeof(uint32_t), s);
  if (e != cudaSuccess) return cuda_fail(e);

  hs2::IdxArgs a{};
  a.mode = mode == HS2_FULL ? 0 : 1;
  a.w_idx = w_idx;
  a.bt = k_idx->block_table;
  a.seq_len = k_idx->seq_len;
  a.max_pages = k_idx->max_pages;
  a.num_pages = k_idx->num_pages;
  a.max_t = max_t;
  a.pool = pool_blocks;
  a.pool_cnt = pool_cnt;
  a.max_blocks = max_blocks;
  a.keys = (uint32_t*)(ws + p.off_keys);
  a.ld_keys = p.ld_keys;
  a.bkeys = (uint32_t*)(ws + p.off_bkeys);
  a.ld_bkeys = p.ld_bkeys;
  a.hist = (uint32_t*)(ws + p.off_hist);
  a.bhist = a.hist + (size_t)B * 4096;
  a.dev_err = dev_err;
  const long long ntile_max = (p.ld_keys + 127) / 128;
  // one wave of 152 SMs (one CTA per SM) over every batch row
  const long long per_cta = std::max<long long>(1, (ntile_max * B + 151) / 152);
  a.tiles_per_cta = (int)per_cta;
  const int grid_x = (int)((ntile_max + per_cta - 1) / per_cta);
  e = profiled(HS2_STAGE_INDEXER, s, [&] { return hs2::launch_lightning_scan(tm_k, tm_q, a, B, grid_x, s); });
  if (e != cudaSuccess) return cuda_fail(e);

  hs2::SelectArgs sa{};
  sa.seq_len = k_idx->seq_len;
  sa.max_t = max_t;
  sa.max_pages = k_idx->max_pages;
  sa.pool = pool_blocks;
  sa.pool_cnt = pool_cnt;
  sa.max_blocks = max_blocks;
  sa.dev_err = dev_err;
  sa.mode = mode == HS2_FULL ? 1 : 3;
  sa.k = k_top;
  sa.kcap = k_top;
  sa.keys = a.keys;
  sa.ld_keys = p.ld_keys;
  sa.hist = a.hist;
  sa.out = idx;
  sa.cnt = idx_cnt;
  hs2::SelectJobs jobs{};
  jobs.job[0] = sa;
  jobs.n = 1;
  if (mode == HS2_FULL) {  // the pool's block selection runs in the same launch
    sa.mode = 2;
    sa.k = max_blocks;
    sa.kcap = max_blocks;
    sa.keys = a.bkeys;
    sa.ld_keys = p.ld_bkeys;
    sa.hist = a.bhist;
    sa.out = pool_blocks;
    sa.cnt = pool_cnt;
    jobs.job[1] = sa;
    jobs.n = 2;
  }
  e = hs2::launch_select_rows(jobs, B, s);
  if (e != cudaSuccess) return cuda_fail(e);
  return HS2_OK;
}

}  // extern "C"

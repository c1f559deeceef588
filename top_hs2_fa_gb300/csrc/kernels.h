// kernels.h — launch parameters shared between the C ABI layer and the kernels.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace hs2 {

// Launch with programmatic stream serialization: the kernel may begin while the previous
// launch on the stream finishes, so it must call griddep_wait before reading anything that
// launch may write (and griddep_launch_dependents to let the next one begin early).
template <typename... Params, typename... Args>
inline cudaError_t launch_pdl(void (*kern)(Params...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                              Args&&... args) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, static_cast<Args&&>(args)...);
  return e != cudaSuccess ? e : cudaGetLastError();
}

constexpr int kCombineThreads = 512;

// One attention pass over a set of rows of one group's paged KV, producing per
// (query, head, chunk) partial softmax state (m, l in base 2; unnormalised o).
struct AttnArgs {
  const void* q;  // [Bq][Hq][D], kv dtype
  int Hq, G, D;
  const void* k;
  const void* v;
  const int32_t* bt;
  const int32_t* seq_len;
  int max_pages, num_pages, Hkv;
  int max_t;         // host-declared bound on t; longer queries are flagged and skipped
  int prefill;       // 1: query qi is causal row qi of sequence 0 (t = qi + 1)
  float scale_log2;  // softmax scale * log2(e)
  int gather;        // 0: rows = split of pps pages (FA); 1: rows = W(t) ∪ S(t) (SA)
  int pps;           // pages per split (FA)
  int nsplit;        // chunk stride of the partial arrays
  int w;
  const int32_t* idx;  // [Bq][Hkv][kcap] (SA)
  const int32_t* cnt;  // [Bq][Hkv] (SA)
  int kcap;
  float2* part_ml;  // [Bq][Hq][nsplit]
  float* part_o;    // [Bq][Hq][nsplit][D]
  uint16_t* lcode;  // [Bq][Hq][ld_logits] selection logits as codes below their group max (logit_code), or null
  float* lmax;      // [Bq][Hq][ld_logits / 16] each 16-key group's max base-2 logit
  float* out_o;     // [Bq][Hq][D] final output (kernels that normalise in place)
  int32_t* arrive;  // SA stream: per-unit arrival counters, zero at launch (the merges leave them zero)
  const float* k_scale;  // FP8 cache: [num_pages][Hkv] dequantisation scales, else null
  const float* v_scale;
  const uint8_t* k_sf;  // FP4 cache: [num_pages][Hkv][64][D/16] E4M3 scales of 16 channels, else null
  const uint8_t* v_sf;
  const float* sink;  // SA: [Hq] sink logits (natural log), or null
  const float* gate;  // SA: [Bq][Hq][D] output gate logits, or null
  const void* k_new;  // decode FA with a fused append: [Bq][Hkv][D] rows of key t-1, or null
  const void* v_new;
  long long ld_logits;
  int32_t* dev_err;
};

// Decode KV append over up to kMaxAppendCaches independent caches in one launch.
constexpr int kMaxAppendCaches = 8;
struct AppendCache {
  void* k;
  void* v;  // null: a key-only cache
  const int32_t* bt;
  const int32_t* seq_len;
  const void* k_new;  // [B][Hkv][row_bytes]
  const void* v_new;
  int num_pages, max_pages, Hkv, row_bytes, B;
};
struct AppendArgs {
  AppendCache c[kMaxAppendCaches];
  int n, B;  // B: the largest batch of the caches
  int32_t* dev_err;
};

// Decode SA stream: units = (row, KV head, group of 8 query heads), hg groups per pair;
// `total` = units * ms steps of 16 entries cut into nwarps equal ranges; partials hold up
// to maxc warps per unit, 8 heads each.
struct SaStreamArgs {
  int nwarps, hg, ms, maxc;
  long long total;
  int early;  // resolve rows before waiting on the previous launch
};

struct CombineArgs {
  const float2* part_ml;
  const float* part_o;
  int nsplit, G, Hq, Hkv, D;
  int prefill;
  const int32_t* seq_len;
  int max_pages;
  int max_t;
  int gather;  // partials are SA chunks of 128 rows of W ∪ S (1) or FA splits of pps pages (0)
  int w;
  const int32_t* sa_cnt;  // SA: [Bq][Hkv] selected counts
  int pps;
  float* o;    // [Bq][Hq][D]
  float* lse;  // [Bq][Hq] natural log, or null
  const float* sink;  // SA partials: [Hq] sink logits, or null
  const float* gate;  // SA partials: [Bq][Hq][D] output gate logits, or null
  int select;  // 1: run the window-excluding top-k from the logits
  int sel_block;  // 1: token-level selection; > 1: whole blocks of that many far positions
  int k, kcap;
  int32_t* idx;  // [Bq][Hkv][kcap]
  int32_t* cnt;  // [Bq][Hkv]
  const uint16_t* lcode;  // [Bq][Hq][ld_logits] logit codes and [Bq][Hq][ld_logits / 16] group maxima
  const float* lmax;
  uint32_t* scores;  // [Bq][Hkv][ld_logits] selection keys (scratch)
  uint32_t* hist;    // [Bq][Hkv][4096] top-digit histograms (scratch, zeroed per call)
  long long ld_logits;
  int32_t* dev_err;
};

// CSA2 lightning-indexer scan (mode 0: every position s < t; mode 1: the pool's positions).
struct IdxArgs {
  int mode;
  const float* w_idx;  // [B][64]
  const int32_t* bt;
  const int32_t* seq_len;
  int max_pages, num_pages, max_t;
  int tiles_per_cta;
  const int32_t* pool;      // [B][max_blocks] (mode 1)
  const int32_t* pool_cnt;  // [B] (mode 1)
  int max_blocks;
  uint32_t* keys;  // [B][ld_keys] candidate keys
  long long ld_keys;
  uint32_t* bkeys;  // [B][ld_bkeys] 8-block maxima (mode 0)
  long long ld_bkeys;
  uint32_t* hist;   // [B][4096]
  uint32_t* bhist;  // [B][4096] (mode 0)
  int32_t* dev_err;
};

// Causal FA forward of one sequence's n query rows (bf16, head_dim 128, tcgen05).
struct PfArgs {
  int n, Hq, Hkv, G;
  const int32_t* bt;  // block table row of the sequence
  int max_pages, num_pages;
  const int32_t* seq_len;  // [1]
  float scale_log2;
  float* o;     // [n][Hq][128]
  float* lse;   // [n][Hq] natural log, or null
  float* lse2;  // [n][Hq] base-2 (scratch for the selection)
  int32_t* dev_err;
};

// Window-excluding top-k of the causal rows [row0, row1) of a bf16 prefill.
struct PsArgs {
  int n, row0, row1, Hq, Hkv, G, w, k, cap;
  const int32_t* bt;
  int max_pages, num_pages;
  const int32_t* seq_len;
  float scale_log2;
  const float* lse2;    // [n][Hq] base-2 lse from the forward kernel
  uint32_t* cand_key;   // [(row1-row0)][Hkv][cap]
  int32_t* cand_pos;    // [(row1-row0)][Hkv][cap]
  int32_t* cand_cnt;    // [(row1-row0)][Hkv]
  uint32_t* cand_drop;  // [(row1-row0)][Hkv] largest key dropped past capacity
  uint32_t* cand_tau;   // [(row1-row0)][Hkv] threshold (diagnostic)
  int32_t* idx;         // [n][Hkv][k]
  int32_t* cnt;         // [n][Hkv]
  // completion of the rows the candidates cannot prove: their (row - row0) * Hkv + g go to
  // redo_list (redo_cnt zeroed before the scan), and each CTA of the completion pass keeps
  // one row's exact keys in redo_keys + blockIdx.x * ld_redo
  const void* q;        // [n][Hq][128] bf16 queries
  const void* kpool;    // [num_pages][Hkv][64][128] bf16 keys
  int32_t* redo_list;   // [(row1-row0)][Hkv]
  int32_t* redo_cnt;    // [1]
  uint32_t* redo_keys;  // [kPsCompleteCtas][ld_redo]
  long long ld_redo;
  int32_t* dev_err;
};

// CTAs of the prefill selection's completion pass (each takes flagged rows in turn).
constexpr int kPsCompleteCtas = 304;

// Row-wise exact top-k over precomputed keys, starting from a global top-digit histogram.
struct SelectArgs {
  int mode;  // 1: positions [0, t); 2: 8-blocks [0, ceil(t/8)); 3: pool candidates (mapped)
  const int32_t* seq_len;
  int max_t, max_pages;
  const int32_t* pool;
  const int32_t* pool_cnt;
  int max_blocks;
  int k, kcap;
  const uint32_t* keys;
  long long ld_keys;
  const uint32_t* hist;
  int32_t* out;  // [B][kcap]
  int32_t* cnt;  // [B]
  int32_t* dev_err;
};

cudaError_t launch_fa_decode_mma(const AttnArgs& a, int Bq, cudaStream_t s);
cudaError_t launch_kv_append(const AppendArgs& a, cudaStream_t s);
cudaError_t launch_attn_partial(const AttnArgs& a, int Bq, int bf16, cudaStream_t s);
cudaError_t launch_combine(const CombineArgs& a, int Bq, cudaStream_t s);
// Whether launch_combine runs the fused merge + score + top-k kernel (which needs no
// zeroed global histogram) for these arguments.
bool score_select_fused(const CombineArgs& a, int Bq);
bool sa_mma_supported(int G, int D, int bf16, int w, int k);
// Decode: plan the warp stream on the current device (false if it does not apply);
// a.part_ml / a.part_o hold [units][maxc][8] partials and a.arrive [units] zeroed counters
// (the kernel's merges leave them zero again).
bool sa_stream_plan(int G, int D, int kv_dtype, int w, int k, int Bq, int Hkv, SaStreamArgs* sp, int* grid);
cudaError_t launch_sa_stream(const AttnArgs& a, const SaStreamArgs& sp, int grid, cudaStream_t s);
cudaError_t launch_sa_mma(const AttnArgs& a, int Bq, cudaStream_t s);
size_t lightning_scan_smem();
cudaError_t launch_lightning_scan(const CUtensorMap& tm_k, const CUtensorMap& tm_q, const IdxArgs& a, int B,
                                  int grid_x, cudaStream_t s);
// Independent selections over the same batch in one launch (grid y = job).
constexpr int kMaxSelectJobs = 2;
struct SelectJobs {
  SelectArgs job[kMaxSelectJobs];
  int n;
};
cudaError_t launch_select_rows(const SelectJobs& jobs, int B, cudaStream_t s);
cudaError_t launch_prefill_trivial_select(int32_t* idx, int32_t* cnt, int n, int Hkv, int w, int k, cudaStream_t s);
size_t fa_prefill_fwd_smem();
size_t prefill_scan_smem();
// The selection scan's sampled sweep: every kPsSampleStride-th key, through a tensor map of
// those rows only (box: the kPsSampleRowsPerPage sampled rows of a 64-row page).
constexpr int kPsSampleStride = 8;
constexpr int kPsSampleRowsPerPage = 64 / kPsSampleStride;
cudaError_t launch_prefill_select(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tks,
                                  const PsArgs& a, cudaStream_t s);
cudaError_t launch_fa_prefill_fwd(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const PfArgs& a,
                                  cudaStream_t s);

cudaError_t launch_wait_selftest(int32_t* dev_err, unsigned long long limit_ns, cudaStream_t s);

}  // namespace hs2

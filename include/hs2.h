/*
 * hs2.h — C ABI of the group-shared top-k sparse attention library (libhs2).
 *
 * One Cross group of a HySparse2 model = one FA layer + its SA layers over one
 * shared paged KV cache. The FA layer attends causally to every visible key and
 * emits, per query and KV head, the top-k positions outside a forced recent
 * window; each SA layer reuses that KV and those positions with its own query,
 * attending to window ∪ top-k under one softmax. The CSA2 variant replaces the
 * FA selection by a hierarchical lightning indexer (Full / Reindex / Reuse).
 *
 * Pages this interface restates (cited by title and section):
 *   [HS2]  "HySparse2：整体架构、KV 生命周期与 PD 分离"
 *          §5 (KV Reuse), §7.1-7.4 (forced window + out-of-window top-k, one
 *          normalisation, direct access to paged KV).
 *   [CSA2] "2.3.1 · CSA、HCA 与 CSA2: 压缩序列上的稀疏检索和跨层复用"
 *          §3.1 (Full / Reindex / Reuse), §3.2 (hierarchical sparse indexer).
 *   [L10]  "Lecture 10 · 混合架构与稀疏注意力：Mamba、Marconi 与 DeepSeek-V3.2"
 *          §5.1 (lightning indexer score), §5.5 (paged gather through a block table).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - Positions are 0-based. A query that sees t keys sits at position t-1; its
 *   own key is already in the cache. Window W(t) = [max(0,t-w), t-1]; far range
 *   F(t) = [0, t-w-1]; the FA selects min(k, max(0, t-w)) positions of F(t).
 * - GQA: query head h reads KV head g = h / (Hq / Hkv).
 * - All pointers are DEVICE pointers unless stated otherwise. The caller owns
 *   every buffer (inputs, outputs, workspace, dev_err). The library never
 *   allocates, frees or synchronises; every call is asynchronous on `stream`
 *   (a cudaStream_t passed as void*; NULL = the legacy default stream).
 * - Return value: host-side validation and launch status. HS2_ERR_ARG means
 *   nothing was launched. HS2_ERR_CUDA means a launch failed (the CUDA error is
 *   cleared and reported by hs2_last_cuda_error()).
 * - dev_err (optional, may be NULL): int32 device word the kernels OR error bits
 *   into (HS2_DEV_*) when they meet an out-of-range block-table entry or index,
 *   or give up a bounded wait. Bad accesses are skipped, never performed. The
 *   caller zeroes it and reads it after synchronising.
 * - Outputs are float32 whatever the input dtype (fp32 accumulation).
 * - Index sets are written sorted ascending, padded with -1, with a count array.
 *   Among equal scores the lower position (or lower block id) wins.
 */
#ifndef HS2_H
#define HS2_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define HS2_ABI_VERSION 6

typedef enum {
  HS2_OK = 0,
  HS2_ERR_ARG = -1,         /* invalid shape, pointer, alignment or workspace size */
  HS2_ERR_UNSUPPORTED = -2, /* valid but not implemented combination (e.g. head_dim 96) */
  HS2_ERR_CUDA = -3,        /* a CUDA launch / runtime call failed */
  HS2_ERR_DEVICE = -4,      /* reserved for callers that fold dev_err into a status */
  HS2_ERR_SCRATCH_LIMIT = -5 /* problem needs more scratch than hs2_fa_select_noalloc holds */
} hs2_status;

/* device-side error bits (ORed into *dev_err) */
#define HS2_DEV_BAD_PAGE 1    /* block-table entry outside [0, num_pages) */
#define HS2_DEV_BAD_INDEX 2   /* selected position outside F(t) (or outside [0,t) with w=0) */
#define HS2_DEV_TIMEOUT 4     /* a bounded wait (mbarrier / TMA / MMA) gave up */
#define HS2_DEV_BAD_LENGTH 8  /* seq_len < 1 or beyond max_pages * page_size */
#define HS2_DEV_SELECT 16     /* reserved: no longer raised. A prefill row whose streamed
                                 candidates cannot prove its top-k is recomputed exactly over
                                 its whole far range inside hs2_fa_select */

typedef enum { HS2_F32 = 0, HS2_BF16 = 1, HS2_FP8_E4M3 = 2, HS2_FP4_E2M1 = 3 } hs2_dtype;

/* Paged KV of ONE group, shared by its FA and SA layers ([HS2] §5, §7.2).
 * k, v:        [num_pages][Hkv][page_size][d] elements of `dtype`, 16-byte aligned.
 *              v may be NULL for an indexer-key cache (hs2_hier_reindex).
 * block_table: int32 [batch][max_pages]; entry j of sequence b is the physical page
 *              holding logical positions [j*page_size, (j+1)*page_size).
 * seq_len:     int32 [batch], keys visible to the query (its own included), >= 1.
 * k_scale, v_scale: HS2_FP8_E4M3 and HS2_FP4_E2M1 only (else NULL): float32
 *              [num_pages][Hkv]; FP8: a stored E4M3 code c of page p, KV head g stands for
 *              c * scale[p][g].
 * k_sf, v_sf:  HS2_FP4_E2M1 only (else NULL): uint8 E4M3 codes [num_pages][Hkv][page_size]
 *              [d/16], one per 16 channels of a row ([CSA2] §3, "KV 字节与 FP4": E2M1 main KV
 *              with an E4M3 scale per 16 channels). k and v then hold [num_pages][Hkv]
 *              [page_size][d/2] bytes, channel 2i in the low nibble of byte i (E2M1: sign,
 *              2 exponent bits with bias 1, 1 mantissa bit); channel c of a row stands for
 *              e2m1(code) * e4m3(sf[c / 16]) * scale[p][g].
 *              FP8 and FP4 caches are read by hs2_fa_select (decode) and hs2_sa_reuse
 *              (decode); queries are bf16; prefill and the KV append refuse them.
 * page_size must be 64; d must be 64 or 128.                                        */
typedef struct {
  const void* k;
  const void* v;
  const int32_t* block_table;
  const int32_t* seq_len;
  int32_t batch;
  int32_t num_pages;
  int32_t max_pages;
  int32_t page_size;
  int32_t Hkv;
  int32_t d;
  hs2_dtype dtype;
  const float* k_scale;
  const float* v_scale;
  const uint8_t* k_sf;
  const uint8_t* v_sf;
} hs2_kv;

/* ---------------------------------------------------------------------------
 * FA layer + window-excluding top-k selection  ([HS2] §5, §7.2; the "oracle"
 * selection of the appendix: the FA's own exactly computed attention scores).
 *
 * decode (prefill = 0): one query per sequence; q is [batch][Hq][d] of kv->dtype,
 *   B_or_n must equal kv->batch; query b sees t_b = seq_len[b] keys.
 * prefill (prefill = 1): one sequence (kv->batch == 1), n = B_or_n query rows,
 *   q is [n][Hq][d]; row i sees t_i = i + 1 keys; requires n <= seq_len[0].
 *
 * Per query and head h: x_h(s) = scale * q_h . k_g(s) for s < t;
 *   o[..][h][:] = sum_s softmax(x_h)(s) v_g(s);  lse[..][h] = log sum_s exp x_h(s).
 * Per query and KV head g: score_g(s) = sum_{h in g} exp(x_h(s) - lse_h) over
 *   s in F(t); idx[..][g][:] = the min(k, |F|) best positions (score descending,
 *   lower position first on ties), ascending, -1 padded; idx_cnt[..][g] = count.
 * Outputs: o float32 [B_or_n][Hq][d]; lse float32 [B_or_n][Hq] (may be NULL);
 *   idx int32 [B_or_n][Hkv][k]; idx_cnt int32 [B_or_n][Hkv].
 * workspace: device scratch of at least hs2_fa_select_workspace(...) bytes,
 *   256-byte aligned; contents on entry are ignored.
 * max_t: the largest seq_len of the call (decode) or n (prefill).
 * Requirements: Hq % Hkv == 0, Hq / Hkv <= 32, k >= 0, w >= 0.                     */
size_t hs2_fa_select_workspace(int B_or_n, int Hq, const hs2_kv* kv, int max_t, int k, int prefill);
hs2_status hs2_fa_select(const void* q, int B_or_n, int Hq, const hs2_kv* kv, int max_t, int w,
                         int k, float scale, int prefill, float* o, float* lse, int32_t* idx,
                         int32_t* idx_cnt, void* workspace, size_t ws_bytes, int32_t* dev_err,
                         void* stream);

/* hs2_fa_select with block-level selection, the first HySparse version's scheme ([HS2] §2:
 * 16 blocks of 64 tokens = 1024 positions). sel_block = 1 is hs2_fa_select. sel_block > 1
 * (decode only; sel_block a multiple of 4, at most 4096, and k a multiple of sel_block): far position s belongs to
 * block s / sel_block, a block's key is the largest selection score among its far
 * positions, and the min(k / sel_block, #blocks) best blocks by (key descending, block
 * ascending) are taken whole: idx holds their far positions ascending (-1 padded),
 * idx_cnt their number. Prefill with sel_block > 1: HS2_ERR_UNSUPPORTED. The workspace
 * size is hs2_fa_select_workspace's. */
hs2_status hs2_fa_select_ex(const void* q, int B_or_n, int Hq, const hs2_kv* kv, int max_t, int w,
                            int k, float scale, int prefill, int sel_block, float* o, float* lse,
                            int32_t* idx, int32_t* idx_cnt, void* workspace, size_t ws_bytes,
                            int32_t* dev_err, void* stream);

/* ---------------------------------------------------------------------------
 * Decode KV append  ([HS2] §10.1, step 3: once the source hidden state is ready, each
 * Cross group's cache gains one entry; §4.2: the groups' KV branches are independent).
 * The new token is the last visible key of its sequence: for every cache c < n_caches and
 * sequence b < kvs[c].batch, with t = kvs[c].seq_len[b] (already counting the new token),
 *   K row t-1 of KV head g  <-  k_new[c][b][g][:]   (and V likewise from v_new[c]),
 * i.e. slot (t-1) % 64 of page block_table[b][(t-1) / 64]. One launch for all caches.
 * kvs: host array of n_caches descriptors (1 <= n_caches <= 8), bf16 or f32 pools; an FP8
 *   pool returns HS2_ERR_UNSUPPORTED (its per-page scale would have to change). A key-only
 *   cache (v = NULL, e.g. a CSA2 indexer-key cache) takes k_new only.
 * k_new, v_new: host arrays of n_caches device pointers, each [batch][Hkv][d] in the
 *   cache's dtype, 16-byte aligned; v_new may be NULL when every cache is key-only.
 * The pools are written through the descriptors' k / v pointers, which must therefore be
 *   writable device memory owned by the caller. The page holding position t-1 must belong
 *   to that sequence alone for the duration of the call.
 * Device-side: t < 1 or t > 64 * max_pages sets HS2_DEV_BAD_LENGTH, a block-table entry
 *   outside [0, num_pages) sets HS2_DEV_BAD_PAGE; that sequence's rows are not written. */
hs2_status hs2_kv_append(int n_caches, const hs2_kv* kvs, const void* const* k_new, const void* const* v_new,
                         int32_t* dev_err, void* stream);

/* Decode FA + selection with the current token's K/V append fused in (hs2_fa_select_ex,
 * decode only, plus hs2_kv_append of one cache): k_new / v_new [batch][Hq / G = Hkv][d]
 * (device, kv->dtype, 16-byte aligned) are written to position t-1 as hs2_kv_append does,
 * and the scan uses them for key t-1. On the bf16 tensor-core scan the write happens inside
 * the scan kernel, which takes key t-1 from k_new / v_new rather than the pool; otherwise
 * (f32, or a head-sharing factor that path does not take) a separate append kernel runs
 * first on the same stream. Outputs equal those of hs2_kv_append followed by
 * hs2_fa_select_ex. FP8 pools: HS2_ERR_UNSUPPORTED. The workspace size is
 * hs2_fa_select_workspace(B, Hq, kv, max_t, k, 0). */
hs2_status hs2_fa_select_append(const void* q, int B, int Hq, const hs2_kv* kv, int max_t, int w, int k,
                                float scale, int sel_block, const void* k_new, const void* v_new, float* o,
                                float* lse, int32_t* idx, int32_t* idx_cnt, void* workspace, size_t ws_bytes,
                                int32_t* dev_err, void* stream);

/* ---------------------------------------------------------------------------
 * hs2_fa_select_noalloc — hs2_fa_select for callers that cannot allocate device
 * memory (an engine that has reserved nearly all HBM for its KV pool and forbids
 * further cudaMalloc, or a latency-critical thread that must not call cudaMalloc /
 * cudaFree because they can synchronise the device). It takes no workspace: its
 * scratch is a file-scope device array of hs2_fa_select_noalloc_capacity() bytes
 * (64 MiB) that every GPU loading the library holds until the process exits. The
 * pages have no counterpart to this entry point; it is a deployment convenience.
 * Arguments, outputs and results are exactly those of hs2_fa_select.
 * - Returns HS2_ERR_SCRATCH_LIMIT, launching nothing, when
 *   hs2_fa_select_workspace(...) of the call exceeds the capacity.
 * - The first call on a device looks up the array's device address on that device
 *   (it must be the current device); make that first call before any stream capture.
 *   The address is looked up again when the device's current context has changed since
 *   (after a cudaDeviceReset, say); make the first call after such a change before any
 *   stream capture too.
 * - All calls share the one array: calls that overlap on the GPU (concurrent streams
 *   or host threads) race and corrupt each other's results; serialise them.
 * - It allocates nothing and calls no cudaMalloc / cudaFree.                        */
size_t hs2_fa_select_noalloc_capacity(void);
hs2_status hs2_fa_select_noalloc(const void* q, int B_or_n, int Hq, const hs2_kv* kv, int max_t, int w,
                                 int k, float scale, int prefill, float* o, float* lse, int32_t* idx,
                                 int32_t* idx_cnt, int32_t* dev_err, void* stream);

/* ---------------------------------------------------------------------------
 * SA layer: KV and index reuse with the layer's own query  ([HS2] §5, §7.2, §7.4).
 * For each query and head h of KV head g:
 *   U = W(t) ∪ {idx[..][g][j] : j < idx_cnt[..][g]}   (the caller guarantees the
 *   indices lie in F(t), i.e. outside the window; with w = 0 any s < t),
 *   o[..][h][:] = sum_{s in U} softmax_U(scale * q_h . k_g(s)) v_g(s), one softmax.
 * Shapes and the decode / prefill convention are those of hs2_fa_select; idx and
 * idx_cnt have the layout hs2_fa_select writes ([B_or_n][Hkv][k], [B_or_n][Hkv]).
 * workspace: at least hs2_sa_reuse_workspace(...) bytes, 256-byte aligned, no
 *   initialisation needed; calls that run at the same time need workspaces of their own. */
size_t hs2_sa_reuse_workspace(int B_or_n, int Hq, const hs2_kv* kv, int w, int k, int prefill);
hs2_status hs2_sa_reuse(const void* q, int B_or_n, int Hq, const hs2_kv* kv, int w,
                        const int32_t* idx, const int32_t* idx_cnt, int k, float scale, int prefill,
                        float* o, void* workspace, size_t ws_bytes, int32_t* dev_err, void* stream);

/* hs2_sa_reuse with the SA layers' per-head sink bias and output sigmoid gate
 * ([HS2] §17.1). sink: float32 [Hq] natural-log logits, or NULL: one more key per head
 * with logit sink[h] and a zero value, i.e. the single softmax denominator over W ∪ S
 * gains exp(sink[h]) (-inf = no sink). gate: float32 [B_or_n][Hq][d] logits, or NULL:
 * the output is multiplied elementwise by 1 / (1 + exp(-gate)). Both are read-only,
 * device memory, owned by the caller.
 * flags: 0 or HS2_SA_OVERLAP. The decode kernel is always launched so that it may start
 *   while the previous launch on `stream` finishes (programmatic dependent launch), and
 *   waits for that launch before it reads anything. HS2_SA_OVERLAP (decode) is for the SA
 *   layers of a group after the first, each issued right after the one before it:
 *   - the call reads idx, idx_cnt, kv->block_table and kv->seq_len before that wait, so
 *     those four must have been complete before the previous launch on the stream began
 *     (not written by it);
 *   - `workspace` must be the one the previous hs2_sa_reuse call on this stream used,
 *     with the same B_or_n, Hq, kv sizes, w and k: the call keeps the state that call
 *     left in it instead of clearing it, and makes no launch but its kernel.
 *   Prefill ignores the flag; other bits: HS2_ERR_ARG.
 * Everything else as hs2_sa_reuse (which is this call with sink = gate = NULL, flags = 0);
 * the workspace size does not change. */
#define HS2_SA_OVERLAP 1
hs2_status hs2_sa_reuse_ex(const void* q, int B_or_n, int Hq, const hs2_kv* kv, int w,
                           const int32_t* idx, const int32_t* idx_cnt, int k, float scale, int prefill,
                           const float* sink, const float* gate, int flags, float* o, void* workspace,
                           size_t ws_bytes, int32_t* dev_err, void* stream);

/* ---------------------------------------------------------------------------
 * CSA2 hierarchical sparse indexer  ([CSA2] §3.1-3.2; score from [L10] §5.1).
 * I(s) = sum_j w_idx[b][j] * max(0, q_idx[b][j] . k_idx(s)), unscaled, where k_idx(s)
 * is row s of the indexer-key cache k_idx (Hkv = 1, d = di, v = NULL), shared by
 * all Hi indexer heads.
 * HS2_FULL: score every s < t; idx[b] = top-min(k_top, t) positions; block maxima
 *   over blocks [blk*j, blk*j+blk) ∩ [0,t); pool_blocks[b] = top-min(max_blocks,
 *   ceil(t/blk)) block ids (maximum descending, lower id first), ascending, -1
 *   padded; pool_cnt[b] = count.  (pool_blocks / pool_cnt are outputs.)
 * HS2_REINDEX: score only the positions of the given pool (inputs pool_blocks /
 *   pool_cnt); idx[b] = top-min(k_top, |pool positions|), ascending.
 * (Reuse layers call nothing: they pass the previous idx to hs2_sa_reuse.)
 * q_idx: [batch][Hi][di] of k_idx->dtype; w_idx: float32 [batch][Hi];
 * idx: int32 [batch][k_top]; idx_cnt: int32 [batch]; blk must divide page_size.
 * workspace: at least hs2_hier_reindex_workspace(...) bytes, 256-byte aligned.     */
typedef enum { HS2_FULL = 0, HS2_REINDEX = 1 } hs2_idx_mode;
size_t hs2_hier_reindex_workspace(hs2_idx_mode mode, int Hi, const hs2_kv* k_idx, int max_t,
                                  int k_top, int blk, int max_blocks);
hs2_status hs2_hier_reindex(hs2_idx_mode mode, const void* q_idx, const float* w_idx, int Hi,
                            const hs2_kv* k_idx, int max_t, int k_top, int blk, int max_blocks,
                            int32_t* pool_blocks, int32_t* pool_cnt, int32_t* idx, int32_t* idx_cnt,
                            void* workspace, size_t ws_bytes, int32_t* dev_err, void* stream);

/* ---------------------------------------------------------------------------
 * Diagnostics.
 * hs2_profile_next: the next call on this host thread that runs `stage` records the
 * cudaEvent_t handles `start` and `stop` (passed as void*, created by the caller) on
 * that call's stream immediately before and after the stage's main kernel; one-shot,
 * NULL events clear it. Lets a caller time the dominant kernel inside a running step. */
typedef enum {
  HS2_STAGE_FA_SCAN = 0,    /* FA scan over all visible keys (hs2_fa_select) */
  HS2_STAGE_SA_GATHER = 1,  /* SA gather-attention (hs2_sa_reuse) */
  HS2_STAGE_INDEXER = 2     /* lightning-indexer scan (hs2_hier_reindex) */
} hs2_stage;
void hs2_profile_next(hs2_stage stage, void* start, void* stop);
/* hs2_selftest_wait_timeout: launches one warp that waits, through the library's bounded
 * mbarrier wait and with a limit of timeout_us microseconds (1 .. 2000000), on a barrier nothing
 * arrives on; the wait gives up, HS2_DEV_TIMEOUT is set in *dev_err (device memory) and the
 * kernel finishes. Lets a caller check the device-side timeout path without a fault. */
hs2_status hs2_selftest_wait_timeout(int timeout_us, int32_t* dev_err, void* stream);
/* hs2_fa_select_launches / hs2_sa_reuse_launches: how many kernels hs2_fa_select_ex (with
 * append != 0: hs2_fa_select_append) and hs2_sa_reuse_ex launch for these arguments (device
 * memsets not counted), or -1 for arguments they reject on the host. Lets a caller account
 * for the library's launches inside a step; launches nothing (it may query the current
 * device's properties, as the calls themselves do to plan their grids). */
int hs2_fa_select_launches(int B_or_n, int Hq, const hs2_kv* kv, int max_t, int w, int k, int prefill,
                           int sel_block, int append);
int hs2_sa_reuse_launches(int B_or_n, int Hq, const hs2_kv* kv, int w, int k, int prefill);
const char* hs2_strerror(hs2_status st);
int hs2_last_cuda_error(void); /* cudaError_t of the last HS2_ERR_CUDA, 0 if none */
int hs2_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* HS2_H */

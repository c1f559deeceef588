// kv_append.cu — decode KV append: the new token's K and V rows of every sequence written
// into its paged cache, for several independent caches in one launch.
//
// At decode, once the source hidden state is ready, each of the four Cross groups gains one
// KV entry ("HySparse2：整体架构、KV 生命周期与 PD 分离", §10.1, step 3), and the groups' KV
// branches are independent of one another (§4.2), so their appends share a launch. The new
// token is the last visible key: it goes to position t-1 (t = seq_len[b]), i.e. slot
// (t-1) % 64 of page block_table[b][(t-1) / 64].
#include "common.cuh"
#include "kernels.h"

namespace hs2 {

// grid (largest batch, caches), 128 threads: each thread moves 16-byte units of the K and V rows of
// every KV head.
__global__ void __launch_bounds__(128) kv_append_kernel(const AppendArgs a) {
  const int b = blockIdx.x;
  const AppendCache& c = a.c[blockIdx.y];
  if (b >= c.B) return;
  const int t = c.seq_len[b];
  if (t < 1 || t > c.max_pages * kPage) {
    if (threadIdx.x == 0) flag_error(a.dev_err, HS2_DEV_BAD_LENGTH);
    return;
  }
  const int pos = t - 1;
  const int phys = c.bt[(size_t)b * c.max_pages + pos / kPage];
  if (phys < 0 || phys >= c.num_pages) {
    if (threadIdx.x == 0) flag_error(a.dev_err, HS2_DEV_BAD_PAGE);
    return;
  }
  const int slot = pos % kPage;
  const int upr = c.row_bytes / 16;  // 16-byte units per row
  const int per_kind = c.Hkv * upr;
  const int total = (c.v ? 2 : 1) * per_kind;
  for (int i = threadIdx.x; i < total; i += blockDim.x) {
    const int kind = i / per_kind, r = i % per_kind, g = r / upr, u = r % upr;
    const uint8_t* src =
        reinterpret_cast<const uint8_t*>(kind ? c.v_new : c.k_new) + ((size_t)b * c.Hkv + g) * c.row_bytes + 16 * u;
    uint8_t* dst = reinterpret_cast<uint8_t*>(kind ? c.v : c.k) +
                   (((size_t)phys * c.Hkv + g) * kPage + slot) * c.row_bytes + 16 * u;
    *reinterpret_cast<uint4*>(dst) = __ldg(reinterpret_cast<const uint4*>(src));
  }
}

cudaError_t launch_kv_append(const AppendArgs& a, cudaStream_t s) {
  if (a.n < 1 || a.n > kMaxAppendCaches || a.B < 1) return cudaErrorInvalidValue;
  kv_append_kernel<<<dim3(a.B, a.n), 128, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace hs2

// noalloc.cu — hs2_fa_select_noalloc: the FA scan + top-k without a caller workspace.
//
// Some callers cannot hand the library a scratch buffer: an inference engine that has
// reserved (nearly) all HBM for its paged KV pool at start-up and forbids further
// cudaMalloc calls, or a latency-critical host thread that must not call cudaMalloc /
// cudaFree because they may synchronise the device. For them this entry point keeps
// its scratch in a file-scope device array instead of a workspace argument.
//
// The array is a module global: every GPU that loads the library holds kNoAllocScratch
// bytes of it until the process exits. In host code the symbol is only a host-side
// stand-in, never a device address; the device address is fetched per device with
// cudaGetSymbolAddress (with that device current) on the first call made on it, and
// fetched again whenever the device's current context is a different one (after a
// cudaDeviceReset the module is loaded anew and the array may sit elsewhere).
// Every call shares the array: calls that overlap on the GPU (other streams, other
// host threads) race on it. Nothing in it needs to start at zero: each call writes every
// scratch element it later reads.
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "../../include/hs2.h"

namespace {

constexpr size_t kNoAllocScratch = size_t(64) << 20;  // 64 MiB
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratch];

std::mutex g_setup_mu;
void* g_scratch_ptr[kMaxDevices] = {};
unsigned long long g_scratch_ctx[kMaxDevices] = {};  // id of the context the address belongs to

// The unique id of the calling thread's current context (cuCtxGetCurrent + cuCtxGetId, taken
// from the driver at run time so the library needs no link against it); 0 if unavailable.
unsigned long long current_context_id() {
  using GetCurrent = CUresult (*)(CUcontext*);
  using GetId = CUresult (*)(CUcontext, unsigned long long*);
  static GetCurrent get_current = nullptr;
  static GetId get_id = nullptr;
  static bool looked_up = false;
  if (!looked_up) {
    void* f1 = nullptr;
    void* f2 = nullptr;
    cudaDriverEntryPointQueryResult q1, q2;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f1, 12000, cudaEnableDefault, &q1) == cudaSuccess &&
        q1 == cudaDriverEntryPointSuccess)
      get_current = (GetCurrent)f1;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f2, 12000, cudaEnableDefault, &q2) == cudaSuccess &&
        q2 == cudaDriverEntryPointSuccess)
      get_id = (GetId)f2;
    (void)cudaGetLastError();
    looked_up = true;
  }
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || !ctx || get_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return id;
}

// Device address of the scratch array on the current device, looked up once per device and
// again whenever that device's current context has changed since.
hs2_status scratch_for_current_device(void** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return HS2_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return HS2_ERR_UNSUPPORTED;
  e = cudaSetDevice(dev);  // makes the device's primary context current (created if need be)
  if (e != cudaSuccess) return HS2_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_setup_mu);
  const unsigned long long ctx = current_context_id();
  if (!g_scratch_ptr[dev] || ctx == 0 || ctx != g_scratch_ctx[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || !p) {
      (void)cudaGetLastError();
      return HS2_ERR_CUDA;
    }
    g_scratch_ptr[dev] = p;
    g_scratch_ctx[dev] = ctx;
  }
  *out = g_scratch_ptr[dev];
  return HS2_OK;
}

}  // namespace

extern "C" {

size_t hs2_fa_select_noalloc_capacity(void) { return kNoAllocScratch; }

hs2_status hs2_fa_select_noalloc(const void* q, int B_or_n, int Hq, const hs2_kv* kv, int max_t, int w, int k,
                                 float scale, int prefill, float* o, float* lse, int32_t* idx, int32_t* idx_cnt,
                                 int32_t* dev_err, void* stream) {
  const size_t need = hs2_fa_select_workspace(B_or_n, Hq, kv, max_t, k, prefill);
  if (need == 0 && B_or_n > 0) return HS2_ERR_ARG;
  if (need > kNoAllocScratch) return HS2_ERR_SCRATCH_LIMIT;
  void* scratch = nullptr;
  const hs2_status st = scratch_for_current_device(&scratch);
  if (st != HS2_OK) return st;
  return hs2_fa_select(q, B_or_n, Hq, kv, max_t, w, k, scale, prefill, o, lse, idx, idx_cnt, scratch,
                       kNoAllocScratch, dev_err, stream);
}

}  // extern "C"

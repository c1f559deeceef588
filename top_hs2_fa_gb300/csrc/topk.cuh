// topk.cuh — block-wide exact top-k by radix select (ties -> lower candidate index).
//
// Keys are uint32 whose unsigned order equals the score order (non-negative fp32
// bit patterns). The k-th largest key T is found with three histogram passes
// (digits of 11, 11 and 10 bits, most significant first) over the candidates that
// still match the chosen prefix; warp-aggregated shared-memory atomics keep equal
// digits from serialising. Candidates > T are all taken; of those == T the
// lowest-indexed ones fill the remaining slots. The chosen candidates are emitted
// in ascending candidate order, so the output is sorted when candidates are.
#pragma once
#include "common.cuh"

namespace hs2 {

template <int NT>
struct TopkSmem {
  uint32_t hist[2048];
  int warp_tot[NT / 32];
  int bcast[2];
};

// Exclusive scan of one int per thread over the block (all NT threads must call).
template <int NT>
HS2_DEVI int block_exclusive_scan(int v, int* warp_tot, int* total_out = nullptr) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_tot[wid] = x;
  __syncthreads();
  if (wid == 0) {
    int t = lane < NT / 32 ? warp_tot[lane] : 0;
    int s = t;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int y = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += y;
    }
    if (lane < NT / 32) warp_tot[lane] = s - t;  // exclusive prefix of warp totals
    if (lane == 31 && total_out) *total_out = s;
  }
  __syncthreads();
  int r = warp_tot[wid] + x - v;
  __syncthreads();
  return r;
}

// key(i) -> uint32 key of candidate i (i < n); emit(j, i): output slot j <- candidate i.
// kk = number to select (<= n). All NT threads of the block must call.
template <int NT, typename KeyFn, typename EmitFn>
__device__ void block_topk(int n, int kk, KeyFn key, EmitFn emit, TopkSmem<NT>& sm) {
  const int tid = threadIdx.x;
  const int lane = tid & 31;
  if (kk <= 0 || n <= 0) return;
  if (kk >= n) {
    for (int i = tid; i < n; i += NT) emit(i, i);
    return;
  }
  uint32_t prefix = 0, mask = 0;
  int remaining = kk;
#pragma unroll 1
  for (int pass = 0; pass < 3; ++pass) {
    const int sh = pass == 0 ? 21 : (pass == 1 ? 10 : 0);
    const int nb = pass == 2 ? 1024 : 2048;
    for (int i = tid; i < 2048; i += NT) sm.hist[i] = 0;
    __syncthreads();
    for (int i0 = 0; i0 < n; i0 += NT) {
      const int i = i0 + tid;
      uint32_t u = 0;
      bool part = false;
      if (i < n) {
        u = key(i);
        part = (u & mask) == prefix;
      }
      const unsigned pm = __ballot_sync(0xffffffffu, part);
      if (part) {
        const uint32_t dig = (u >> sh) & (uint32_t)(nb - 1);
        const unsigned peers = __match_any_sync(pm, dig);
        if (lane == __ffs(peers) - 1) atomicAdd(&sm.hist[dig], (uint32_t)__popc(peers));
      }
    }
    __syncthreads();
    // suffix scan: the digit where the count of larger digits first reaches `remaining`
    constexpr int kMaxPer = 2048 / NT;
    const int per = nb / NT;
    const int lo = (NT - 1 - tid) * per;  // thread 0 owns the highest bins
    int local = 0;
#pragma unroll
    for (int j = 0; j < kMaxPer; ++j)
      if (j < per) local += (int)sm.hist[lo + j];
    int above = block_exclusive_scan<NT>(local, sm.warp_tot);  // count in bins above this range
    if (above < remaining && above + local >= remaining) {
      int run = above;
      for (int j = per - 1; j >= 0; --j) {
        const int c = (int)sm.hist[lo + j];
        if (run + c >= remaining) {
          sm.bcast[0] = lo + j;
          sm.bcast[1] = remaining - run;
          break;
        }
        run += c;
      }
    }
    __syncthreads();
    const uint32_t dig = (uint32_t)sm.bcast[0];
    remaining = sm.bcast[1];
    prefix |= dig << sh;
    mask |= (uint32_t)(nb - 1) << sh;
    __syncthreads();
  }
  const uint32_t T = prefix;
  const int take_eq = remaining;  // how many candidates equal to T are taken (lowest first)
  // compaction over thread-contiguous segments, in candidate order
  const int seg = (n + NT - 1) / NT;
  const int lo = min(n, tid * seg), hi = min(n, lo + seg);
  int n_eq = 0, n_gt = 0;
  for (int i = lo; i < hi; ++i) {
    const uint32_t u = key(i);
    n_eq += (u == T);
    n_gt += (u > T);
  }
  const int eq_before = block_exclusive_scan<NT>(n_eq, sm.warp_tot);
  const int eq_take = max(0, min(n_eq, take_eq - eq_before));
  int pos = block_exclusive_scan<NT>(n_gt + eq_take, sm.warp_tot);
  int eq_seen = eq_before;
  for (int i = lo; i < hi; ++i) {
    const uint32_t u = key(i);
    bool sel = u > T;
    if (u == T) {
      sel = eq_seen < take_eq;
      ++eq_seen;
    }
    if (sel) emit(pos++, i);
  }
}

}  // namespace hs2

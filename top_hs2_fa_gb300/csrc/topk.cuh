// topk.cuh — block-wide exact top-k by radix select (ties -> lower candidate index).
//
// Keys are uint32 whose unsigned order equals the score order (non-negative fp32 bit
// patterns). The k-th largest key T is found digit by digit, most significant first:
// a histogram of the current digit over the candidates that still match the chosen
// prefix, then a suffix scan that finds the digit holding the k-th largest. Digits are
// 12, 12 and 8 bits wide. Warp-aggregated shared-memory atomics keep lanes that share
// a digit from serialising. Candidates > T are all taken; of those == T the lowest-
// indexed fill the remaining slots. Chosen candidates are emitted in ascending
// candidate order, so the output is sorted whenever the candidates are.
#pragma once
#include "common.cuh"

namespace hs2 {

constexpr int kRadixBins = 4096;

template <int NT>
struct TopkSmem {
  uint32_t hist[kRadixBins];
  int warp_tot[NT / 32];
  int bcast[2];
};

// Exclusive scan of one int per thread over the block (all NT threads must call).
template <int NT>
HS2_DEVI int block_exclusive_scan(int v, int* warp_tot) {
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
  }
  __syncthreads();
  int r = warp_tot[wid] + x - v;
  __syncthreads();
  return r;
}

// Add `cnt` to hist[dig] for every participating lane, one atomic per distinct digit.
HS2_DEVI void hist_add_warp(uint32_t* hist, bool part, uint32_t dig) {
  const unsigned pm = __ballot_sync(0xffffffffu, part);
  if (part) {
    const unsigned peers = __match_any_sync(pm, dig);
    if ((threadIdx.x & 31) == __ffs(peers) - 1) atomicAdd(&hist[dig], (uint32_t)__popc(peers));
  }
}

// Given a histogram of nb bins (the current digit), find the digit that holds the
// `remaining`-th largest candidate; returns it and updates `remaining` to the rank
// inside that digit. All NT threads must call; hist is read-only here.
template <int NT>
HS2_DEVI uint32_t find_digit(const uint32_t* hist, int nb, int& remaining, TopkSmem<NT>& sm) {
  constexpr int kMaxPer = kRadixBins / NT;
  const int tid = threadIdx.x;
  const int per = nb >= NT ? nb / NT : 1;
  const int owners = nb / per;
  const bool own = tid < owners;
  const int lo = own ? (owners - 1 - tid) * per : 0;  // thread 0 owns the highest bins
  int local = 0;
#pragma unroll
  for (int j = 0; j < kMaxPer; ++j)
    if (own && j < per) local += (int)hist[lo + j];
  const int above = block_exclusive_scan<NT>(local, sm.warp_tot);  // count in bins above this range
  if (own && above < remaining && above + local >= remaining) {
    int run = above;
    for (int j = per - 1; j >= 0; --j) {
      const int c = (int)hist[lo + j];
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
  __syncthreads();
  return dig;
}

// One refinement pass: histogram of bits [sh, sh+bits) over candidates whose key matches
// prefix under mask, then choose the digit. Updates prefix, mask, remaining.
template <int NT, typename KeyFn>
__device__ void radix_pass(int n, KeyFn key, int sh, int bits, uint32_t& prefix, uint32_t& mask,
                           int& remaining, TopkSmem<NT>& sm) {
  const int nb = 1 << bits;
  for (int i = threadIdx.x; i < nb; i += NT) sm.hist[i] = 0;
  __syncthreads();
  for (int i0 = 0; i0 < n; i0 += NT) {
    const int i = i0 + threadIdx.x;
    uint32_t u = 0;
    bool part = false;
    if (i < n) {
      u = key(i);
      part = (u & mask) == prefix;
    }
    hist_add_warp(sm.hist, part, (u >> sh) & (uint32_t)(nb - 1));
  }
  __syncthreads();
  const uint32_t dig = find_digit<NT>(sm.hist, nb, remaining, sm);
  prefix |= dig << sh;
  mask |= (uint32_t)(nb - 1) << sh;
}

// Order-preserving compaction of the candidates > T plus the first take_eq candidates
// == T. Warp w owns the contiguous range [w*wseg, (w+1)*wseg); lanes read consecutive
// candidates. All NT threads must call.
template <int NT, typename KeyFn, typename EmitFn>
__device__ void compact_selected(int n, KeyFn key, uint32_t T, int take_eq, EmitFn emit, TopkSmem<NT>& sm) {
  constexpr int NW = NT / 32;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int wseg = (n + NW - 1) / NW;
  const int wlo = min(n, warp * wseg), whi = min(n, wlo + wseg);
  int n_eq = 0, n_gt = 0;
  for (int i = wlo + lane; i < whi; i += 32) {
    const uint32_t u = key(i);
    n_eq += (u == T);
    n_gt += (u > T);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    n_eq += __shfl_xor_sync(0xffffffffu, n_eq, o);
    n_gt += __shfl_xor_sync(0xffffffffu, n_gt, o);
  }
  __syncthreads();
  if (lane == 0) sm.warp_tot[warp] = n_eq;
  __syncthreads();
  int eq_before = 0;
  for (int w = 0; w < warp; ++w) eq_before += sm.warp_tot[w];
  const int eq_take = max(0, min(n_eq, take_eq - eq_before));
  __syncthreads();
  if (lane == 0) sm.warp_tot[warp] = n_gt + eq_take;
  __syncthreads();
  int pos = 0;
  for (int w = 0; w < warp; ++w) pos += sm.warp_tot[w];
  const unsigned lt = (1u << lane) - 1u;
  int eq_seen = eq_before;
  for (int base = wlo; base < whi; base += 32) {
    const int i = base + lane;
    const bool valid = i < whi;
    const uint32_t u = valid ? key(i) : 0u;
    const bool gt = valid && u > T;
    const bool eq = valid && u == T;
    const unsigned beq = __ballot_sync(0xffffffffu, eq);
    const bool sel = gt || (eq && eq_seen + __popc(beq & lt) < take_eq);
    const unsigned bs = __ballot_sync(0xffffffffu, sel);
    if (sel) emit(pos + __popc(bs & lt), i);
    pos += __popc(bs);
    eq_seen += __popc(beq);
  }
  __syncthreads();
}

// key(i) -> uint32 key of candidate i (i < n); emit(j, i): output slot j <- candidate i.
// kk = number to select. All NT threads of the block must call.
template <int NT, typename KeyFn, typename EmitFn>
__device__ void block_topk(int n, int kk, KeyFn key, EmitFn emit, TopkSmem<NT>& sm) {
  if (kk <= 0 || n <= 0) return;
  if (kk >= n) {
    for (int i = threadIdx.x; i < n; i += NT) emit(i, i);
    return;
  }
  uint32_t prefix = 0, mask = 0;
  int remaining = kk;
  radix_pass<NT>(n, key, 20, 12, prefix, mask, remaining, sm);
  radix_pass<NT>(n, key, 8, 12, prefix, mask, remaining, sm);
  radix_pass<NT>(n, key, 0, 8, prefix, mask, remaining, sm);
  compact_selected<NT>(n, key, prefix, remaining, emit, sm);
}

}  // namespace hs2

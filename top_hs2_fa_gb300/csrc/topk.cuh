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
// One shared-memory atomic per key: cheaper than hist_add_warp's ballot and match when
// the digits of a warp's keys are spread out (the first digit of scores over a sequence),
// dearer when they pile onto a few bins (later radix passes, tied keys).
HS2_DEVI void hist_add(uint32_t* hist, bool part, uint32_t dig) {
  if (part) atomicAdd(&hist[dig], 1u);
}
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

// Number of entries of the ascending array a[0..n) that are < x.
HS2_DEVI int count_below(const int* a, int n, int x) {
  int lo = 0, hi = n;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (a[mid] < x) lo = mid + 1;
    else hi = mid;
  }
  return lo;
}

// Exact top-kk of n keys read from global memory, given the global histogram of their top
// 12 bits (ghist, kRadixBins bins). The row must start 16-byte aligned and be readable up to
// n rounded up to a multiple of 4. One coalesced pass (V keys per thread per chunk, V a
// multiple of 4) splits the keys into
//   A: top 12 bits above the digit d that holds the kk-th key — all selected, and
//   C: top 12 bits equal to d — the candidates,
// both in index order in shared memory (la: cap_a ints, lc: cap_c (index, key) pairs). The
// rank inside C is refined by radix select over C alone; the chosen part of C goes to lsel
// (kk ints) in index order, and A and it are merged: emit(j, i) writes output slot j (ascending
// index order) <- key index i. Returns false, having emitted nothing, when C or A exceed their
// buffers (the caller then runs block_topk-style passes over all keys). All NT threads call.
// ghist = null: the histogram is already in sm.hist (filled by the calling CTA).
template <int NT, int V, typename EmitFn>
__device__ bool filter_topk(const uint32_t* gkeys, int n, int kk, const uint32_t* ghist, int* la, int cap_a,
                            uint2* lc, int cap_c, int* lsel, EmitFn emit, TopkSmem<NT>& sm) {
  static_assert(V % 4 == 0 && NT * V < 65536, "chunk counts are packed in 16 bits");
  const int tid = threadIdx.x;
  if (ghist)
    for (int i = tid; i < kRadixBins; i += NT) sm.hist[i] = __ldcg(ghist + i);
  __syncthreads();
  int remaining = kk;
  const uint32_t d = find_digit<NT>(sm.hist, kRadixBins, remaining, sm);
  const int nA = kk - remaining, nC = (int)sm.hist[d];
  if (nC > cap_c || nA > cap_a) return false;  // block-uniform (shared values)
  int baseA = 0, baseC = 0;
  for (int c0 = 0; c0 < n; c0 += NT * V) {
    const int i0 = c0 + tid * V;
    uint32_t kv[V];
#pragma unroll
    for (int q = 0; q < V / 4; ++q) {
      uint4 x = make_uint4(0u, 0u, 0u, 0u);
      if (i0 + 4 * q < n) x = __ldcg(reinterpret_cast<const uint4*>(gkeys + i0 + 4 * q));
      kv[4 * q] = x.x;
      kv[4 * q + 1] = x.y;
      kv[4 * q + 2] = x.z;
      kv[4 * q + 3] = x.w;
    }
    int ca = 0, cc = 0;
#pragma unroll
    for (int v = 0; v < V; ++v) {
      const bool ok = i0 + v < n;
      const uint32_t dg = kv[v] >> 20;
      ca += ok && dg > d;
      cc += ok && dg == d;
    }
    const int mine = ca | (cc << 16);
    const int off = block_exclusive_scan<NT>(mine, sm.warp_tot);
    int oa = baseA + (off & 0xffff), oc = baseC + (off >> 16);
#pragma unroll
    for (int v = 0; v < V; ++v) {
      const int i = i0 + v;
      if (i < n) {
        const uint32_t dg = kv[v] >> 20;
        if (dg > d) la[oa++] = i;
        else if (dg == d) lc[oc++] = make_uint2((uint32_t)i, kv[v]);
      }
    }
    if (tid == NT - 1) sm.bcast[0] = off + mine;
    __syncthreads();
    const int tot = sm.bcast[0];
    baseA += tot & 0xffff;
    baseC += tot >> 16;
    __syncthreads();
  }
  // refine inside C (keys share the top 12 bits d), then take its chosen part in order
  uint32_t prefix = d << 20, mask = 0xfff00000u;
  auto ckey = [&](int j) { return lc[j].y; };
  radix_pass<NT>(nC, ckey, 8, 12, prefix, mask, remaining, sm);
  radix_pass<NT>(nC, ckey, 0, 8, prefix, mask, remaining, sm);
  compact_selected<NT>(nC, ckey, prefix, remaining, [&](int j, int i) { lsel[j] = (int)lc[i].x; }, sm);
  const int nS = kk - nA;
  for (int j = tid; j < nA; j += NT) emit(j + count_below(lsel, nS, la[j]), la[j]);
  for (int j = tid; j < nS; j += NT) emit(j + count_below(la, nA, lsel[j]), lsel[j]);
  __syncthreads();
  return true;
}

// filter_topk over a thread-block cluster: the kk-th key's digit d comes from the global
// histogram in every CTA (the same value everywhere); CTA `rank` of `nrank` splits its
// contiguous slice [lo, hi) of the keys (lo a multiple of 4) into its own A and C lists;
// rank 0 gathers every CTA's C list through distributed shared memory, in rank order (so in
// index order), refines it by radix select and keeps the chosen part in lsel; then every CTA
// emits its own A entries and the chosen entries inside its slice at their global output
// slots (the A counts of the lower ranks plus the local merge rank). `cta_sync` is the
// cluster barrier and `remote(ptr, r)` maps a shared-memory pointer to rank r's copy. Returns
// false, uniformly and before any cluster barrier, when a list would overflow (the caller
// then runs the single-CTA fallback on rank 0). meta: 2 ints of shared memory.
template <int NT, int V, typename EmitFn, typename SyncFn, typename RemoteFn>
__device__ bool cluster_filter_topk(const uint32_t* gkeys, int n, int kk, const uint32_t* ghist, int* la, int cap_a,
                                    uint2* lc, int cap_c, int* lsel, int* meta, int rank, int nrank, EmitFn emit,
                                    SyncFn cta_sync, RemoteFn remote, TopkSmem<NT>& sm) {
  static_assert(V % 4 == 0 && NT * V < 65536, "chunk counts are packed in 16 bits");
  const int tid = threadIdx.x;
  for (int i = tid; i < kRadixBins; i += NT) sm.hist[i] = __ldcg(ghist + i);
  __syncthreads();
  int remaining = kk;
  const uint32_t d = find_digit<NT>(sm.hist, kRadixBins, remaining, sm);
  const int nA = kk - remaining, nC = (int)sm.hist[d];
  if (nC > cap_c || nA > cap_a) return false;  // uniform across the cluster
  const int per = (((n + nrank - 1) / nrank) + 3) & ~3;
  const int lo = min(n, rank * per), hi = min(n, lo + per);
  int baseA = 0, baseC = 0;
  for (int c0 = lo; c0 < hi; c0 += NT * V) {
    const int i0 = c0 + tid * V;
    uint32_t kv[V];
#pragma unroll
    for (int q = 0; q < V / 4; ++q) {
      uint4 x = make_uint4(0u, 0u, 0u, 0u);
      if (i0 + 4 * q < hi) x = __ldcg(reinterpret_cast<const uint4*>(gkeys + i0 + 4 * q));
      kv[4 * q] = x.x;
      kv[4 * q + 1] = x.y;
      kv[4 * q + 2] = x.z;
      kv[4 * q + 3] = x.w;
    }
    int ca = 0, cc = 0;
#pragma unroll
    for (int v = 0; v < V; ++v) {
      const bool ok = i0 + v < hi;
      const uint32_t dg = kv[v] >> 20;
      ca += ok && dg > d;
      cc += ok && dg == d;
    }
    const int mine = ca | (cc << 16);
    const int off = block_exclusive_scan<NT>(mine, sm.warp_tot);
    int oa = baseA + (off & 0xffff), oc = baseC + (off >> 16);
#pragma unroll
    for (int v = 0; v < V; ++v) {
      const int i = i0 + v;
      if (i < hi) {
        const uint32_t dg = kv[v] >> 20;
        if (dg > d) la[oa++] = i;
        else if (dg == d) lc[oc++] = make_uint2((uint32_t)i, kv[v]);
      }
    }
    if (tid == NT - 1) sm.bcast[0] = off + mine;
    __syncthreads();
    const int tot = sm.bcast[0];
    baseA += tot & 0xffff;
    baseC += tot >> 16;
    __syncthreads();
  }
  if (tid == 0) {
    meta[0] = baseA;
    meta[1] = baseC;
  }
  cta_sync();
  const int nS = kk - nA;
  if (rank == 0) {
    // append the other ranks' candidates after this CTA's own, in rank order
    int off = baseC;
    for (int r = 1; r < nrank; ++r) {
      const int nr = remote(meta, r)[1];
      const uint2* src = remote(lc, r);
      for (int j = tid; j < nr; j += NT) lc[off + j] = src[j];
      off += nr;
    }
    __syncthreads();
    uint32_t prefix = d << 20, mask = 0xfff00000u;
    auto ckey = [&](int j) { return lc[j].y; };
    radix_pass<NT>(nC, ckey, 8, 12, prefix, mask, remaining, sm);
    radix_pass<NT>(nC, ckey, 0, 8, prefix, mask, remaining, sm);
    compact_selected<NT>(nC, ckey, prefix, remaining, [&](int j, int i) { lsel[j] = (int)lc[i].x; }, sm);
  }
  cta_sync();
  int prefA = 0;
  for (int r = 0; r < rank; ++r) prefA += remote(meta, r)[0];
  const int* lsel0 = remote(lsel, 0);
  for (int j = tid; j < baseA; j += NT) emit(prefA + j + count_below(lsel0, nS, la[j]), la[j]);
  const int j0 = count_below(lsel0, nS, lo), j1 = count_below(lsel0, nS, hi);
  for (int j = j0 + tid; j < j1; j += NT) {
    const int i = lsel0[j];
    emit(j + prefA + count_below(la, baseA, i), i);
  }
  cta_sync();  // rank 0's lists stay alive until every rank has read them
  return true;
}

}  // namespace hs2

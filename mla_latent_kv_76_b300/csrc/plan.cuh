// Split-KV work partition shared by the decode partial kernels and the combine.
//
// Even split (both decode paths): every sequence b is cut into tiles (64 tokens
// on the shape-generic path, 128 on the tensor-core path); the tiles of all
// sequences, in batch order, form one list of T tiles.  Worker g of G owns the
// contiguous range [floor(g T / G), floor((g+1) T / G)), which may cover the end
// of one sequence and the start of the next.  Each (worker, sequence) segment
// writes one partial to slot g + b; slots are unique because worker ranges are
// ordered (if worker g touches sequence b, worker g + 1 starts at b or later).
// The combine merges, for sequence b, the slots of workers g_first(b) ..
// g_last(b) whose range meets b's tiles.
//
// Sequence-aligned plan (tensor-core path, chosen per call when cheaper): see
// plan_entries / plan_prefix below.
#pragma once

#include <climits>

#include <stdint.h>

#include "common.cuh"
#include "kernels.h"

namespace mla {

// Visible length of sequence b after validation against the cache capacity;
// an invalid length counts as an empty sequence and is reported.
MLA_DEVI int effective_len(const int32_t* seqlens, int b, int64_t capacity, int32_t* status) {
  const int L = seqlens[b];
  if (L < 0 || (int64_t)L > capacity) {
    report(status, MLA_ERR_DEVICE_BOUNDS);
    return 0;
  }
  return L;
}

MLA_HD int tiles_of(int L, int tile = kTileTokens) { return (L + tile - 1) / tile; }

// floor(n / d) for n >= 0, d > 0.  64-bit integer division is a long software
// sequence on the GPU (it cost microseconds in the decode prologue), so the
// common case where both fit in 32 bits takes the 32-bit instruction.
MLA_HD int64_t div_floor(int64_t n, int64_t d) {
  if ((uint64_t)n <= 0xFFFFFFFFull && (uint64_t)d <= 0xFFFFFFFFull) return (int64_t)((uint32_t)n / (uint32_t)d);
  return n / d;
}

MLA_HD int64_t worker_begin(int g, int64_t T, int G) { return div_floor((int64_t)g * T, G); }

// Largest g with worker_begin(g) <= x, i.e. the worker owning tile x.
MLA_HD int worker_of(int64_t x, int64_t T, int G) {
  const int64_t g = div_floor((x + 1) * (int64_t)G - 1, T);
  return (int)(g < G - 1 ? g : G - 1);
}

// Exclusive prefix of tiles_of(effective_len(b), tile) over b into pre[0..B]
// (shared memory); every thread of the block takes part.  Invalid lengths
// are reported once, by the thread that scans them.
// When `lens` is given, the validated lengths are stored there too (shared memory).
MLA_DEVI void tile_prefix(const int32_t* seqlens, int B, int64_t cap, int32_t* status, int* pre,
                          int tile = kTileTokens, int* lens = nullptr) {
  const int tid = threadIdx.x, nthr = blockDim.x;
  const int per = (B + nthr - 1) / nthr;
  const int b0 = tid * per, b1 = min(B, b0 + per);
  int local = 0;
  for (int b = b0; b < b1; ++b) {
    const int L = effective_len(seqlens, b, cap, status);
    if (lens) lens[b] = L;
    local += tiles_of(L, tile);
  }
  __shared__ int warp_sums[32];
  const int lane = tid & 31, warp = tid >> 5;
  int incl = local;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) warp_sums[warp] = incl;
  __syncthreads();
  int warp_off = 0;
  for (int w = 0; w < warp; ++w) warp_off += warp_sums[w];
  int run = warp_off + incl - local;
  for (int b = b0; b < b1; ++b) {
    pre[b] = run;
    run += tiles_of(lens ? lens[b] : effective_len(seqlens, b, cap, nullptr), tile);
  }
  if (tid == nthr - 1) pre[B] = run;  // the last thread's running sum is the total
  __syncthreads();
}

// The sequence owning tile x: the largest b with pre[b] <= x.
MLA_HD int seq_of_tile(const int* pre, int B, int64_t x) {
  int lo = 0, hi = B - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (pre[mid] <= x) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// ---------------------------------------------------------------- sequence-aligned plan
// (tensor-core decode) Sequence b with t_b > 0 tiles is cut into w_b entries,
//   w_b = min(t_b, 1 + floor((G - n) t_b / T))    (w_b = 1 when G <= n),
// n = number of non-empty sequences, T = total tiles, G = workers.  Entry k of
// b covers tiles [floor(t_b k / w_b), floor(t_b (k+1) / w_b)) (never empty, as
// w_b <= t_b), and the entries total at most max(G, n).  Worker g takes
// entries [floor(g E / G), floor((g+1) E / G)), so a worker never straddles
// two sequences when E <= G (each one writes a single partial, with no second
// epilogue or query reload), and otherwise takes whole sequences.  Entry e's
// partial lives in slot e.
MLA_HD int plan_entries(int t, int64_t T, int n, int G) {
  if (t <= 0) return 0;
  if (G <= n) return 1;
  const int64_t w = 1 + div_floor((int64_t)(G - n) * t, T);
  return (int)(w < t ? w : t);
}
MLA_HD int entry_start(int k, int t, int w) { return (int)div_floor((int64_t)t * k, w); }
// The entry (index within its sequence) holding tile tau of a sequence of t tiles.
MLA_HD int entry_of_tile(int tau, int t, int w) { return (int)div_floor((int64_t)(tau + 1) * w - 1, t); }

// Exclusive prefix of plan_entries over b into W[0..B] (shared memory), from the
// tile prefix pre[0..B]; every thread of the block takes part and gets the same
// return value: whether the sequence-aligned plan is preferred over the even
// split of the tile list.  The aligned plan costs its longest entry (tiles); the
// even split costs at most Q + kSegPenaltyTiles * ceil(Q / t_min) (Q = ceil(T/G)
// tiles per worker, t_min the shortest non-empty sequence; a worker can meet at
// most that many sequence boundaries, and each extra sequence costs one more
// partial write and a query reload, ~kSegPenaltyTiles 128-token tile times).
// Uniform batches keep the aligned plan (16 x 4096 over 74 workers: 8 vs 10);
// many ragged sequences take the even split (64 sequences of 1024..8192
// tokens: 64 vs 48).
constexpr int kSegPenaltyTiles = 3;
// The choice itself: cost_aligned = the aligned plan's longest entry (tiles),
// T total tiles, G workers, t_min the shortest non-empty sequence's tiles.
MLA_HD bool prefer_aligned(int cost_aligned, int64_t T, int G, int t_min) {
  if (T == 0) return true;
  const int64_t q = div_floor(T + G - 1, G);
  const int64_t cost_split = q + (int64_t)kSegPenaltyTiles * div_floor(q + t_min - 1, t_min);
  return cost_aligned <= cost_split;
}
MLA_DEVI bool plan_prefix(const int* pre, int B, int G, int* W) {
  const int tid = threadIdx.x, nthr = blockDim.x, lane = tid & 31, warp = tid >> 5;
  const int per = (B + nthr - 1) / nthr;
  const int b0 = tid * per, b1 = min(B, b0 + per);
  __shared__ int red[32], redmin[32], redmax[32];
  __shared__ int s_n, s_tmin;
  int n = 0, tmin = INT_MAX;
  for (int b = b0; b < b1; ++b) {
    const int t = pre[b + 1] - pre[b];
    if (t > 0) {
      ++n;
      tmin = min(tmin, t);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    n += __shfl_xor_sync(0xffffffffu, n, o);
    tmin = min(tmin, __shfl_xor_sync(0xffffffffu, tmin, o));
  }
  if (lane == 0) {
    red[warp] = n;
    redmin[warp] = tmin;
  }
  __syncthreads();
  if (tid == 0) {
    int t = 0, m = INT_MAX;
    for (int w = 0; w < (nthr + 31) / 32; ++w) {
      t += red[w];
      m = min(m, redmin[w]);
    }
    s_n = t;
    s_tmin = m;
  }
  __syncthreads();
  const int64_t T = pre[B];
  int local = 0, lmax = 0;
  for (int b = b0; b < b1; ++b) {
    const int t = pre[b + 1] - pre[b];
    const int w = plan_entries(t, T, s_n, G);
    local += w;
    if (w > 0) lmax = max(lmax, (t + w - 1) / w);
  }
  int incl = local;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) lmax = max(lmax, __shfl_xor_sync(0xffffffffu, lmax, o));
  __syncthreads();  // red[] is reused
  if (lane == 31) red[warp] = incl;
  if (lane == 0) redmax[warp] = lmax;
  __syncthreads();
  int warp_off = 0, cost_aligned = 0;
  for (int w = 0; w < (nthr + 31) / 32; ++w) {
    if (w < warp) warp_off += red[w];
    cost_aligned = max(cost_aligned, redmax[w]);
  }
  int run = warp_off + incl - local;
  for (int b = b0; b < b1; ++b) {
    W[b] = run;
    run += plan_entries(pre[b + 1] - pre[b], T, s_n, G);
  }
  if (tid == nthr - 1) W[B] = run;
  __syncthreads();
  return prefer_aligned(cost_aligned, T, G, s_tmin);
}

// One warp builds the whole plan (tensor-core decode prologue): validated
// lengths lens[0..B), tile prefix pre[0..B] and entry prefix W[0..B] in shared
// memory, the same values as tile_prefix + plan_prefix; every lane returns
// whether the sequence-aligned plan is preferred.  Only warp shuffles and
// __syncwarp: no block-wide barrier, so the other warps of the block can set up
// barriers and tensor memory meanwhile (the block-wide version cost ~2 us of
// serial barriers and loops at the start of every CTA).
MLA_DEVI bool warp_plan(const int32_t* seqlens, int B, int64_t cap, int32_t* status, int G, int tile, int* lens,
                        int* pre, int* W) {
  const int lane = threadIdx.x & 31;
  for (int b = lane; b < B; b += 32) lens[b] = effective_len(seqlens, b, cap, status);
  __syncwarp();
  const int per = (B + 31) / 32, b0 = min(B, lane * per), b1 = min(B, b0 + per);
  int tl = 0, n = 0, tmin = INT_MAX;
  for (int b = b0; b < b1; ++b) {
    const int t = tiles_of(lens[b], tile);
    tl += t;
    if (t > 0) {
      ++n;
      tmin = min(tmin, t);
    }
  }
  int incl = tl;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    n += __shfl_xor_sync(0xffffffffu, n, o);
    tmin = min(tmin, __shfl_xor_sync(0xffffffffu, tmin, o));
  }
  const int T = __shfl_sync(0xffffffffu, incl, 31);
  int run = incl - tl, wl = 0, cost = 0;
  for (int b = b0; b < b1; ++b) {
    pre[b] = run;
    const int t = tiles_of(lens[b], tile);
    run += t;
    const int w = plan_entries(t, T, n, G);
    wl += w;
    if (w > 0) cost = max(cost, (t + w - 1) / w);
  }
  int winc = wl;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, winc, o);
    if (lane >= o) winc += v;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) cost = max(cost, __shfl_xor_sync(0xffffffffu, cost, o));
  int wr = winc - wl;
  for (int b = b0; b < b1; ++b) {
    W[b] = wr;
    wr += plan_entries(tiles_of(lens[b], tile), T, n, G);
  }
  if (lane == 31) {
    pre[B] = T;
    W[B] = winc;
  }
  __syncwarp();
  return prefer_aligned(cost, T, G, tmin);
}

// The sequence owning entry e < W[B]: the largest b with W[b] <= e.
MLA_HD int seq_of_entry(const int* W, int B, int64_t e) { return seq_of_tile(W, B, e); }

// First global tile of entry e (T for e == E).
MLA_HD int64_t entry_tile(const int* pre, const int* W, int B, int64_t e) {
  if (e >= W[B]) return pre[B];
  const int b = seq_of_entry(W, B, e);
  const int t = pre[b + 1] - pre[b], w = W[b + 1] - W[b];
  return pre[b] + entry_start((int)(e - W[b]), t, w);
}

}  // namespace mla

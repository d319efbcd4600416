// Split-KV work partition shared by the decode partial kernels and the combine.
//
// Every sequence b is cut into ceil(L_b / 64) tiles; the tiles of all
// sequences, in batch order, form one list of T tiles.  Worker g of G owns
// the contiguous range [floor(g T / G), floor((g+1) T / G)), which may cover
// the end of one sequence and the start of the next.  Each (worker, sequence)
// segment writes one partial (o, lse) to slot g + b; slots are unique because
// worker ranges are ordered (if worker g touches sequence b, worker g + 1
// starts at b or later).  The combine merges, for sequence b, the slots of
// workers g_first(b) .. g_last(b) whose range meets b's tiles.
#pragma once

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

MLA_DEVI int tiles_of(int L, int tile = kTileTokens) { return (L + tile - 1) / tile; }

MLA_DEVI int64_t worker_begin(int g, int64_t T, int G) { return (int64_t)g * T / G; }

// Largest g with worker_begin(g) <= x, i.e. the worker owning tile x.
MLA_DEVI int worker_of(int64_t x, int64_t T, int G) {
  const int64_t g = ((x + 1) * (int64_t)G - 1) / T;
  return (int)(g < G - 1 ? g : G - 1);
}

// Exclusive prefix of tiles_of(effective_len(b), tile) over b into pre[0..B]
// (shared memory); every thread of the block takes part.  Invalid lengths
// are reported once, by the thread that scans them.
MLA_DEVI void tile_prefix(const int32_t* seqlens, int B, int64_t cap, int32_t* status, int* pre,
                          int tile = kTileTokens) {
  const int tid = threadIdx.x, nthr = blockDim.x;
  const int per = (B + nthr - 1) / nthr;
  const int b0 = tid * per, b1 = min(B, b0 + per);
  int local = 0;
  for (int b = b0; b < b1; ++b) local += tiles_of(effective_len(seqlens, b, cap, status), tile);
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
    run += tiles_of(effective_len(seqlens, b, cap, nullptr), tile);
  }
  if (tid == nthr - 1) pre[B] = run;  // the last thread's running sum is the total
  __syncthreads();
}

// The sequence owning tile x: the largest b with pre[b] <= x.
MLA_DEVI int seq_of_tile(const int* pre, int B, int64_t x) {
  int lo = 0, hi = B - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (pre[mid] <= x) lo = mid; else hi = mid - 1;
  }
  return lo;
}

}  // namespace mla

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

MLA_DEVI int tiles_of(int L) { return (L + kTileTokens - 1) / kTileTokens; }

MLA_DEVI int64_t worker_begin(int g, int64_t T, int G) { return (int64_t)g * T / G; }

// Largest g with worker_begin(g) <= x, i.e. the worker owning tile x.
MLA_DEVI int worker_of(int64_t x, int64_t T, int G) {
  const int64_t g = ((x + 1) * (int64_t)G - 1) / T;
  return (int)(g < G - 1 ? g : G - 1);
}

}  // namespace mla

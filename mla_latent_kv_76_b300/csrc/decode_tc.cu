// Tensor-core split-KV decode for the DeepSeek-V3 head shape: n_h = 128,
// d_c = 512, d_R = 64 (576-wide cache rows), on tcgen05 / TMEM / TMA.
//
// What is computed ("结合 DeepSeek 推理代码看 MLA": score = (q^C W^UK).c^KV +
// q^R.k^R; worked example steps 4-5: scale, causal mask, softmax, z = A.kv):
// for every head i and visible token j of a sequence
//   s_j = scale * [q~_i ; q^R_i] . [c_j ; k^R_j],   z_i = sum_j softmax(s)_j c_j.
//
// Decomposition.  The fp32 accumulator O = 128 heads x 512 latent fills the
// whole tensor memory of one SM, so each 128-token tile is shared by the two
// CTAs of a cluster (one per SM), split by contraction rather than by columns:
//   score CTA (rank 0)  S = [q~; q^R] . [c; k^R]^T over all 576 columns,
//                       M = 128 heads x N = 128 tokens per tcgen05.mma, with
//                       the query held in TMEM; online softmax; the bf16
//                       weights P go to the peer through distributed shared
//                       memory (16 KB per 64 tokens, the only exchange).
//   value CTA (rank 1)  O += P . C[:, 0:512] (M = 128, N = 256, K = 64 tokens
//                       per half tile), the whole accumulator in TMEM.
// Every cache byte is read from HBM once by the score CTA; the value CTA
// re-reads the latent columns a few microseconds later, from L2.
//
// Score CTA, 384 threads: warp 0 lane 0 TMA producer (a ring of 3 slots,
// each three 64-column chunks of 128 tokens, 128-byte swizzle; the first
// segment's query arrives through the ring ahead of tile 0), warp 1 MMA issue
// (S double-buffered in TMEM; one barrier wait and one commit per 12 MMAs),
// warps 4-7 / 8-11 softmax for token columns 0-63 / 64-127 (thread = head),
// warps 2 / 3 ship each warpgroup's P to the value CTA as one bulk copy.
// Value CTA: warp 0 lane 0 TMA (2 stages of 64 tokens x 512 columns, one 64 KB
// box each), warp 1 MMA, warp 2 lane 0 the ring helper (paged cache: it loads
// part of every score slot into the score CTA's ring, multicast to rank 0),
// warp 3 zeroes the rows past the sequence end in the last half tile (NaN
// garbage must not meet a zero weight), warps 4-11 rescale O and write the
// segment's partial (thread = head, two column halves).  The value MMA thread
// frees the score CTA's staging once a P has landed, and its commit after the
// MMAs that read a P buffer arrives on the score CTA's barrier for that buffer.
//
// Copies are few and large: an SM's TMA unit completes a roughly fixed number
// of copies per microsecond whatever their size up to ~24 KB (measured on
// B300), and copies issued from several lanes of one warp were slower than
// from one thread.  On the contiguous cache a slot is one 4-D box; on the
// paged cache a chunk's two 64-token halves come from unrelated blocks, so a
// slot takes six 8 KB boxes, shared between the two SMs' TMA units.
//
// Online softmax with a lazily updated reference maximum m_ref (base 2):
// P = 2^(x - m_ref); m_ref moves, and O and the weight sums are rescaled, only
// when a tile's maximum exceeds m_ref by more than kRescaleThreshold.  P is
// rounded to bf16 for the value MMA (kind::f16 takes bf16 operands).  Two sums
// are kept: lq of the rounded weights normalises z, so z is an exact convex
// combination of the weights the MMA multiplied; l of the fp32 weights gives
// lse.  The partial of a segment is O unnormalised plus (m_ref, l, lq); the
// combine kernel merges partials exactly.
#include <cuda.h>
#include <mutex>

#include "common.cuh"
#include "kernels.h"
#include "plan.cuh"
#include "tc.cuh"

namespace mla {
namespace {

constexpr int kH = 128, kDC = 512, kD = 576;
constexpr int kTile = 128;           // tokens per score tile (two 64-token halves)
constexpr int kThreads = 384;
constexpr int kTcMaxBatch = 1024;
constexpr float kRescaleThreshold = 16.f;

// ---- P hand-off unit: 64 tokens of bf16 weights for 128 heads, then metadata
constexpr int kPBytes = kH * 128;                  // 128 heads x 64 tokens bf16 (SW128 K-major)
constexpr int kPMetaAlpha = kPBytes;               // alpha[128] fp32
constexpr int kPMetaFlags = kPBytes + 512;         // flag[4] int32 (per warp: O must be rescaled)
constexpr int kPBufBytes = kPBytes + 1024;
// ---- score CTA shared memory
constexpr int kChunk128 = kTile * 128;            // 128 tokens x 64 bf16 columns
constexpr int kSlots = 3;                          // slot t holds chunks 3t .. 3t + 2 of a tile
constexpr int kSlotBytes = 3 * kChunk128;
constexpr int kOffRing = 0;
constexpr int kOffQrope = kOffRing + kSlots * kSlotBytes;  // RoPE part of Q, 128 heads x 64 bf16 (SW128)
constexpr int kOffStaging = kOffQrope + kH * 128;          // [2 wg] P hand-off staging
constexpr int kOffXmax = kOffStaging + 2 * kPBufBytes;     // [2 parity][2 wg][128] fp32
constexpr int kOffLsum = kOffXmax + 2 * 2 * kH * 4;        // [2][128] fp32: weight sums of warpgroup 1
// ---- value CTA shared memory
constexpr int kVStages = 2;
constexpr int kChunkBytes = 64 * 128;              // 64 tokens x 64 bf16 columns
constexpr int kVStageBytes = 8 * kChunkBytes;      // the 512 latent columns of 64 tokens
constexpr int kPBufs = 4;
constexpr int kOffStage = 0;
constexpr int kOffP = kOffStage + kVStages * kVStageBytes;  // [4] P hand-off buffers
// ---- common tail
constexpr int kOffBar = (kOffLsum + 2 * kH * 4 > kOffP + kPBufs * kPBufBytes) ? kOffLsum + 2 * kH * 4
                                                                             : kOffP + kPBufs * kPBufBytes;
constexpr int kNumBars = 40;
constexpr int kOffMisc = kOffBar + kNumBars * 8;   // tmem base, abort flag, event descriptor, plan scalars
constexpr int kOffPrefix = kOffMisc + 64;          // lens[B], pre[B + 1], W[B + 1]

// score CTA barriers
constexpr int kBarCfull = 0, kBarCempty = 3, kBarSfull = 20, kBarSfree = 22, kBarQready = 24, kBarPfree = 25,
              kBarScDrained = 29, kBarXmax = 30, kBarLsum = 32, kBarStgFull = 33, kBarStgFree = 35, kBarQrope = 37;
// value CTA barriers
// kBarRingFree + t mirrors the score CTA's kBarCempty + t (same offset; the
// score MMA thread's commits arrive on both): the value CTA's ring helper
// waits on it before loading into the score CTA's slot t
constexpr int kBarRingFree = kBarCempty;
constexpr int kBarFull = 0, kBarEmpty = 10, kBarFix = 12, kBarPfull = 6, kBarOcomp = 14, kBarEvt = 15,
              kBarEvtdone = 16, kBarVcDrained = 17;

// TMEM columns
// score CTA: S double buffer [0, 256) (128 tokens each), the query's 512 latent
// columns as packed bf16 [256, 512); its 64 RoPE columns live in shared memory
constexpr uint32_t kColS = 0, kColQ = 256;

enum { kEvtRescale = 1, kEvtEpilogue = 2, kEvtExit = 3 };

size_t tc_smem_bytes(int batch) { return (size_t)kOffPrefix + (3 * (size_t)batch + 2) * 4 + 1024; }
static_assert(kOffPrefix + (3 * kTcMaxBatch + 2) * 4 + 1024 <= 227 * 1024, "shared memory of one CTA");

struct TcParams {
  const __nv_bfloat16* q;
  const __nv_bfloat16* pool;
  const int32_t* block_table;
  int32_t max_blocks;
  int32_t num_blocks;
  int64_t seq_stride;
  const int32_t* seqlens;
  int32_t batch;
  int32_t paged;
  float scale_log2;
  int32_t workers;  // CTA pairs
  float* o_part;    // [(G + B)][128 float4 columns][128 heads][4]  unnormalised
  float* m_part;    // [(G + B)][128]       reference maximum, log2 units
  float* l_part;    // [(G + B)][128]       sum of the fp32 weights relative to m_part (for lse)
  float* lq_part;   // [(G + B)][128]       sum of the bf16-rounded weights the MMA used (normalises z)
  int32_t* status;
  int32_t* plan_hdr;   // [plan kind (1: sequence-aligned, 0: even tile split), tiles T, workers G] for the combine
  int32_t* seqplan;    // [B][2] for the combine: sequence b's partial slots (aligned) or workers (even split)
};

struct Seg {
  int b, t_begin, ntile, len;
};

MLA_DEVI Seg seg_at(const int* pre, const int* lens, int B, int64_t x, int64_t hi) {
  Seg s;
  s.b = seq_of_tile(pre, B, x);
  s.t_begin = (int)(x - pre[s.b]);
  const int64_t e = pre[s.b + 1] < hi ? pre[s.b + 1] : hi;
  s.ntile = (int)(e - x);
  s.len = lens[s.b];
  return s;
}

// 64-token halves of tile tt that hold visible tokens (1 or 2).
MLA_DEVI int halves_of(const Seg& s, int tt) { return min(2, (s.len - tt * kTile + 63) >> 6); }

// Does half w of tile tt contain the sequence end with a partial block?
MLA_DEVI bool half_is_tail(const Seg& s, int tt, int w) {
  const int lo = tt * kTile + 64 * w;
  return (s.len & 63) != 0 && lo <= s.len - 1 && s.len - 1 < lo + 64;
}

// Paged block id of half w of tile tt, or -1 if it is out of range.
MLA_DEVI int half_block(const TcParams& p, const Seg& s, int tt, int w) {
  const int lb = 2 * tt + w;
  if (lb >= p.max_blocks) return -1;
  const int blk = p.block_table[(int64_t)s.b * p.max_blocks + lb];
  return (blk >= 0 && blk < p.num_blocks) ? blk : -1;
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    decode_tc_kernel(const __grid_constant__ CUtensorMap map_s, const __grid_constant__ CUtensorMap map_v,
                     const __grid_constant__ CUtensorMap q_map, const __grid_constant__ CUtensorMap q_map3,
                     const TcParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + kOffBar);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + kOffMisc);
  int* abort_flag = reinterpret_cast<int*>(sm + kOffMisc + 4);
  volatile int* evt_desc = reinterpret_cast<volatile int*>(sm + kOffMisc + 8);  // type, buffer, slot
  int64_t* range = reinterpret_cast<int64_t*>(sm + kOffMisc + 32);                // this worker's [lo, hi)
  int* aligned_s = reinterpret_cast<int*>(sm + kOffMisc + 48);
  int* lens = reinterpret_cast<int*>(sm + kOffPrefix);
  int* pre = lens + p.batch;
  int* Wp = pre + p.batch + 1;  // entries prefix of the split plan

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t rank = tc::cluster_rank();
  const int g = (int)(blockIdx.x >> 1);
  const int64_t cap = p.paged ? (int64_t)p.max_blocks * 64 : p.seq_stride;

  // Prologue, three warps in parallel: warp 0 builds the split plan (lengths,
  // tile and entry prefixes, this worker's tile range), warp 1 allocates tensor
  // memory, warp 2 initialises the barriers.
  if (warp == 0) {
    const bool al = warp_plan(p.seqlens, p.batch, cap, p.status, p.workers, kTile, lens, pre, Wp);
    if (lane == 0) {
      const int B = p.batch, G = p.workers;
      const int64_t E = Wp[B], T = pre[B];
      // worker g's contiguous run of tiles: entries [g E / G, (g + 1) E / G) of the
      // sequence-aligned plan, or the even split [g T / G, (g + 1) T / G)
      range[0] = al ? entry_tile(pre, Wp, B, div_floor((int64_t)g * E, G)) : worker_begin(g, T, G);
      range[1] = al ? entry_tile(pre, Wp, B, div_floor((int64_t)(g + 1) * E, G)) : worker_begin(g + 1, T, G);
      *aligned_s = al ? 1 : 0;
      if (blockIdx.x == 0) {
        p.plan_hdr[0] = al ? 1 : 0;
        p.plan_hdr[1] = (int)T;
        p.plan_hdr[2] = G;
      }
    }
    if (blockIdx.x == 0) {
      // which partials the combine merges for each sequence: slots first..last of
      // the aligned plan, or the workers first..last of the even split (slot g + b;
      // workers without tiles in between wrote nothing); last < first: no tiles
      const int B = p.batch, G = p.workers, T = pre[B];
      for (int b = lane; b < B; b += 32) {
        const int t = pre[b + 1] - pre[b];
        int first = 0, last = -1;
        if (t > 0) {
          first = al ? Wp[b] : worker_of(pre[b], T, G);
          last = al ? Wp[b + 1] - 1 : worker_of(pre[b + 1] - 1, T, G);
        }
        p.seqplan[2 * b] = first;
        p.seqplan[2 * b + 1] = last;
      }
    }
    // the combine may be scheduled now; it waits for this grid to finish before reading
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  } else if (warp == 1) {
    tc::tmem_alloc(tmem_slot, 512);
  } else if (tid == 64) {
    if (rank == 0) {
      for (int i = 0; i < kSlots; ++i) {
        // the producer's expect_tx (+ the copies' bytes), on the paged cache also
        // the value CTA ring helper's arrival: the helper then takes part in
        // every fill, so this CTA can never run two fills ahead of it
        tc::mbar_init(&bars[kBarCfull + i], p.paged ? 2 : 1);
        tc::mbar_init(&bars[kBarCempty + i], 1);
      }
      tc::mbar_init(&bars[kBarQrope], 1);
      for (int i = 0; i < 2; ++i) {
        tc::mbar_init(&bars[kBarSfull + i], 1);
        tc::mbar_init(&bars[kBarSfree + i], 256);
        tc::mbar_init(&bars[kBarStgFull + i], 128);
        tc::mbar_init(&bars[kBarStgFree + i], 1);
      }
      tc::mbar_init(&bars[kBarQready], 256);
      for (int i = 0; i < kPBufs; ++i) tc::mbar_init(&bars[kBarPfree + i], 1);
      tc::mbar_init(&bars[kBarScDrained], 1);
      tc::mbar_init(&bars[kBarXmax], 256);
      tc::mbar_init(&bars[kBarXmax + 1], 256);
      tc::mbar_init(&bars[kBarLsum], 256);
    } else {
      for (int i = 0; i < kVStages; ++i) {
        tc::mbar_init(&bars[kBarFull + i], 1);  // the producer's expect_tx (+ the copy's bytes)
        tc::mbar_init(&bars[kBarEmpty + i], 1 + 32);
        tc::mbar_init(&bars[kBarFix + i], 32);
      }
      for (int i = 0; i < kPBufs; ++i) {
        tc::mbar_init(&bars[kBarPfull + i], 1);  // the score CTA's expect_tx arrival + the copy
      }
      tc::mbar_init(&bars[kBarOcomp], 1);
      tc::mbar_init(&bars[kBarEvt], 1);
      tc::mbar_init(&bars[kBarEvtdone], 256);
      tc::mbar_init(&bars[kBarVcDrained], 1);
      for (int i = 0; i < kSlots; ++i) tc::mbar_init(&bars[kBarRingFree + i], 1);
    }
    *abort_flag = 0;
    tc::fence_mbar_init();
  }
  tc::tc_fence_before();
  tc::cluster_sync();  // the plan and both CTAs' barriers are visible before any use or remote arrival
  tc::tc_fence_after();
  const uint32_t tb = *tmem_slot;
  const tc::Abort ab{abort_flag, p.status};

  const int B = p.batch;
  const int64_t lo = range[0], hi = range[1];
  const bool aligned = *aligned_s != 0;
  // the partial slot of a segment: the plan entry it starts with, or worker + sequence
  auto slot_of = [&](const Seg& s) -> int64_t {
    if (!aligned) return (int64_t)g + s.b;
    const int t = pre[s.b + 1] - pre[s.b], w = Wp[s.b + 1] - Wp[s.b];
    return (int64_t)Wp[s.b] + entry_of_tile(s.t_begin, t, w);
  };

  if (rank == 0) {
    // ================================================================ score CTA
    if (warp == 0) {
      if (lane == 0) {
        // ---------------------------------------------------------- TMA producer (one thread)
        // A copy costs the SM's TMA unit a roughly fixed time up to ~24 KB
        // (measured on B300: ~2.6 copies/us per SM), so on the contiguous cache a
        // ring slot (three 64-column chunks of 128 tokens) is one 48 KB 4-D box.
        // On the paged cache a chunk's two 64-token halves come from two blocks
        // at unrelated addresses and must land 8 KB apart, so a slot takes six
        // 8 KB boxes.  Copies from divergent lanes of one warp were slower still
        // than from one thread.
        tc::prefetch_map(&map_s);
        bool ok = true;
        int m = 0;                      // tiles loaded so far
        int fills[kSlots] = {0, 0, 0};  // fills issued per slot (for the exit drain)
        // Fill 0 of the ring is the first segment's query (128 heads x 576, the
        // same 128-byte-swizzled chunk layout): chunks 0-7 into the three slots
        // for the MMA thread to copy into tensor memory (which frees each slot
        // for tile 0), the RoPE chunk (8) straight to its own buffer.
        if (lo < hi) {
          const int b0 = seq_of_tile(pre, B, lo);
          tc::mbar_expect_tx(&bars[kBarCfull + 0], 3 * kChunk128);
          tc::tma_load_4d(sm + kOffRing, &q_map, 0, 0, 0, b0, &bars[kBarCfull + 0]);
          tc::mbar_expect_tx(&bars[kBarCfull + 1], 3 * kChunk128);
          tc::tma_load_4d(sm + kOffRing + kSlotBytes, &q_map, 0, 0, 3, b0, &bars[kBarCfull + 1]);
          tc::mbar_expect_tx(&bars[kBarCfull + 2], 2 * kChunk128);
          tc::tma_load_3d(sm + kOffRing + 2 * kSlotBytes, &q_map3, 6 * 64, 0, b0, &bars[kBarCfull + 2]);
          tc::tma_load_3d(sm + kOffRing + 2 * kSlotBytes + kChunk128, &q_map3, 7 * 64, 0, b0, &bars[kBarCfull + 2]);
          tc::mbar_expect_tx(&bars[kBarQrope], kChunk128);
          tc::tma_load_3d(sm + kOffQrope, &q_map3, 8 * 64, 0, b0, &bars[kBarQrope]);
          for (int t = 0; t < kSlots; ++t) fills[t] = 1;
        }
        for (int64_t x = lo; x < hi && ok;) {
          const Seg s = seg_at(pre, lens, B, x, hi);
          x += s.ntile;
          // the next segment's query (147 KB) is warmed in L2 a whole segment ahead
          if (x < hi) tc::prefetch_l2(p.q + (int64_t)seq_of_tile(pre, B, x) * kH * kD, (uint32_t)(kH * kD * 2));
          for (int j = 0; j < s.ntile && ok; ++j, ++m) {
            const int tt = s.t_begin + j;
            const int nh = p.paged ? halves_of(s, tt) : 0;
            int blk[2] = {-1, -1};
            for (int w = 0; w < nh; ++w) {
              blk[w] = half_block(p, s, tt, w);
              if (blk[w] < 0) report(p.status, MLA_ERR_DEVICE_BOUNDS);
            }
#pragma unroll 1
            for (int t = 0; t < kSlots; ++t) {
              if (!tc::wait<false>(&bars[kBarCempty + t], m & 1, ab)) {  // fill m (0: the query) consumed
                ok = false;
                break;
              }
              uint8_t* dst = sm + kOffRing + t * kSlotBytes;
              uint64_t* fb = &bars[kBarCfull + t];
              ++fills[t];
              if (p.paged) {
                // chunk 3t + cc of block w (the tile's 64-token half w) at dst + cc * 16 KB + w * 8 KB
                int nvalid = 0;
                for (int w = 0; w < nh; ++w) {
                  if (blk[w] >= 0) {
                    ++nvalid;
                  } else {  // unreadable block: its rows count as zeros
                    for (int cc = 0; cc < 3; ++cc) {
                      uint4* z = reinterpret_cast<uint4*>(dst + cc * kChunk128 + w * kChunkBytes);
                      for (int i = 0; i < kChunkBytes / 16; ++i) z[i] = make_uint4(0, 0, 0, 0);
                    }
                  }
                }
                if (nvalid < nh) tc::fence_async_smem();
                if (nvalid == 0) {
                  tc::mbar_arrive(fb);
                  continue;
                }
                // this CTA copies the first half's boxes of slots 0 and 1; the value
                // CTA's ring helper copies the rest into this slot (both signal this
                // barrier), so the two SMs' TMA units share the tile's copies
                tc::mbar_expect_tx(fb, nvalid * 3 * kChunkBytes);
                if (blk[0] >= 0 && t < kSlots - 1)  // the helper takes both halves of the last slot
                  for (int cc = 0; cc < 3; ++cc)
                    tc::tma_load_4d(dst + cc * kChunk128, &map_s, 0, 0, 3 * t + cc, blk[0], fb);
              } else {
                // contiguous cache: 128 tokens x chunks 3t .. 3t + 2, chunk-major (rows
                // past the sequence are masked by the softmax; past the allocation they
                // read as zero)
                tc::mbar_expect_tx(fb, kSlotBytes);
                tc::tma_load_4d(dst, &map_s, 0, tt * kTile, 3 * t, s.b, fb);
              }
            }
          }
        }
        // no copy in flight at exit: the last fill of every slot has landed
        for (int t = 0; t < kSlots; ++t)
          if (fills[t] > 0) tc::wait_drain<false>(&bars[kBarCfull + t], (fills[t] - 1) & 1, ab);
        if (lo < hi) tc::wait_drain<false>(&bars[kBarQrope], 0, ab);
      }
    } else if (warp == 1) {
      if (lane == 0) {
        // ---------------------------------------------------------- score MMA
        constexpr uint32_t idS = tc::idesc_bf16(128, kTile, 0, 0);
        const uint32_t ring = smem_u32(sm + kOffRing);
        const uint32_t qrope = smem_u32(sm + kOffQrope);
        int m = 0, k = 0;
        bool ok = true;
        for (int64_t x = lo; x < hi && ok; ++k) {
          const Seg s = seg_at(pre, lens, B, x, hi);
          x += s.ntile;
          if (k == 0) {
            // the first segment's query, ring fill 0: latent chunks 0-7 into tensor
            // memory (the copies run ahead of the MMAs issued below), then each
            // slot goes back to the producer; the RoPE chunk is read in place
#pragma unroll
            for (int t = 0; t < kSlots; ++t) {
              if (!tc::wait<false>(&bars[kBarCfull + t], 0, ab)) {
                ok = false;
                break;
              }
              tc::tc_fence_after();
#pragma unroll
              for (int cc = 0; cc < 3; ++cc) {
                const int c = 3 * t + cc;
                if (c < 8)
#pragma unroll
                  for (int kk = 0; kk < 4; ++kk)
                    tc::tmem_cp_128x256b(tb + kColQ + c * 32 + kk * 8,
                                         tc::smem_desc(ring + t * kSlotBytes + cc * kChunk128 + kk * 32, 16, 1024));
              }
              tc::mma_commit_multicast(&bars[kBarCempty + t], 3);  // and the value CTA's mirror
            }
            if (!ok || !tc::wait<false>(&bars[kBarQrope], 0, ab)) break;
          } else if (!tc::wait<false>(&bars[kBarQready], (k - 1) & 1, ab)) {  // a later segment's query
            break;
          }
          for (int j = 0; j < s.ntile && ok; ++j, ++m) {
            // S is double-buffered: buffer m & 1 is free once the softmax read tile m - 2
            if (m >= 2 && !tc::wait<false>(&bars[kBarSfree + (m & 1)], ((m >> 1) - 1) & 1, ab)) {
              ok = false;
              break;
            }
            tc::tc_fence_after();
            const uint32_t dS = tb + kColS + (m & 1) * kTile;
            // straight-line issue: per ring slot (three chunks) one wait, twelve MMAs, one commit
#pragma unroll
            for (int t = 0; t < kSlots; ++t) {
              if (!tc::wait<false>(&bars[kBarCfull + t], (m + 1) & 1, ab)) {  // phase 0 held the query
                ok = false;
                break;
              }
              tc::tc_fence_after();
              {
                // chunk c of the slot: 128 tokens x 64 columns, N = 128
#pragma unroll
                for (int cc = 0; cc < 3; ++cc) {
                  const int c = 3 * t + cc;
                  const uint32_t sa = ring + t * kSlotBytes + cc * kChunk128;
                  if (c < 8) {
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                      tc::mma_ts(dS, tb + kColQ + c * 32 + kk * 8, tc::smem_desc(sa + kk * 32, 16, 1024), idS,
                                 (c | kk) != 0 ? 1u : 0u);
                  } else {
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                      tc::mma_ss(dS, tc::smem_desc(qrope + kk * 32, 16, 1024), tc::smem_desc(sa + kk * 32, 16, 1024),
                                 idS, 1u);
                  }
                }
              }
              tc::mma_commit_multicast(&bars[kBarCempty + t], 3);  // and the value CTA's mirror
            }
            if (ok) tc::mma_commit(&bars[kBarSfull + (m & 1)]);
          }
        }
        tc::mma_commit(&bars[kBarScDrained]);
        tc::wait_drain<false>(&bars[kBarScDrained], 0, ab);
      }
    } else if (warp == 2 || warp == 3) {
      if (lane == 0) {
        // ---------------------------------------------------------- P hand-off for warpgroup (warp - 2)
        const int w = warp - 2;
        uint8_t* stg = sm + kOffStaging + w * kPBufBytes;
        const uint32_t r_p = tc::map_peer(sm + kOffP, 1);
        const uint32_t r_pfull = tc::map_peer(&bars[kBarPfull], 1);
        int hh = 0, u = 0;
        bool ok = true;
        for (int64_t x = lo; x < hi && ok;) {
          const Seg s = seg_at(pre, lens, B, x, hi);
          x += s.ntile;
          for (int j = 0; j < s.ntile && ok; ++j) {
            const int nh = halves_of(s, s.t_begin + j);
            if (w < nh) {
              const int hidx = hh + w;
              const int pb = hidx % kPBufs, up = hidx / kPBufs;
              if (!tc::wait<false>(&bars[kBarStgFull + w], u & 1, ab)) { ok = false; break; }
              if (up >= 1 && !tc::wait<true>(&bars[kBarPfree + pb], (up - 1) & 1, ab)) { ok = false; break; }
              // the value CTA's MMA thread frees the staging (kBarStgFree) once the copy landed
              tc::bulk_copy_to_peer(r_p + pb * kPBufBytes, stg, kPBufBytes, r_pfull + pb * 8);
              ++u;
            }
            hh += nh;
          }
        }
        // The value CTA's MMA commits arrive on kBarPfree asynchronously: before this
        // CTA may exit, the last arrival on every P buffer must have landed.
        if (w == 0 && ok)
          for (int pb = 0; pb < kPBufs; ++pb) {
            const int uses = (hh - pb + kPBufs - 1) / kPBufs;
            if (uses >= 1) tc::wait<true>(&bars[kBarPfree + pb], (uses - 1) & 1, ab);
          }
      }
    } else if (warp >= 4) {
      // ------------------------------------------------------------ softmax (thread = head)
      const int w = (warp - 4) >> 2;  // token columns [64 w, 64 w + 64) of each tile
      const int h = (tid - 128) & 127;
      const uint32_t lane_t = tb + ((uint32_t)((warp & 3) * 32) << 16);
      float* xmax = reinterpret_cast<float*>(sm + kOffXmax);
      float* lsum = reinterpret_cast<float*>(sm + kOffLsum);
      uint8_t* stg = sm + kOffStaging + w * kPBufBytes;  // this warpgroup's P hand-off staging
      int sends = 0;

      auto load_q = [&](int b) {
        const __nv_bfloat16* row = p.q + ((int64_t)b * kH + h) * kD;
        const uint4* src = reinterpret_cast<const uint4*>(row + 256 * w);  // latent [256 w, 256 w + 256)
        // RoPE columns [32 w, 32 w + 32) of the row: 16-byte pieces 4 w .. 4 w + 3 of a
        // 128-byte-swizzled K-major row; loaded with the first half of the latent part
        const uint4* srcr = reinterpret_cast<const uint4*>(row + kDC);
        uint4 rq[4];
#pragma unroll
        for (int c = 0; c < 4; ++c) rq[c] = __ldg(srcr + 4 * w + c);
#pragma unroll 1
        for (int c2 = 0; c2 < 2; ++c2) {  // 16 loads in flight per thread per round
          uint32_t r[2][32];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const uint4 v = __ldg(src + c2 * 16 + i);
            r[i >> 3][4 * (i & 7)] = v.x;
            r[i >> 3][4 * (i & 7) + 1] = v.y;
            r[i >> 3][4 * (i & 7) + 2] = v.z;
            r[i >> 3][4 * (i & 7) + 3] = v.w;
          }
          tc::tmem_st32(lane_t + kColQ + 128 * w + c2 * 64, r[0]);
          tc::tmem_st32(lane_t + kColQ + 128 * w + c2 * 64 + 32, r[1]);
        }
#pragma unroll
        for (int c = 0; c < 4; ++c)
          *reinterpret_cast<uint4*>(sm + kOffQrope + h * 128 + (((4 * w + c) ^ (h & 7)) * 16)) = rq[c];
        tc::fence_async_smem();
        tc::tmem_wait_st();
        tc::tc_fence_before();
        tc::mbar_arrive(&bars[kBarQready]);
      };

      int m = 0, hh = 0, k = 0;
      bool ok = true;
      for (int64_t x = lo; x < hi && ok; ++k) {
        const Seg s = seg_at(pre, lens, B, x, hi);
        x += s.ntile;
        float m_ref = -INFINITY, l = 0.f, lq = 0.f;
        for (int j = 0; j < s.ntile; ++j, ++m) {
          const int tt = s.t_begin + j;
          const int nh = halves_of(s, tt);
          if (!tc::wait<false>(&bars[kBarSfull + (m & 1)], (m >> 1) & 1, ab)) {
            ok = false;
            break;
          }
          tc::tc_fence_after();
          uint32_t sa[32], sb[32];
          const uint32_t sc = lane_t + kColS + (m & 1) * kTile + 64 * w;
          tc::tmem_ld32(sc, sa);
          tc::tmem_ld32(sc + 32, sb);
          tc::tmem_wait_ld();
          tc::tc_fence_before();
          tc::mbar_arrive(&bars[kBarSfree + (m & 1)]);
          const int nvalid = s.len - tt * kTile - 64 * w;  // may be <= 0
          if (nvalid < 64) {  // columns past the sequence end take no weight
#pragma unroll
            for (int c = 0; c < 32; ++c) {
              if (c >= nvalid) sa[c] = __float_as_uint(-INFINITY);
              if (c + 32 >= nvalid) sb[c] = __float_as_uint(-INFINITY);
            }
          }
          // maximum of the raw scores (the scale is positive, so it commutes with max)
          float mx[16];
#pragma unroll
          for (int i = 0; i < 16; ++i)
            mx[i] = fmaxf(tc::max3(__uint_as_float(sa[i]), __uint_as_float(sa[i + 16]), __uint_as_float(sb[i])),
                          __uint_as_float(sb[i + 16]));
#pragma unroll
          for (int i = 0; i < 5; ++i) mx[i] = tc::max3(mx[i], mx[i + 5], mx[i + 10]);
          float mt = fmaxf(tc::max3(mx[0], mx[1], mx[2]), tc::max3(mx[3], mx[4], mx[15])) * p.scale_log2;
          // tile maximum over both halves (bounded rendezvous of the two warpgroups)
          float* xm = xmax + (m & 1) * 2 * kH;
          xm[w * kH + h] = mt;
          tc::mbar_arrive(&bars[kBarXmax + (m & 1)]);
          if (!tc::wait<false>(&bars[kBarXmax + (m & 1)], (m >> 1) & 1, ab)) {
            ok = false;
            break;
          }
          mt = fmaxf(xm[h], xm[kH + h]);
          float alpha = 1.f;
          if (j == 0) {
            m_ref = mt;
          } else if (mt > m_ref + kRescaleThreshold) {
            alpha = exp2f(m_ref - mt);
            l *= alpha;
            lq *= alpha;
            m_ref = mt;
          }
          // P = 2^(s scale_log2 - m_ref), one fused multiply-add per pair: bf16 for
          // the value MMA; l sums the fp32 weights, lq the rounded ones
          uint32_t pk[32];
          {
            const uint64_t c2 = tc::f2(p.scale_log2, p.scale_log2), nm2 = tc::f2(-m_ref, -m_ref);
            uint64_t la[2] = {tc::f2(0.f, 0.f), tc::f2(0.f, 0.f)}, qa[2] = {la[0], la[0]};
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              const uint32_t u0 = i < 16 ? sa[2 * i] : sb[2 * i - 32], u1 = i < 16 ? sa[2 * i + 1] : sb[2 * i - 31];
              const float2 x = tc::f2_split(tc::f2_fma(tc::f2u(u0, u1), c2, nm2));
              const float p0 = tc::ex2(x.x), p1 = tc::ex2(x.y);
              pk[i] = tc::cvt_bf16x2(p0, p1);
              la[i & 1] = tc::f2_add(la[i & 1], tc::f2(p0, p1));
              qa[i & 1] = tc::f2_add(qa[i & 1], tc::f2u(pk[i] << 16, pk[i] & 0xFFFF0000u));
            }
            const float2 ls = tc::f2_split(tc::f2_add(la[0], la[1])), lr = tc::f2_split(tc::f2_add(qa[0], qa[1]));
            l += ls.x + ls.y;
            lq += lr.x + lr.y;
          }
          if (w < nh) {
            // stage this half's P (+ alpha and per-warp rescale flags); warp 2 + w ships it
            if (sends >= 1 && !tc::wait<false>(&bars[kBarStgFree + w], (sends - 1) & 1, ab)) {
              ok = false;
              break;
            }
#pragma unroll
            for (int c = 0; c < 8; ++c)
              *reinterpret_cast<uint4*>(stg + h * 128 + ((c ^ (h & 7)) * 16)) =
                  make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
            const bool any = __any_sync(0xffffffffu, alpha != 1.f);
            if (w == 0) reinterpret_cast<float*>(stg + kPMetaAlpha)[h] = alpha;
            if (lane == 0) reinterpret_cast<int*>(stg + kPMetaFlags)[warp & 3] = (w == 0 && any) ? 1 : 0;
            tc::fence_async_smem();
            tc::mbar_arrive(&bars[kBarStgFull + w]);
            ++sends;
          }
          hh += nh;
        }
        if (!ok) break;
        // ---- segment end: (m_ref, l) of the partial, then the next segment's query
        // (the next write of lsum comes a whole tile later, past a rendezvous with warpgroup 0)
        if (w == 1) {
          lsum[h] = l;
          lsum[kH + h] = lq;
        }
        tc::mbar_arrive(&bars[kBarLsum]);
        if (!tc::wait<false>(&bars[kBarLsum], k & 1, ab)) break;
        if (w == 0) {
          const int64_t slot = slot_of(s);
          p.m_part[slot * kH + h] = m_ref;
          p.l_part[slot * kH + h] = l + lsum[h];
          p.lq_part[slot * kH + h] = lq + lsum[kH + h];
        }
        if (x < hi) load_q(seq_of_tile(pre, B, x));
      }
    }
  } else {
    // ================================================================ value CTA
    if (warp == 0) {
      if (lane == 0) {
        // ---------------------------------------------------------- TMA producer (one thread)
        // one 64 KB box per 64-token half tile: its 512 latent columns, chunk-major
        tc::prefetch_map(&map_v);
        int hh = 0;
        bool ok = true;
        for (int64_t x = lo; x < hi && ok;) {
          const Seg s = seg_at(pre, lens, B, x, hi);
          x += s.ntile;
          for (int j = 0; j < s.ntile && ok; ++j) {
            const int tt = s.t_begin + j;
            const int nh = halves_of(s, tt);
            for (int w = 0; w < nh; ++w, ++hh) {
              const int st = hh % kVStages, u = hh / kVStages;
              if (u >= 1 && !tc::wait<false>(&bars[kBarEmpty + st], (u - 1) & 1, ab)) {
                ok = false;
                break;
              }
              uint8_t* dst = sm + kOffStage + st * kVStageBytes;
              uint64_t* fb = &bars[kBarFull + st];
              if (p.paged) {
                const int blk = half_block(p, s, tt, w);
                if (blk < 0) {
                  uint4* z = reinterpret_cast<uint4*>(dst);
                  for (int i = 0; i < kVStageBytes / 16; ++i) z[i] = make_uint4(0, 0, 0, 0);
                  tc::fence_async_smem();
                  tc::mbar_arrive(fb);
                  continue;
                }
                tc::mbar_expect_tx(fb, kVStageBytes);
                tc::tma_load_4d(dst, &map_v, 0, 0, 0, blk, fb);
              } else {
                tc::mbar_expect_tx(fb, kVStageBytes);
                tc::tma_load_4d(dst, &map_v, 0, tt * kTile + 64 * w, 0, s.b, fb);
              }
            }
          }
        }
        for (int k = 1; k <= kVStages && k <= hh; ++k) {  // no copy in flight at exit
          const int m = hh - k;
          tc::wait_drain<false>(&bars[kBarFull + m % kVStages], (m / kVStages) & 1, ab);
        }
      }
    } else if (warp == 1) {
      if (lane == 0) {
        // ---------------------------------------------------------- value MMA
        constexpr uint32_t idO = tc::idesc_bf16(128, 256, 0, 1);
        const uint32_t r_stgfree = tc::map_peer(&bars[kBarStgFree], 0);
        const uint32_t stg0 = smem_u32(sm + kOffStage);
        const uint32_t pb0 = smem_u32(sm + kOffP);
        int hh = 0, oc = 0, ev = 0;
        int ntail[kVStages] = {0, 0};
        bool ok = true;
        auto post = [&](int type, int a, int b2) -> bool {  // one event at a time
          evt_desc[0] = type;
          evt_desc[1] = a;
          evt_desc[2] = b2;
          tc::mbar_arrive(&bars[kBarEvt]);
          ++ev;
          return type == kEvtExit || tc::wait<false>(&bars[kBarEvtdone], (ev - 1) & 1, ab);
        };
        auto drain = [&]() -> bool {
          tc::mma_commit(&bars[kBarOcomp]);
          return tc::wait<false>(&bars[kBarOcomp], (oc++) & 1, ab);
        };
        for (int64_t x = lo; x < hi && ok;) {
          const Seg s = seg_at(pre, lens, B, x, hi);
          x += s.ntile;
          bool first_half = true;
          for (int j = 0; j < s.ntile && ok; ++j) {
            const int tt = s.t_begin + j;
            const int nh = halves_of(s, tt);
            for (int w = 0; w < nh; ++w, ++hh) {
              const int st = hh % kVStages, pb = hh % kPBufs;
              if (!tc::wait<false>(&bars[kBarFull + st], (hh / kVStages) & 1, ab)) { ok = false; break; }
              if (half_is_tail(s, tt, w)) {
                if (!tc::wait<false>(&bars[kBarFix + st], ntail[st] & 1, ab)) { ok = false; break; }
                ++ntail[st];
              }
              if (!tc::wait<false>(&bars[kBarPfull + pb], (hh / kPBufs) & 1, ab)) { ok = false; break; }
              // P landed (the copy's bytes completed the barrier just observed), so the
              // score CTA may reuse its staging; this arrive orders nothing of this thread's
              tc::mbar_arrive_cluster_addr_relaxed(r_stgfree + w * 8);
              const volatile int* fl = reinterpret_cast<const volatile int*>(sm + kOffP + pb * kPBufBytes + kPMetaFlags);
              if (fl[0] | fl[1] | fl[2] | fl[3]) {  // the reference maximum moved: rescale O first
                if (!drain() || !post(kEvtRescale, pb, 0)) { ok = false; break; }
              }
              tc::tc_fence_after();
              const uint32_t sa = stg0 + st * kVStageBytes, pa = pb0 + pb * kPBufBytes;
#pragma unroll
              for (int n2 = 0; n2 < 2; ++n2)
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                  tc::mma_ss(tb + n2 * 256, tc::smem_desc(pa + kk * 32, 16, 1024),
                             tc::smem_desc(sa + n2 * 4 * kChunkBytes + kk * 2048, kChunkBytes, 1024), idO,
                             (first_half && kk == 0) ? 0u : 1u);
              tc::mma_commit(&bars[kBarEmpty + st]);
              // P buffer pb is free once these MMAs are done: signal the score CTA's
              // kBarPfree + pb directly (same offset in the peer, cluster rank 0)
              tc::mma_commit_multicast(&bars[kBarPfree + pb], 1);
              first_half = false;
            }
          }
          if (!ok) break;
          // segment end: the partial's O goes out before the next segment overwrites it
          if (!drain() || !post(kEvtEpilogue, 0, (int)slot_of(s))) break;
        }
        post(kEvtExit, 0, 0);
        tc::mma_commit(&bars[kBarVcDrained]);
        tc::wait_drain<false>(&bars[kBarVcDrained], 0, ab);
      }
    } else if (warp == 2) {
      if (lane == 0 && p.paged) {
        // ---------------------------------------------------------- ring helper (paged cache)
        // The second 64-token half of every score slot, and the first half of
        // the last slot too: three 8 KB boxes per half into the score CTA's ring
        // (multicast to rank 0 only), signalled on its full barrier, so this SM's
        // TMA unit takes 12 of a tile's 18 copies; a slot is reloaded once the
        // score MMAs' commit has arrived on this CTA's mirror of the slot's free
        // barrier.
        bool ok = true;
        int m = 0;
        const uint32_t r_cfull = tc::map_peer(&bars[kBarCfull], 0);
        if (lo < hi)
          for (int t = 0; t < kSlots; ++t) tc::mbar_arrive_cluster_addr_relaxed(r_cfull + 8 * t);  // the query's fill
        for (int64_t x = lo; x < hi && ok;) {
          const Seg s = seg_at(pre, lens, B, x, hi);
          x += s.ntile;
          for (int j = 0; j < s.ntile && ok; ++j, ++m) {
            const int tt = s.t_begin + j;
            const int blk = halves_of(s, tt) > 1 ? half_block(p, s, tt, 1) : -1;
            const int blk0 = half_block(p, s, tt, 0);
#pragma unroll 1
            for (int t = 0; t < kSlots; ++t) {
              if (!tc::wait<false>(&bars[kBarRingFree + t], m & 1, ab)) {  // fill m (0: the query) consumed
                ok = false;
                break;
              }
              if (blk >= 0)
                for (int cc = 0; cc < 3; ++cc)
                  tc::tma_load_4d_multicast(sm + kOffRing + t * kSlotBytes + cc * kChunk128 + kChunkBytes, &map_s, 0,
                                            0, 3 * t + cc, blk, &bars[kBarCfull + t], 1);
              if (t == kSlots - 1 && blk0 >= 0)  // and the first half of the last slot
                for (int cc = 0; cc < 3; ++cc)
                  tc::tma_load_4d_multicast(sm + kOffRing + t * kSlotBytes + cc * kChunk128, &map_s, 0, 0, 3 * t + cc,
                                            blk0, &bars[kBarCfull + t], 1);
              tc::mbar_arrive_cluster_addr_relaxed(r_cfull + 8 * t);  // fill m + 1 has this helper's part
            }
          }
        }
        // the copies land in the score CTA, which drains its ring before the
        // final cluster barrier; this CTA leaves only after that barrier
      }
    } else if (warp == 3) {
      // ------------------------------------------------------------ tail zeroing
      const int t = tid - 96;
      int hh = 0;
      bool ok = true;
      for (int64_t x = lo; x < hi && ok;) {
        const Seg s = seg_at(pre, lens, B, x, hi);
        x += s.ntile;
        for (int j = 0; j < s.ntile && ok; ++j) {
          const int tt = s.t_begin + j;
          const int nh = halves_of(s, tt);
          for (int w = 0; w < nh; ++w, ++hh) {
            const int st = hh % kVStages;
            if (!tc::wait<false>(&bars[kBarFull + st], (hh / kVStages) & 1, ab)) {
              ok = false;
              break;
            }
            if (half_is_tail(s, tt, w)) {
              uint8_t* stg = sm + kOffStage + st * kVStageBytes;
              const int r0 = s.len & 63;
              const int per_chunk = (64 - r0) * 8;  // 16-byte pieces per chunk
              for (int i = t; i < 8 * per_chunk; i += 32) {
                const int c = i / per_chunk, k = i % per_chunk;
                *reinterpret_cast<uint4*>(stg + c * kChunkBytes + (r0 + (k >> 3)) * 128 + (k & 7) * 16) =
                    make_uint4(0, 0, 0, 0);
              }
              tc::fence_async_smem();
              tc::mbar_arrive(&bars[kBarFix + st]);
            }
            tc::mbar_arrive(&bars[kBarEmpty + st]);
          }
        }
      }
    } else if (warp >= 4) {
      // ------------------------------------------------------------ rescale / epilogue (thread = head)
      // warps 4-7 take accumulator columns [0, 256), warps 8-11 columns [256, 512)
      const int h = (tid - 128) & 127;
      const int c0 = warp >= 8 ? 8 : 0;  // first 32-column group of this warpgroup
      const uint32_t lane_t = tb + ((uint32_t)((warp & 3) * 32) << 16);
      for (int e = 0;; ++e) {
        if (!tc::wait<false>(&bars[kBarEvt], e & 1, ab)) break;
        tc::tc_fence_after();
        const int type = evt_desc[0], arg = evt_desc[1], slot = evt_desc[2];
        if (type == kEvtExit) break;
        if (type == kEvtRescale) {
          const float a = reinterpret_cast<const float*>(sm + kOffP + arg * kPBufBytes + kPMetaAlpha)[h];
#pragma unroll 1
          for (int c = c0; c < c0 + 8; c += 2) {
            uint32_t r0[32], r1[32];
            tc::tmem_ld32(lane_t + c * 32, r0);
            tc::tmem_ld32(lane_t + c * 32 + 32, r1);
            tc::tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              r0[i] = __float_as_uint(__uint_as_float(r0[i]) * a);
              r1[i] = __float_as_uint(__uint_as_float(r1[i]) * a);
            }
            tc::tmem_st32(lane_t + c * 32, r0);
            tc::tmem_st32(lane_t + c * 32 + 32, r1);
          }
          tc::tmem_wait_st();
        } else {
          // partial layout [slot][128 float4 columns j][128 heads][4]: for each j the
          // 32 lanes of a warp store 512 contiguous bytes
          float4* dst = reinterpret_cast<float4*>(p.o_part) + (int64_t)slot * (kDC / 4) * kH + h;
#pragma unroll 1
          for (int c = c0; c < c0 + 8; c += 2) {
            uint32_t r0[32], r1[32];
            tc::tmem_ld32(lane_t + c * 32, r0);
            tc::tmem_ld32(lane_t + c * 32 + 32, r1);
            tc::tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              dst[(c * 8 + i) * kH] = make_float4(__uint_as_float(r0[4 * i]), __uint_as_float(r0[4 * i + 1]),
                                                  __uint_as_float(r0[4 * i + 2]), __uint_as_float(r0[4 * i + 3]));
              dst[(c * 8 + 8 + i) * kH] = make_float4(__uint_as_float(r1[4 * i]), __uint_as_float(r1[4 * i + 1]),
                                                      __uint_as_float(r1[4 * i + 2]), __uint_as_float(r1[4 * i + 3]));
            }
          }
        }
        tc::tc_fence_before();
        tc::mbar_arrive(&bars[kBarEvtdone]);
      }
    }
  }

  tc::tc_fence_before();
  __syncthreads();
  __syncwarp();
  tc::cluster_sync();  // the peer may still be storing into this CTA's shared memory until here
  if (warp == 1) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tb, 512);
  }
}

// ------------------------------------------------------------------ combine
// Partials are unnormalised: O_s with reference maximum m_s (log2 units), the
// fp32 weight sum l_s and the rounded weight sum lq_s.  M = max_s m_s,
// L = sum_s l_s 2^(m_s - M), Lq = sum_s lq_s 2^(m_s - M),
// z = sum_s 2^(m_s - M) O_s / Lq, lse = (M + log2 L) ln 2.
// Block (column group of 16, sequence b), thread = head: the partial reads are
// 512 contiguous bytes per warp.
template <bool ZF32>
__global__ void __launch_bounds__(128) combine_tc_kernel(const DecodeLaunch a) {
  const int jg = blockIdx.x, b = blockIdx.y, h = threadIdx.x;
  // launched as a programmatic dependent of the partial pass: wait for it (and
  // its memory) before reading anything it wrote
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const float* m_part = a.lse_part;
  const float* l_part = a.l_part;
  const float* lq_part = a.lq_part;
  // the partial pass's plan: kind, tiles, workers, and this sequence's partials
  const bool aligned = a.plan_flag[0] != 0;
  const int T = a.plan_flag[1], G = a.plan_flag[2];
  const int64_t g0 = a.seqplan[2 * b], g1 = a.seqplan[2 * b + 1];
  // this block: latent columns [16 jg, 16 jg + 16) of every head of sequence b
  float* zf = static_cast<float*>(a.z_out) + ((int64_t)b * kH + h) * kDC + jg * 16;
  __nv_bfloat16* zb = static_cast<__nv_bfloat16*>(a.z_out) + ((int64_t)b * kH + h) * kDC + jg * 16;
  // a partial pass that gave up on a bounded wait left partials unwritten: the
  // outputs are NaN then, not stale numbers
  const bool failed = a.status != nullptr && *reinterpret_cast<volatile int32_t*>(a.status) == MLA_ERR_DEVICE_TIMEOUT;
  if (g1 < g0 || failed) {
    const float zv = failed ? __int_as_float(0x7fc00000) : 0.f;
    for (int d = 0; d < 16; ++d) {
      if (ZF32) zf[d] = zv; else zb[d] = __float2bfloat16_rn(zv);
    }
    if (jg == 0 && a.lse_out) a.lse_out[(int64_t)b * kH + h] = failed ? zv : -INFINITY;
    return;
  }
  // partials four at a time, all their loads in flight together; the running
  // maximum M moves as chunks arrive (acc and L rescaled by 2^(M_old - M_new))
  float M = -INFINITY, L = 0.f, Lq = 0.f;
  float4 acc[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) acc[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int64_t g = g0; g <= g1; g += 4) {
    float mv[4], lv[4], lqv[4];
    float4 v[4][4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int64_t gg = g + u;
      const int64_t slot = aligned ? gg : gg + b;
      const bool ok = gg <= g1 && (aligned || worker_begin((int)gg + 1, T, G) > worker_begin((int)gg, T, G));
      mv[u] = -INFINITY;
      lv[u] = 0.f;
      lqv[u] = 0.f;
#pragma unroll
      for (int i = 0; i < 4; ++i) v[u][i] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (ok) {
        mv[u] = m_part[slot * kH + h];
        lv[u] = l_part[slot * kH + h];
        lqv[u] = lq_part[slot * kH + h];
        const float4* src = reinterpret_cast<const float4*>(a.o_part) + (slot * (kDC / 4) + jg * 4) * kH + h;
#pragma unroll
        for (int i = 0; i < 4; ++i) v[u][i] = src[i * kH];
      }
    }
    const float Mn = fmaxf(M, fmaxf(fmaxf(mv[0], mv[1]), fmaxf(mv[2], mv[3])));
    if (Mn == -INFINITY) continue;
    const float sc = (M == -INFINITY) ? 0.f : exp2f(M - Mn);
    L *= sc;
    Lq *= sc;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      acc[i].x *= sc;
      acc[i].y *= sc;
      acc[i].z *= sc;
      acc[i].w *= sc;
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const float w = (mv[u] == -INFINITY) ? 0.f : exp2f(mv[u] - Mn);
      L += w * lv[u];
      Lq += w * lqv[u];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        acc[i].x += w * v[u][i].x;
        acc[i].y += w * v[u][i].y;
        acc[i].z += w * v[u][i].z;
        acc[i].w += w * v[u][i].w;
      }
    }
    M = Mn;
  }
  const float inv = 1.f / Lq;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float4 v = make_float4(acc[i].x * inv, acc[i].y * inv, acc[i].z * inv, acc[i].w * inv);
    if (ZF32) {
      reinterpret_cast<float4*>(zf)[i] = v;
    } else {
      reinterpret_cast<uint2*>(zb)[i] = make_uint2(pack_bf16x2(v.x, v.y), pack_bf16x2(v.z, v.w));
    }
  }
  if (jg == 0 && a.lse_out) a.lse_out[(int64_t)b * kH + h] = (M + log2f(L)) * kLn2;
}

// ---------------------------------------------------------------- host side
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(f);
  });
  return fn;
}

}  // namespace

bool tc_supported(const DecodeLaunch& a) {
  return a.n_heads == kH && a.d_latent == kDC && a.d_rope == 64 && a.batch <= kTcMaxBatch;
}

cudaError_t launch_decode_tc(const DecodeLaunch& a, cudaStream_t s) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return cudaErrorNotSupported;
  // The cache as a 4-D tensor (64 columns, tokens, 9 column chunks, sequence or
  // block): a box spans 64 columns x rows x chunks and lands chunk-major, each
  // chunk a 128-byte-swizzled K-major tile.
  const bool paged = a.block_table != nullptr;
  const cuuint64_t row = (cuuint64_t)kD * 2;
  const cuuint64_t cdims[4] = {64, paged ? (cuuint64_t)64 : (cuuint64_t)a.seq_stride, 9,
                               paged ? (cuuint64_t)a.num_blocks : (cuuint64_t)a.batch};
  const cuuint64_t cstrides[3] = {row, 128, (paged ? (cuuint64_t)64 : (cuuint64_t)a.seq_stride) * row};
  const cuuint32_t es[4] = {1, 1, 1, 1};
  auto encode = [&](CUtensorMap* m, const void* base, cuuint32_t rank, const cuuint64_t* dims,
                    const cuuint64_t* strides, const cuuint32_t* box) {
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void*>(base), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
  };
  // score CTA: three chunks of a 128-token tile (contiguous) or one chunk of a 64-token block (paged)
  CUtensorMap map_s, map_v, q_map, q_map3;
  const cuuint32_t box_s[4] = {64, paged ? 64u : (cuuint32_t)kTile, paged ? 1u : 3u, 1};
  // value CTA: the eight latent chunks of 64 tokens
  const cuuint32_t box_v[4] = {64, 64, 8, 1};
  // the query [B][128][576]: three chunks of all heads (4-D), or one chunk (3-D)
  const cuuint64_t qdims[4] = {64, (cuuint64_t)kH, 9, (cuuint64_t)a.batch};
  const cuuint64_t qstrides[3] = {row, 128, (cuuint64_t)kH * row};
  const cuuint32_t qbox[4] = {64, 128, 3, 1};
  const cuuint64_t q3dims[3] = {(cuuint64_t)kD, (cuuint64_t)kH, (cuuint64_t)a.batch};
  const cuuint64_t q3strides[2] = {row, (cuuint64_t)kH * row};
  const cuuint32_t q3box[3] = {64, 128, 1};
  if (!encode(&map_s, a.pool, 4, cdims, cstrides, box_s) || !encode(&map_v, a.pool, 4, cdims, cstrides, box_v) ||
      !encode(&q_map, a.q, 4, qdims, qstrides, qbox) || !encode(&q_map3, a.q, 3, q3dims, q3strides, q3box))
    return cudaErrorInvalidValue;
  TcParams p;
  p.q = static_cast<const __nv_bfloat16*>(a.q);
  p.pool = static_cast<const __nv_bfloat16*>(a.pool);
  p.block_table = a.block_table;
  p.max_blocks = a.max_blocks;
  p.num_blocks = a.num_blocks;
  p.seq_stride = a.seq_stride;
  p.seqlens = a.seqlens;
  p.batch = a.batch;
  p.paged = a.block_table != nullptr;
  p.scale_log2 = a.scale * kLog2e;
  p.workers = a.workers;
  p.o_part = a.o_part;
  p.m_part = a.lse_part;
  p.l_part = a.l_part;
  p.lq_part = a.lq_part;
  p.status = a.status;
  p.plan_hdr = a.plan_flag;
  p.seqplan = a.seqplan;
  const size_t smem = tc_smem_bytes(a.batch);
  cudaError_t e = ensure_smem<decode_tc_kernel>((int)smem);
  if (e != cudaSuccess) return e;
  decode_tc_kernel<<<2 * a.workers, kThreads, smem, s>>>(map_s, map_v, q_map, q_map3, p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  // the combine as a programmatic dependent launch: its blocks are scheduled as
  // the partial pass's CTAs exit instead of after the whole grid has drained
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(kDC / 16, a.batch);
  cfg.blockDim = dim3(128);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return a.z_is_fp32 ? cudaLaunchKernelEx(&cfg, combine_tc_kernel<true>, a)
                     : cudaLaunchKernelEx(&cfg, combine_tc_kernel<false>, a);
}

}  // namespace mla

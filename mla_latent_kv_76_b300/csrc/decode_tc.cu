// Tensor-core split-KV decode for the DeepSeek-V3 head shape: n_h = 128,
// d_c = 512, d_R = 64 (576-wide cache rows), on tcgen05 / TMEM / TMA.
//
// What is computed ("结合 DeepSeek 推理代码看 MLA": score = (q^C W^UK).c^KV +
// q^R.k^R; worked example steps 4-5: scale, causal mask, softmax, z = A.kv):
// for every head i and visible token j of a sequence
//   s_j = scale * [q~_i ; q^R_i] . [c_j ; k^R_j],   z_i = sum_j softmax(s)_j c_j.
//
// Decomposition.  The fp32 accumulator O = 128 heads x 512 latent fills the
// whole tensor memory of one SM, so each 64-token tile is shared by the two
// CTAs of a cluster (one per SM), split by contraction rather than by columns:
//   score CTA (rank 0)  S = [q~; q^R] . [c; k^R]^T over all 576 columns,
//                       M = 128 heads x N = 64 tokens per tcgen05.mma, with
//                       the whole query (latent and RoPE parts) held in TMEM;
//                       online softmax; each thread writes its bf16 weights P
//                       straight into the value CTA's shared memory with
//                       st.async (the only data exchange, 16.5 KB per tile).
//   value CTA (rank 1)  O += P . C[:, 0:512] (M = 128, N = 256 x 2, K = 64),
//                       the whole accumulator in TMEM.
// Every cache byte is read from HBM once, by the score CTA; the value CTA
// re-reads the latent columns from L2, fetching tile m only once the score
// CTA has its rows (a counter in the value CTA's shared memory that the score
// MMA thread bumps): issued earlier, the two requests for one line would both
// wait on DRAM and the value stages would hold data twice as long.
//
// Copies.  Measured on B300: what bounds a TMA stream is the number of copies
// per SM (8 KB copies cap the GPU near 4.3 TB/s, 24 KB copies from half the
// SMs reach ~6.3 TB/s) and copies issued by divergent lanes of one warp run
// ~40 % slower than copies issued by separate warps.  So the cache is viewed
// through 4-D tensor maps [64 columns][rows][9 column chunks][block or
// sequence] whose chunk dimension lies outside the row dimension: one copy
// then lands several 64-column chunks of a 64-token block, each as its own
// 128-byte-swizzled [64 rows][128 B] operand tile.  The score CTA's ring has
// eight 24 KB slots (three chunks of one block each), filled by four producer
// warps; the value CTA takes a block's eight latent chunks (64 KB) per copy.
// Paged block ids are read 32 tiles at a time by each producer warp.
//
// Score CTA, 512 threads: warps 0-3 TMA (slot s belongs to warp s % 4; the
// first segment's query arrives through ring slots 0-5 ahead of the cache),
// warp 4 MMA issue (S triple-buffered in TMEM; one barrier wait and one commit
// per 12 MMAs), warps 8-11 / 12-15 softmax for token columns 0-31 / 32-63 of
// every tile (thread = head).  Value CTA: warps 0-1 TMA (two 64 KB stages, one
// per warp), warps 2-3 zero the rows past the sequence end in its last tile
// (NaN garbage must not meet a zero weight), warp 4 MMA, warps 8-15 rescale O
// and write the segment's partial (thread = head, two column halves).  The
// value MMA's commit after the MMAs that read a P buffer arrives on the score
// CTA's barrier for that buffer.
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
constexpr int kTile = 64;            // tokens per tile: one paged block
constexpr int kThreads = 512;
constexpr int kTcMaxBatch = 1024;
constexpr float kRescaleThreshold = 16.f;
constexpr int kChunkBytes = 64 * 128;  // 64 rows x 64 bf16 columns, 128-byte swizzled

// ---- P hand-off unit: one tile's bf16 weights for 128 heads, then metadata
constexpr int kPBytes = kH * 128;                  // 128 heads x 64 tokens bf16 (SW128 K-major)
constexpr int kPMetaAlpha = kPBytes;               // alpha[128] fp32
constexpr int kPMetaFlags = kPBytes + 512;         // flag[4] int32 (per warp: O must be rescaled)
constexpr int kPMsgBytes = kPBytes + 512 + 16;     // what the score CTA writes per tile
constexpr int kPBufBytes = kPBytes + 1024;
// ---- score CTA shared memory
constexpr int kSlots = 8;                          // ring slots: three column chunks of one block each
constexpr int kSlotChunks = 3;
constexpr int kSlotBytes = kSlotChunks * kChunkBytes;
constexpr int kQItems = 6;                         // query: 2 head halves x 3 chunk groups, ring slots 0-5
constexpr int kSBufs = 3;                          // S buffers in TMEM
constexpr int kOffRing = 0;
constexpr int kOffXmax = kOffRing + kSlots * kSlotBytes;    // [2 parity][2 wg][128] fp32
constexpr int kOffLsum = kOffXmax + 2 * 2 * kH * 4;         // [2][128] fp32: weight sums of warpgroup 1
// ---- value CTA shared memory
constexpr int kVStages = 2;
constexpr int kVStageBytes = 8 * kChunkBytes;      // the 512 latent columns of one block
constexpr int kPBufs = 4;
constexpr int kOffStage = 0;
constexpr int kOffP = kOffStage + kVStages * kVStageBytes;  // [4] P buffers, written by the score CTA
// ---- common tail
constexpr int kOffBar = (kOffLsum + 2 * kH * 4 > kOffP + kPBufs * kPBufBytes) ? kOffLsum + 2 * kH * 4
                                                                             : kOffP + kPBufs * kPBufBytes;
constexpr int kNumBars = 40;
constexpr int kOffMisc = kOffBar + kNumBars * 8;   // tmem base, abort flag, event descriptor, progress
constexpr int kOffPrefix = kOffMisc + 32;          // tile prefix, plan entry prefix, lengths

static_assert(kQItems <= kSlots && kSlots % 4 == 0, "ring layout");
static_assert(kSlotBytes % 1024 == 0 && kPBufBytes % 1024 == 0 && kVStageBytes % 1024 == 0,
              "swizzled operand tiles need 1024-byte alignment");

// score CTA barriers
constexpr int kBarFull = 0, kBarEmpty = 8, kBarSfull = 16, kBarSfree = 19, kBarQready = 22, kBarPfree = 23,
              kBarXmax = 27, kBarLsum = 29, kBarQread = 30, kBarScDrained = 31;
// value CTA barriers (kBarPfree's offsets, 23-26, stay unused here: the value
// MMA's multicast commit names that offset in the score CTA)
constexpr int kBarVFull = 0, kBarVEmpty = 2, kBarFix = 4, kBarPfull = 6, kBarOcomp = 10, kBarEvt = 11,
              kBarEvtdone = 12, kBarVcDrained = 13;
static_assert(kBarScDrained < kNumBars && kBarVcDrained < kBarPfree, "barrier map");

// TMEM columns of the score CTA: S buffers [0, 192) (64 tokens each), the
// query's RoPE part [192, 224) and its 512 latent columns [256, 512), both as
// packed bf16 pairs
constexpr uint32_t kColS = 0, kColQr = 192, kColQ = 256;

enum { kEvtRescale = 1, kEvtEpilogue = 2, kEvtExit = 3 };

size_t tc_smem_bytes(int batch) { return (size_t)kOffPrefix + 3 * (size_t)(batch + 1) * 4 + 1024; }

struct TcParams {
  const __nv_bfloat16* q;
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
  int32_t* plan_flag;  // 1: sequence-aligned plan, 0: even tile split (read by the combine)
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

// Does tile tt hold the sequence end inside a partly filled block?
MLA_DEVI bool tile_is_tail(const Seg& s, int tt) { return (s.len & 63) != 0 && tt == (s.len - 1) >> 6; }

// Block ids of a paged cache, fetched 32 tiles at a time by a whole warp (one
// coalesced load instead of a dependent global read before every copy).
// Entries past the sequence's own tiles are never read.
struct BlockIds {
  int b = -1, base = 0, v = -1;
  // id of tile tt of sequence s (nt tiles), or -1 if out of range; every lane
  // of the warp calls with the same arguments
  MLA_DEVI int get(const TcParams& p, int s, int nt, int tt, int lane) {
    if (s != b || tt < base || tt >= base + 32) {
      b = s;
      base = tt;
      const int t = tt + lane;
      int id = -1;
      if (t < nt) id = p.block_table[(int64_t)s * p.max_blocks + t];
      v = (id >= 0 && id < p.num_blocks) ? id : -1;
    }
    return __shfl_sync(0xffffffffu, v, tt - base);
  }
};

MLA_DEVI void zero_smem(uint8_t* dst, int bytes) {
  uint4* z = reinterpret_cast<uint4*>(dst);
  for (int i = 0; i < bytes / 16; ++i) z[i] = make_uint4(0, 0, 0, 0);
  tc::fence_async_smem();
}

// Bounded wait until a counter in this CTA's shared memory reaches `target`.
MLA_DEVI bool wait_count(const volatile uint32_t* c, uint32_t target, const tc::Abort& ab) {
  if (*c >= target) return true;
  const long long t0 = clock64();
  for (uint32_t it = 1;; ++it) {
    if (*c >= target) return true;
    if ((it & 255u) == 0) {
      if (*ab.flag) return false;
      if (clock64() - t0 > tc::kWaitCycles) {
        *ab.flag = 1;
        report(ab.status, MLA_ERR_DEVICE_TIMEOUT);
        return false;
      }
    }
  }
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    decode_tc_kernel(const __grid_constant__ CUtensorMap map_s, const __grid_constant__ CUtensorMap map_v,
                     const __grid_constant__ CUtensorMap map_q, const TcParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + kOffBar);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + kOffMisc);
  int* abort_flag = reinterpret_cast<int*>(sm + kOffMisc + 4);
  volatile int* evt_desc = reinterpret_cast<volatile int*>(sm + kOffMisc + 8);  // type, buffer, slot
  uint32_t* progress = reinterpret_cast<uint32_t*>(sm + kOffMisc + 24);  // value CTA: tiles whose S is done
  int* pre = reinterpret_cast<int*>(sm + kOffPrefix);
  int* Wp = pre + p.batch + 1;    // entries prefix of the split plan
  int* lens = Wp + p.batch + 1;   // validated sequence lengths

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t rank = tc::cluster_rank();
  const int g = (int)(blockIdx.x >> 1);
  const int64_t cap = p.paged ? (int64_t)p.max_blocks * kTile : p.seq_stride;

  if (tid == 0) {
    if (rank == 0) {
      for (int i = 0; i < kSlots; ++i) {
        tc::mbar_init(&bars[kBarFull + i], 1);   // the producer's expect_tx arrival
        tc::mbar_init(&bars[kBarEmpty + i], 1);  // MMA commit (or the query's release)
      }
      for (int i = 0; i < kSBufs; ++i) {
        tc::mbar_init(&bars[kBarSfull + i], 1);
        tc::mbar_init(&bars[kBarSfree + i], 256);
      }
      for (int i = 0; i < 2; ++i) tc::mbar_init(&bars[kBarXmax + i], 256);
      tc::mbar_init(&bars[kBarQready], 256);
      for (int i = 0; i < kPBufs; ++i) tc::mbar_init(&bars[kBarPfree + i], 1);
      tc::mbar_init(&bars[kBarScDrained], 1);
      tc::mbar_init(&bars[kBarLsum], 256);
      tc::mbar_init(&bars[kBarQread], 256);
    } else {
      for (int i = 0; i < kVStages; ++i) {
        tc::mbar_init(&bars[kBarVFull + i], 1);
        tc::mbar_init(&bars[kBarVEmpty + i], 1 + 64);
        tc::mbar_init(&bars[kBarFix + i], 64);
      }
      for (int i = 0; i < kPBufs; ++i) tc::mbar_init(&bars[kBarPfull + i], 1);  // the score CTA's expect_tx arrival
      tc::mbar_init(&bars[kBarOcomp], 1);
      tc::mbar_init(&bars[kBarEvt], 1);
      tc::mbar_init(&bars[kBarEvtdone], 256);
      tc::mbar_init(&bars[kBarVcDrained], 1);
    }
    *abort_flag = 0;
    *progress = 0;
    tc::fence_mbar_init();
  }
  if (warp == 4) tc::tmem_alloc(tmem_slot, 512);
  tile_prefix(p.seqlens, p.batch, cap, p.status, pre, kTile, lens);  // ends with __syncthreads
  const bool aligned = plan_prefix(pre, p.batch, p.workers, Wp);     // ends with __syncthreads
  if (blockIdx.x == 0 && tid == 0) *p.plan_flag = aligned ? 1 : 0;
  tc::tc_fence_before();
  tc::cluster_sync();  // both CTAs' barriers initialised before any remote arrival
  tc::tc_fence_after();
  const uint32_t tb = *tmem_slot;
  const tc::Abort ab{abort_flag, p.status};

  const int B = p.batch, G = p.workers;
  // worker g's contiguous run of tiles: entries [g E / G, (g + 1) E / G) of the
  // sequence-aligned plan, or the even split [g T / G, (g + 1) T / G)
  const int64_t E = Wp[B], T = pre[B];
  const int64_t lo = aligned ? entry_tile(pre, Wp, B, div_floor((int64_t)g * E, G)) : worker_begin(g, T, G);
  const int64_t hi = aligned ? entry_tile(pre, Wp, B, div_floor((int64_t)(g + 1) * E, G)) : worker_begin(g + 1, T, G);
  // the partial slot of a segment: the plan entry it starts with, or worker + sequence
  auto slot_of = [&](const Seg& s) -> int64_t {
    if (!aligned) return (int64_t)g + s.b;
    const int t = pre[s.b + 1] - pre[s.b], w = Wp[s.b + 1] - Wp[s.b];
    return (int64_t)Wp[s.b] + entry_of_tile(s.t_begin, t, w);
  };

  if (rank == 0) {
    // ================================================================ score CTA
    if (warp < 4) {
      // ------------------------------------------------------------ TMA producer warp: ring slots s % 4 == warp
      if (warp == 0 && lane == 0) {
        tc::prefetch_map(&map_s);
        tc::prefetch_map(&map_q);
      }
      int nfill[2] = {0, 0};  // fills issued per owned slot (slots warp and warp + 4)
      bool ok = true;
      BlockIds ids;
      if (lo < hi && lane == 0) {
        // the first segment's query: 2 head halves x 3 chunk groups into slots 0-5
        const int b0 = seq_of_tile(pre, B, lo);
        for (int i = warp; i < kQItems; i += 4) {
          uint64_t* fb = &bars[kBarFull + i];
          tc::mbar_expect_tx(fb, kSlotBytes);
          tc::tma_load_4d(sm + kOffRing + i * kSlotBytes, &map_q, 0, 64 * (i / 3), kSlotChunks * (i % 3), b0, fb);
          ++nfill[i >> 2];
        }
      }
      int i = kQItems;  // items: the query's, then three per tile; item i goes to slot i % kSlots
      for (int64_t x = lo; x < hi && ok;) {
        const Seg sg = seg_at(pre, lens, B, x, hi);
        x += sg.ntile;
        const int nt = pre[sg.b + 1] - pre[sg.b];
        for (int j = 0; j < sg.ntile && ok; ++j, i += 3) {
          const int tt = sg.t_begin + j;
          if (((i & 3) != warp) && (((i + 1) & 3) != warp) && (((i + 2) & 3) != warp)) continue;  // none mine
          const int blk = p.paged ? ids.get(p, sg.b, nt, tt, lane) : 0;
          if (lane == 0) {
            for (int cg = 0; cg < 3; ++cg) {
              const int item = i + cg, s = item % kSlots;
              if ((s & 3) != warp) continue;
              if (item >= kSlots && !tc::wait<false>(&bars[kBarEmpty + s], ((item / kSlots) - 1) & 1, ab)) {
                ok = false;
                break;
              }
              uint8_t* dst = sm + kOffRing + s * kSlotBytes;
              uint64_t* fb = &bars[kBarFull + s];
              ++nfill[s >> 2];
              if (p.paged && blk < 0) {  // unreadable block: its rows count as zeros
                report(p.status, MLA_ERR_DEVICE_BOUNDS);
                zero_smem(dst, kSlotBytes);
                tc::mbar_arrive(fb);
                continue;
              }
              tc::mbar_expect_tx(fb, kSlotBytes);
              // contiguous cache: rows past the sequence are masked by the softmax;
              // past the allocation they read as zero
              if (p.paged) tc::tma_load_4d(dst, &map_s, 0, 0, kSlotChunks * cg, blk, fb);
              else tc::tma_load_4d(dst, &map_s, 0, tt * kTile, kSlotChunks * cg, sg.b, fb);
            }
          }
          ok = __shfl_sync(0xffffffffu, ok, 0);
        }
      }
      // no copy in flight at exit: the last fill of each owned slot has landed
      if (lane == 0)
        for (int k = 0; k < 2; ++k)
          if (nfill[k] >= 1) tc::wait_drain<false>(&bars[kBarFull + warp + 4 * k], (nfill[k] - 1) & 1, ab);
    } else if (warp == 4) {
      if (lane == 0) {
        // ---------------------------------------------------------- score MMA
        constexpr uint32_t idS = tc::idesc_bf16(128, kTile, 0, 0);
        const uint32_t ring = smem_u32(sm + kOffRing);
        const uint32_t r_progress = tc::map_peer(progress, 1);
        int m = 0, k = 0, i = kQItems;
        bool ok = true;
        for (int64_t x = lo; x < hi && ok; ++k) {
          const Seg sg = seg_at(pre, lens, B, x, hi);
          x += sg.ntile;
          if (!tc::wait<false>(&bars[kBarQready], k & 1, ab)) break;
          for (int j = 0; j < sg.ntile && ok; ++j, ++m) {
            const int buf = m % kSBufs;
            // buffer buf is free once the softmax read tile m - kSBufs
            if (m >= kSBufs && !tc::wait<false>(&bars[kBarSfree + buf], ((m / kSBufs) - 1) & 1, ab)) {
              ok = false;
              break;
            }
            tc::tc_fence_after();
            const uint32_t dS = tb + kColS + buf * kTile;
            // per ring slot (three chunks): one wait, twelve MMAs, one commit
#pragma unroll
            for (int cg = 0; cg < 3; ++cg, ++i) {
              const int s = i % kSlots;
              if (!tc::wait<false>(&bars[kBarFull + s], (i / kSlots) & 1, ab)) {
                ok = false;
                break;
              }
              tc::tc_fence_after();
              const uint32_t sa = ring + s * kSlotBytes;
#pragma unroll
              for (int jj = 0; jj < 3; ++jj) {
                const int c = 3 * cg + jj;
                const uint32_t qa = c < 8 ? kColQ + 32 * c : kColQr;
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                  tc::mma_ts(dS, tb + qa + 8 * kk, tc::smem_desc(sa + jj * kChunkBytes + kk * 32, 16, 1024), idS,
                             (c | kk) != 0 ? 1u : 0u);
              }
              tc::mma_commit(&bars[kBarEmpty + s]);
            }
            if (!ok) break;
            tc::mma_commit(&bars[kBarSfull + buf]);
            // the tile's cache rows are in L2 now: the value CTA may fetch its latent columns
            tc::red_add_remote(r_progress, 1);
          }
        }
        tc::mma_commit(&bars[kBarScDrained]);
        tc::wait_drain<false>(&bars[kBarScDrained], 0, ab);
      }
    } else if (warp >= 8) {
      // ------------------------------------------------------------ softmax (thread = head)
      const int w = (warp - 8) >> 2;  // token columns [32 w, 32 w + 32) of each tile
      const int h = tid & 127;
      const uint32_t lane_t = tb + ((uint32_t)((warp & 3) * 32) << 16);
      float* xmax = reinterpret_cast<float*>(sm + kOffXmax);
      float* lsum = reinterpret_cast<float*>(sm + kOffLsum);
      const uint32_t r_p = tc::map_peer(sm + kOffP, 1);
      const uint32_t r_pfull = tc::map_peer(&bars[kBarPfull], 1);

      // a later segment's query, from global memory: warpgroup 0 takes latent
      // columns [0, 256), warpgroup 1 columns [256, 512) and the RoPE part
      auto load_q = [&](int b) {
        const uint4* row = reinterpret_cast<const uint4*>(p.q + ((int64_t)b * kH + h) * kD);
#pragma unroll 1
        for (int c2 = 0; c2 < 2; ++c2) {  // 16 loads in flight per thread per round
          uint32_t r[2][32];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const uint4 v = __ldg(row + 32 * w + 16 * c2 + i);
            r[i >> 3][4 * (i & 7)] = v.x;
            r[i >> 3][4 * (i & 7) + 1] = v.y;
            r[i >> 3][4 * (i & 7) + 2] = v.z;
            r[i >> 3][4 * (i & 7) + 3] = v.w;
          }
          tc::tmem_st32(lane_t + kColQ + 128 * w + 64 * c2, r[0]);
          tc::tmem_st32(lane_t + kColQ + 128 * w + 64 * c2 + 32, r[1]);
        }
        if (w == 1) {
          uint32_t r[32];
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const uint4 v = __ldg(row + 64 + i);
            r[4 * i] = v.x;
            r[4 * i + 1] = v.y;
            r[4 * i + 2] = v.z;
            r[4 * i + 3] = v.w;
          }
          tc::tmem_st32(lane_t + kColQr, r);
        }
        tc::tmem_wait_st();
        tc::tc_fence_before();
        tc::mbar_arrive(&bars[kBarQready]);
      };

      // the first segment's query, TMA-loaded into ring slots 0-5 (slot 3 hg + cg
      // holds chunks 3 cg .. 3 cg + 2 of heads [64 hg, 64 hg + 64)): warpgroup w
      // moves latent chunks 4 w .. 4 w + 3 (and warpgroup 1 the RoPE chunk) of row h
      // to TMEM, then the slots go back to the producers
      auto q_from_ring = [&]() -> bool {
        for (int s = 0; s < kQItems; ++s)
          if (!tc::wait<false>(&bars[kBarFull + s], 0, ab)) return false;
        const int hg = h >> 6, r = h & 63;
#pragma unroll 1
        for (int cc = 0; cc < 5; ++cc) {
          if (cc == 4 && w == 0) break;
          const int c = cc < 4 ? 4 * w + cc : 8;
          const uint8_t* row =
              sm + kOffRing + (3 * hg + c / 3) * kSlotBytes + (c % 3) * kChunkBytes + r * 128;
          uint32_t v32[32];
#pragma unroll
          for (int jj = 0; jj < 8; ++jj) {
            const uint4 v = *reinterpret_cast<const uint4*>(row + ((jj ^ (r & 7)) * 16));
            v32[4 * jj] = v.x;
            v32[4 * jj + 1] = v.y;
            v32[4 * jj + 2] = v.z;
            v32[4 * jj + 3] = v.w;
          }
          tc::tmem_st32(lane_t + (c < 8 ? kColQ + 32 * c : kColQr), v32);
        }
        tc::tmem_wait_st();
        tc::tc_fence_before();
        // once every softmax thread has read its rows, slots 0-5 go back to the producers
        tc::mbar_arrive(&bars[kBarQread]);
        if (tid == 256 && tc::wait<false>(&bars[kBarQread], 0, ab))
          for (int s = 0; s < kQItems; ++s) tc::mbar_arrive(&bars[kBarEmpty + s]);
        tc::mbar_arrive(&bars[kBarQready]);
        return true;
      };

      int m = 0, k = 0;
      bool ok = true, first = true;
      for (int64_t x = lo; x < hi && ok; ++k) {
        const Seg sg = seg_at(pre, lens, B, x, hi);
        x += sg.ntile;
        if (first && !q_from_ring()) break;
        first = false;
        float m_ref = -INFINITY, l = 0.f, lq = 0.f;
        for (int j = 0; j < sg.ntile; ++j, ++m) {
          const int tt = sg.t_begin + j;
          const int buf = m % kSBufs;
          if (!tc::wait<false>(&bars[kBarSfull + buf], (m / kSBufs) & 1, ab)) {
            ok = false;
            break;
          }
          tc::tc_fence_after();
          uint32_t sv[32];
          tc::tmem_ld32(lane_t + kColS + buf * kTile + 32 * w, sv);
          tc::tmem_wait_ld();
          tc::tc_fence_before();
          tc::mbar_arrive(&bars[kBarSfree + buf]);
          const int nvalid = sg.len - tt * kTile - 32 * w;  // may be <= 0
          float xv[32];
#pragma unroll
          for (int c = 0; c < 32; ++c) xv[c] = (c < nvalid) ? __uint_as_float(sv[c]) * p.scale_log2 : -INFINITY;
          float mx[8];  // tree maximum (independent chains)
#pragma unroll
          for (int i = 0; i < 8; ++i) mx[i] = fmaxf(fmaxf(xv[i], xv[i + 8]), fmaxf(xv[i + 16], xv[i + 24]));
          float mt = fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])), fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7])));
          // tile maximum over both warpgroups (bounded rendezvous)
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
          // P = 2^(x - m_ref): bf16 for the value MMA; l sums the fp32 weights,
          // lq the rounded ones
          uint32_t pk[16];
          float ls[2] = {0.f, 0.f}, lr[2] = {0.f, 0.f};
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float p0 = tc::ex2(xv[2 * i] - m_ref), p1 = tc::ex2(xv[2 * i + 1] - m_ref);
            pk[i] = pack_bf16x2(p0, p1);
            ls[i & 1] += p0 + p1;
            lr[i & 1] += __uint_as_float(pk[i] << 16) + __uint_as_float(pk[i] & 0xFFFF0000u);
          }
          l += ls[0] + ls[1];
          lq += lr[0] + lr[1];
          // this warpgroup's 32 columns of P (+ alpha and per-warp rescale flags) go
          // straight into the value CTA's P buffer pb, free once the value MMA has
          // consumed tile m - 4
          const int pb = m % kPBufs;
          if (m >= kPBufs && !tc::wait<true>(&bars[kBarPfree + pb], ((m / kPBufs) - 1) & 1, ab)) {
            ok = false;
            break;
          }
          const uint32_t dst = r_p + pb * kPBufBytes, dbar = r_pfull + pb * 8;
          if (tid == 256) tc::mbar_expect_tx_remote(dbar, kPMsgBytes);
#pragma unroll
          for (int c = 0; c < 4; ++c)
            tc::st_async_v4(dst + h * 128 + (((4 * w + c) ^ (h & 7)) * 16),
                            make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]), dbar);
          const bool any = __any_sync(0xffffffffu, alpha != 1.f);
          if (w == 0) tc::st_async_b32(dst + kPMetaAlpha + 4 * h, __float_as_uint(alpha), dbar);
          if (w == 0 && lane == 0) tc::st_async_b32(dst + kPMetaFlags + 4 * (warp & 3), any ? 1u : 0u, dbar);
        }
        if (!ok) break;
        // ---- segment end: (m_ref, l, lq) of the partial, then the next segment's query
        // (the next write of lsum comes a whole tile later, past a rendezvous with warpgroup 0)
        if (w == 1) {
          lsum[h] = l;
          lsum[kH + h] = lq;
        }
        tc::mbar_arrive(&bars[kBarLsum]);
        if (!tc::wait<false>(&bars[kBarLsum], k & 1, ab)) break;
        if (w == 0) {
          const int64_t slot = slot_of(sg);
          p.m_part[slot * kH + h] = m_ref;
          p.l_part[slot * kH + h] = l + lsum[h];
          p.lq_part[slot * kH + h] = lq + lsum[kH + h];
        }
        if (x < hi) load_q(seq_of_tile(pre, B, x));
      }
      // The value CTA's MMA commits arrive on kBarPfree asynchronously: before this
      // CTA may exit, the last arrival on every P buffer must have landed.
      if (ok && tid == 256)
        for (int pb = 0; pb < kPBufs && pb < m; ++pb) {
          const int last = pb + ((m - 1 - pb) / kPBufs) * kPBufs;  // the last tile that used buffer pb
          tc::wait<true>(&bars[kBarPfree + pb], (last / kPBufs) & 1, ab);
        }
    }
  } else {
    // ================================================================ value CTA
    if (warp < 2) {
      // ------------------------------------------------------------ TMA producer warp: stage `warp`
      const int st = warp;
      if (st == 0 && lane == 0) tc::prefetch_map(&map_v);
      uint64_t* fb = &bars[kBarVFull + st];
      uint8_t* dst = sm + kOffStage + st * kVStageBytes;
      const volatile uint32_t* prog = progress;
      int m = 0, nf = 0;
      bool ok = true;
      BlockIds ids;
      for (int64_t x = lo; x < hi && ok;) {
        const Seg sg = seg_at(pre, lens, B, x, hi);
        x += sg.ntile;
        const int nt = pre[sg.b + 1] - pre[sg.b];
        for (int j = 0; j < sg.ntile && ok; ++j, ++m) {
          if ((m & 1) != st) continue;
          const int tt = sg.t_begin + j;
          const int blk = p.paged ? ids.get(p, sg.b, nt, tt, lane) : 0;
          if (lane == 0) {
            // the stage is free, and the score CTA has this tile's rows (so they are L2 hits)
            ok = (nf == 0 || tc::wait<false>(&bars[kBarVEmpty + st], (nf - 1) & 1, ab)) &&
                 wait_count(prog, (uint32_t)m + 1, ab);
            if (ok) {
              ++nf;
              if (p.paged && blk < 0) {
                zero_smem(dst, kVStageBytes);
                tc::mbar_arrive(fb);
              } else {
                tc::mbar_expect_tx(fb, kVStageBytes);
                if (p.paged) tc::tma_load_4d(dst, &map_v, 0, 0, 0, blk, fb);
                else tc::tma_load_4d(dst, &map_v, 0, tt * kTile, 0, sg.b, fb);
              }
            }
          }
          ok = __shfl_sync(0xffffffffu, ok, 0);
        }
      }
      if (lane == 0 && nf >= 1) tc::wait_drain<false>(fb, (nf - 1) & 1, ab);  // no copy in flight at exit
    } else if (warp < 4) {
      // ------------------------------------------------------------ tail zeroing
      const int t = tid - 64;
      int m = 0;
      bool ok = true;
      for (int64_t x = lo; x < hi && ok;) {
        const Seg sg = seg_at(pre, lens, B, x, hi);
        x += sg.ntile;
        for (int j = 0; j < sg.ntile; ++j, ++m) {
          const int st = m & 1;
          if (!tc::wait<false>(&bars[kBarVFull + st], (m >> 1) & 1, ab)) {
            ok = false;
            break;
          }
          if (tile_is_tail(sg, sg.t_begin + j)) {
            uint8_t* stg = sm + kOffStage + st * kVStageBytes;
            const int r0 = sg.len & 63;
            const int per_chunk = (64 - r0) * 8;  // 16-byte pieces per chunk
            for (int i = t; i < 8 * per_chunk; i += 64) {
              const int c = i / per_chunk, kq = i % per_chunk;
              *reinterpret_cast<uint4*>(stg + c * kChunkBytes + (r0 + (kq >> 3)) * 128 + (kq & 7) * 16) =
                  make_uint4(0, 0, 0, 0);
            }
            tc::fence_async_smem();
            tc::mbar_arrive(&bars[kBarFix + st]);
          }
          tc::mbar_arrive(&bars[kBarVEmpty + st]);
        }
      }
    } else if (warp == 4) {
      if (lane == 0) {
        // ---------------------------------------------------------- value MMA
        constexpr uint32_t idO = tc::idesc_bf16(128, 256, 0, 1);
        const uint32_t stg0 = smem_u32(sm + kOffStage);
        const uint32_t pb0 = smem_u32(sm + kOffP);
        int m = 0, oc = 0, ev = 0;
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
          const Seg sg = seg_at(pre, lens, B, x, hi);
          x += sg.ntile;
          for (int j = 0; j < sg.ntile; ++j, ++m) {
            const int tt = sg.t_begin + j;
            const int st = m & 1, pb = m % kPBufs;
            if (!tc::wait<false>(&bars[kBarVFull + st], (m >> 1) & 1, ab)) { ok = false; break; }
            if (tile_is_tail(sg, tt)) {
              if (!tc::wait<false>(&bars[kBarFix + st], ntail[st] & 1, ab)) { ok = false; break; }
              ++ntail[st];
            }
            // P arrives by the score CTA's st.async stores; once they are observed, order
            // them before the tensor core's reads of the buffer
            if (!tc::wait<true>(&bars[kBarPfull + pb], (m / kPBufs) & 1, ab)) { ok = false; break; }
            tc::fence_async_smem();
            const volatile int* fl = reinterpret_cast<const volatile int*>(sm + kOffP + pb * kPBufBytes + kPMetaFlags);
            if (j > 0 && (fl[0] | fl[1] | fl[2] | fl[3])) {  // the reference maximum moved: rescale O first
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
                           (j == 0 && kk == 0) ? 0u : 1u);
            tc::mma_commit(&bars[kBarVEmpty + st]);
            // P buffer pb is free once these MMAs are done: signal the score CTA's
            // kBarPfree + pb directly (same offset in the peer, cluster rank 0)
            tc::mma_commit_multicast(&bars[kBarPfree + pb], 1);
          }
          if (!ok) break;
          // segment end: the partial's O goes out before the next segment overwrites it
          if (!drain() || !post(kEvtEpilogue, 0, (int)slot_of(sg))) break;
        }
        post(kEvtExit, 0, 0);
        tc::mma_commit(&bars[kBarVcDrained]);
        tc::wait_drain<false>(&bars[kBarVcDrained], 0, ab);
      }
    } else if (warp >= 8) {
      // ------------------------------------------------------------ rescale / epilogue (thread = head)
      // warps 8-11 take accumulator columns [0, 256), warps 12-15 columns [256, 512)
      const int h = tid & 127;
      const int c0 = warp >= 12 ? 8 : 0;  // first 32-column group of this warpgroup
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
  if (warp == 4) {
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
  const int jg = blockIdx.x, b = blockIdx.y, h = threadIdx.x, warp = h >> 5, lane = h & 31;
  const int G = a.workers;
  const float* m_part = a.lse_part;
  const float* l_part = a.l_part;
  const float* lq_part = a.lq_part;
  const int64_t cap = a.block_table ? (int64_t)a.max_blocks * 64 : a.seq_stride;
  // the split plan of the partial kernel: total tiles T, non-empty sequences n,
  // then the entries of the sequences before b (W_b) and of b itself
  __shared__ long long red[2][4];
  __shared__ long long s_tot[2];
  long long total = 0, nonempty = 0;
  for (int i = h; i < a.batch; i += blockDim.x) {
    const int t = tiles_of(effective_len(a.seqlens, i, cap, nullptr), kTile);
    total += t;
    nonempty += t > 0;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    total += __shfl_xor_sync(0xffffffffu, total, o);
    nonempty += __shfl_xor_sync(0xffffffffu, nonempty, o);
  }
  if (lane == 0) {
    red[0][warp] = total;
    red[1][warp] = nonempty;
  }
  __syncthreads();
  if (h == 0) {
    s_tot[0] = red[0][0] + red[0][1] + red[0][2] + red[0][3];
    s_tot[1] = red[1][0] + red[1][1] + red[1][2] + red[1][3];
  }
  __syncthreads();
  const int64_t T = s_tot[0];
  const int n_ne = (int)s_tot[1];
  long long before = 0, tiles_before = 0;
  for (int i = h; i < b; i += blockDim.x) {
    const int t = tiles_of(effective_len(a.seqlens, i, cap, nullptr), kTile);
    before += plan_entries(t, T, n_ne, G);
    tiles_before += t;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    before += __shfl_xor_sync(0xffffffffu, before, o);
    tiles_before += __shfl_xor_sync(0xffffffffu, tiles_before, o);
  }
  __syncthreads();  // red[] is reused
  if (lane == 0) {
    red[0][warp] = before;
    red[1][warp] = tiles_before;
  }
  __syncthreads();
  const int64_t Wb = red[0][0] + red[0][1] + red[0][2] + red[0][3];
  const int64_t Sb = red[1][0] + red[1][1] + red[1][2] + red[1][3];
  const bool aligned = *a.plan_flag != 0;
  const int nb = tiles_of(effective_len(a.seqlens, b, cap, nullptr), kTile);
  // this block: latent columns [16 jg, 16 jg + 16) of every head of sequence b
  float* zf = static_cast<float*>(a.z_out) + ((int64_t)b * kH + h) * kDC + jg * 16;
  __nv_bfloat16* zb = static_cast<__nv_bfloat16*>(a.z_out) + ((int64_t)b * kH + h) * kDC + jg * 16;
  if (nb == 0) {
    for (int d = 0; d < 16; ++d) {
      if (ZF32) zf[d] = 0.f; else zb[d] = __float2bfloat16_rn(0.f);
    }
    if (jg == 0 && a.lse_out) a.lse_out[(int64_t)b * kH + h] = -INFINITY;
    return;
  }
  // sequence b's partials: slots [Wb, Wb + wb) (aligned plan, every one written),
  // or slot g + b of each worker g whose tiles touch b (even split; a worker with
  // no tiles wrote nothing)
  const int64_t g0 = aligned ? Wb : worker_of(Sb, T, G);
  const int64_t g1 = aligned ? Wb + plan_entries(nb, T, n_ne, G) - 1 : worker_of(Sb + nb - 1, T, G);
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
  // 4-D views [64 columns][rows][9 column chunks][block | sequence]: the chunk
  // dimension (stride 128 B) lies outside the row dimension (stride 1152 B), so
  // a box of k chunks lands as k consecutive [64 rows][128 B] swizzled tiles
  auto make = [&](CUtensorMap* m, const void* base, cuuint64_t rows, cuuint64_t outer, cuuint64_t outer_stride,
                  cuuint32_t box_chunks) -> bool {
    const cuuint64_t dims[4] = {64, rows, 9, outer};
    const cuuint64_t strides[3] = {(cuuint64_t)kD * 2, 128, outer_stride};
    const cuuint32_t box[4] = {64, 64, box_chunks, 1}, es[4] = {1, 1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
  };
  const bool paged = a.block_table != nullptr;
  const cuuint64_t rows = paged ? (cuuint64_t)kTile : (cuuint64_t)a.seq_stride;
  const cuuint64_t outer = paged ? (cuuint64_t)a.num_blocks : (cuuint64_t)a.batch;
  CUtensorMap map_s, map_v, map_q;
  if (!make(&map_s, a.pool, rows, outer, rows * kD * 2, kSlotChunks) ||
      !make(&map_v, a.pool, rows, outer, rows * kD * 2, 8) ||
      !make(&map_q, a.q, kH, (cuuint64_t)a.batch, (cuuint64_t)kH * kD * 2, kSlotChunks))
    return cudaErrorInvalidValue;
  TcParams p;
  p.q = static_cast<const __nv_bfloat16*>(a.q);
  p.block_table = a.block_table;
  p.max_blocks = a.max_blocks;
  p.num_blocks = a.num_blocks;
  p.seq_stride = a.seq_stride;
  p.seqlens = a.seqlens;
  p.batch = a.batch;
  p.paged = paged ? 1 : 0;
  p.scale_log2 = a.scale * kLog2e;
  p.workers = a.workers;
  p.o_part = a.o_part;
  p.m_part = a.lse_part;
  p.l_part = a.l_part;
  p.lq_part = a.lq_part;
  p.status = a.status;
  p.plan_flag = a.plan_flag;
  const size_t smem = tc_smem_bytes(a.batch);
  cudaError_t e = ensure_smem<decode_tc_kernel>((int)smem);
  if (e != cudaSuccess) return e;
  decode_tc_kernel<<<2 * a.workers, kThreads, smem, s>>>(map_s, map_v, map_q, p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  dim3 grid(kDC / 16, a.batch);
  if (a.z_is_fp32) combine_tc_kernel<true><<<grid, 128, 0, s>>>(a);
  else combine_tc_kernel<false><<<grid, 128, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace mla

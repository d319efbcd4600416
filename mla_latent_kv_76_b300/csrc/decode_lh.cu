// Tensor-core split-KV decode for few heads: n_h = 16, d_c = 512, d_R = 64
// (576-wide cache rows), on tcgen05 / TMEM / TMA, one CTA per SM.
//
// What is computed ("结合 DeepSeek 推理代码看 MLA": score = (q^C W^UK).c^KV +
// q^R.k^R; worked example steps 4-5: scale, mask, softmax, z = A.kv): for every
// head i and visible token j of a sequence
//   s_j = scale * [q~_i ; q^R_i] . [c_j ; k^R_j],   z_i = sum_j softmax(s)_j c_j.
//
// With 16 heads a token carries 2 x 16 x 1088 FLOP for 1152 bytes, so the
// cache stream bounds the kernel and every SM streams its own 64-token blocks:
// one 72 KB 4-D TMA box per block (64 tokens x 9 column chunks, chunk-major,
// 128-byte swizzle) into a ring of `slots` buffers.  Per block:
//   score   S[128 x 64] = Q[128 x 576] . C_blk^T   (tcgen05, M = 128 with the
//           16 heads in rows 0-15 and zero rows below, Q held in TMEM, N = 64)
//   softmax on rows 0-15 (one warp), P[16 x 64] bf16 to shared memory
//   value   O^T[512 x 16] += C_blk^T[512 x 64] . P^T[64 x 16]   (four M = 128
//           products over the latent rows, N = 16 heads, K = the 64 tokens;
//           the block's latent chunks read in place as an MN-major operand)
// so the cache bytes are read from HBM once, by the SM that needs them, and
// the accumulators take 64 + 128 TMEM columns beside the query's 288.
//
// Split-KV: the tiles of all sequences in batch order are divided evenly over
// the CTAs ([g T / G, (g + 1) T / G)), each (CTA, sequence) segment writing a
// partial (o / lq, lse) in the layout of the shape-generic path, which the
// shared combine kernel merges.
//
// Online softmax as in the 128-head kernel: a lazily moved reference maximum
// (rescaling O only when a block's maximum exceeds it by more than 16 in log2
// units), bf16 weights for the MMA, l summing the fp32 weights (for lse) and
// lq the rounded ones (normalising z).
#include <cuda.h>
#include <mutex>

#include "common.cuh"
#include "kernels.h"
#include "plan.cuh"
#include "tc.cuh"

namespace mla {
namespace {

constexpr int kH = 16, kDC = 512, kD = 576;
constexpr int kBlk = 64;                    // tokens per block (tile of the plan)
constexpr int kThreads = 384;
constexpr float kRescaleThreshold = 16.f;
constexpr int kChunkBytes = kBlk * 128;     // 64 tokens x 64 bf16 columns
constexpr int kBlkBytes = 9 * kChunkBytes;  // one block, all 576 columns (72 KB)
constexpr int kMaxSlots = 3;
// P hand-off from the softmax warp to the MMA thread: 16 heads x 64 tokens
// bf16 (128-byte-swizzled K-major rows), then alpha[16] and a rescale flag
constexpr int kPBytes = kH * 128;
constexpr int kPMetaAlpha = kPBytes;
constexpr int kPMetaFlag = kPBytes + 64;
constexpr int kPBufBytes = 3072;            // keeps every P buffer 1024-aligned
constexpr int kStatBufs = 4;                // per-segment (m, l, lq) of the 16 heads

// TMEM columns: S double buffer [0, 128), O^T [128, 192) (four 16-column
// blocks, one per 128 latent rows), the query [192, 480) as packed bf16
constexpr uint32_t kColS = 0, kColO = 128, kColQ = 192;

// barriers
constexpr int kBarFull = 0, kBarEmpty = 3, kBarFix = 6, kBarSfull = 9, kBarSfree = 11, kBarPfull = 13,
              kBarPfree = 15, kBarQready = 17, kBarQzero = 24, kBarOcomp = 19, kBarEvt = 20, kBarEvtDone = 21,
              kBarDrained = 22, kBarDrainedV = 23;
constexpr int kBarHand = 25;  // [2]: segment hand-over between the two softmax warps
constexpr int kNumBars = 27;

enum { kEvtRescale = 1, kEvtEpilogue = 2, kEvtExit = 3 };

struct LhLayout {
  int slots, off_p, off_stat, off_bar, off_misc, off_pre, total;
};

// Shared memory for `slots` ring buffers and a batch of B sequences.
MLA_HD LhLayout lh_layout(int slots, int B) {
  LhLayout L;
  L.slots = slots;
  L.off_p = slots * kBlkBytes;
  L.off_stat = L.off_p + 2 * kPBufBytes;                 // [kStatBufs][3][16] fp32
  L.off_bar = L.off_stat + kStatBufs * 3 * kH * 4;
  L.off_misc = L.off_bar + kNumBars * 8;                 // tmem base, abort flag, event descriptor
  L.off_pre = L.off_misc + 64;                           // tile prefix pre[0..B]
  L.total = L.off_pre + (B + 1) * 4 + 1024;              // + alignment slack of the base
  return L;
}

int lh_slots(int B) { return lh_layout(kMaxSlots, B).total <= 227 * 1024 ? kMaxSlots : 2; }

struct LhParams {
  const __nv_bfloat16* q;
  const int32_t* block_table;
  int32_t max_blocks, num_blocks;
  int64_t seq_stride;
  const int32_t* seqlens;
  int32_t batch, paged, workers, slots;
  float scale_log2;
  float* o_part;    // [(G + B)][16][512]  o / lq
  float* lse_part;  // [(G + B)][16]       natural log
  int32_t* status;
  int32_t* plan_hdr;  // [plan kind 0 (even split), tiles T, workers G] for the combine
  int32_t* seqplan;   // [B][2] for the combine: first and last worker whose tiles meet sequence b
};

struct Seg {
  int b, t_begin, ntile, len;
};

MLA_DEVI Seg seg_at(const int* pre, int B, int64_t x, int64_t hi, const LhParams& p, int64_t cap) {
  Seg s;
  s.b = seq_of_tile(pre, B, x);
  s.t_begin = (int)(x - pre[s.b]);
  const int64_t e = pre[s.b + 1] < hi ? pre[s.b + 1] : hi;
  s.ntile = (int)(e - x);
  s.len = effective_len(p.seqlens, s.b, cap, nullptr);
  return s;
}

// Paged block id of tile tt of segment s, or -1 if it is out of range.
MLA_DEVI int tile_block(const LhParams& p, const Seg& s, int tt) {
  if (tt >= p.max_blocks) return -1;
  const int blk = p.block_table[(int64_t)s.b * p.max_blocks + tt];
  return (blk >= 0 && blk < p.num_blocks) ? blk : -1;
}

// Valid rows of tile tt (1 .. 64).
MLA_DEVI int tile_rows(const Seg& s, int tt) { return min(kBlk, s.len - tt * kBlk); }

__global__ void __launch_bounds__(kThreads, 1)
    decode_lh_kernel(const __grid_constant__ CUtensorMap map_c, const LhParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const LhLayout L = lh_layout(p.slots, p.batch);
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + L.off_bar);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + L.off_misc);
  int* abort_flag = reinterpret_cast<int*>(sm + L.off_misc + 4);
  volatile int* evt_desc = reinterpret_cast<volatile int*>(sm + L.off_misc + 8);  // type, buffer, slot
  float* stats = reinterpret_cast<float*>(sm + L.off_stat);
  int* pre = reinterpret_cast<int*>(sm + L.off_pre);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = (int)blockIdx.x, B = p.batch, G = p.workers, S = p.slots;
  const int64_t cap = p.paged ? (int64_t)p.max_blocks * kBlk : p.seq_stride;

  if (tid == 0) {
    for (int i = 0; i < S; ++i) {
      tc::mbar_init(&bars[kBarFull + i], 1);
      tc::mbar_init(&bars[kBarEmpty + i], 1 + 64);  // value MMAs' commit + the tail warps
      tc::mbar_init(&bars[kBarFix + i], 64);
    }
    for (int i = 0; i < 2; ++i) {
      tc::mbar_init(&bars[kBarSfull + i], 1);
      tc::mbar_init(&bars[kBarSfree + i], 1);
      tc::mbar_init(&bars[kBarPfull + i], 1);
      tc::mbar_init(&bars[kBarPfree + i], 1);
    }
    tc::mbar_init(&bars[kBarQready], 1);      // even segments' queries
    tc::mbar_init(&bars[kBarQready + 1], 1);  // odd segments' queries
    tc::mbar_init(&bars[kBarQzero], 64);
    tc::mbar_init(&bars[kBarHand], 1);
    tc::mbar_init(&bars[kBarHand + 1], 1);
    tc::mbar_init(&bars[kBarOcomp], 1);
    tc::mbar_init(&bars[kBarEvt], 1);
    tc::mbar_init(&bars[kBarEvtDone], 128);
    tc::mbar_init(&bars[kBarDrained], 1);
    tc::mbar_init(&bars[kBarDrainedV], 1);
    *abort_flag = 0;
    tc::fence_mbar_init();
  }
  if (warp == 1) tc::tmem_alloc(tmem_slot, 512);
  tile_prefix(p.seqlens, B, cap, p.status, pre, kBlk);  // ends with __syncthreads
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tb = *tmem_slot;
  const tc::Abort ab{abort_flag, p.status};
  const int64_t T = pre[B];
  const int64_t lo = worker_begin(g, T, G), hi = worker_begin(g + 1, T, G);
  if (g == 0) {  // the plan for the combine: the workers whose tiles meet each sequence
    for (int b = tid; b < B; b += kThreads) {
      const int t = pre[b + 1] - pre[b];
      p.seqplan[2 * b] = t > 0 ? worker_of(pre[b], T, G) : 0;
      p.seqplan[2 * b + 1] = t > 0 ? worker_of(pre[b + 1] - 1, T, G) : -1;
    }
    if (tid == 0) {
      p.plan_hdr[0] = 0;
      p.plan_hdr[1] = (int)T;
      p.plan_hdr[2] = G;
    }
  }
  // the combine may be scheduled now; it waits for this grid to finish before reading
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const uint32_t ring = smem_u32(sm);
  const uint32_t pbuf = smem_u32(sm + L.off_p);

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------ TMA producer: one 72 KB box per block
      tc::prefetch_map(&map_c);
      int m = 0;
      bool ok = true;
      for (int64_t x = lo; x < hi && ok;) {
        const Seg s = seg_at(pre, B, x, hi, p, cap);
        x += s.ntile;
        for (int j = 0; j < s.ntile; ++j, ++m) {
          const int tt = s.t_begin + j, st = m % S, u = m / S;
          if (u >= 1 && !tc::wait<false>(&bars[kBarEmpty + st], (u - 1) & 1, ab)) {
            ok = false;
            break;
          }
          uint8_t* dst = sm + st * kBlkBytes;
          uint64_t* fb = &bars[kBarFull + st];
          if (p.paged) {
            const int blk = tile_block(p, s, tt);
            if (blk < 0) {  // unreadable block: its rows count as zeros
              report(p.status, MLA_ERR_DEVICE_BOUNDS);
              uint4* z = reinterpret_cast<uint4*>(dst);
              for (int i = 0; i < kBlkBytes / 16; ++i) z[i] = make_uint4(0, 0, 0, 0);
              tc::fence_async_smem();
              tc::mbar_arrive(fb);
              continue;
            }
            tc::mbar_expect_tx(fb, kBlkBytes);
            tc::tma_load_4d(dst, &map_c, 0, 0, 0, blk, fb);
          } else {
            // rows past the allocation read as zero, rows past the sequence are
            // zeroed by the tail warps before the MMAs read them
            tc::mbar_expect_tx(fb, kBlkBytes);
            tc::tma_load_4d(dst, &map_c, 0, tt * kBlk, 0, s.b, fb);
          }
        }
      }
      for (int k = 1; k <= S && k <= m; ++k) {  // no copy in flight at exit
        const int mm = m - k;
        tc::wait_drain<false>(&bars[kBarFull + mm % S], (mm / S) & 1, ab);
      }
    }
  } else if (warp == 2 || warp == 3) {
    // -------------------------------------------------------------- tail warps: rows past the sequence end
    // of a block are zeroed in the latent chunks (NaN slack must not meet a zero weight)
    const int t = tid - 64;
    int m = 0;
    bool ok = true;
    for (int64_t x = lo; x < hi && ok;) {
      const Seg s = seg_at(pre, B, x, hi, p, cap);
      x += s.ntile;
      for (int j = 0; j < s.ntile; ++j, ++m) {
        const int tt = s.t_begin + j, st = m % S;
        if (!tc::wait<false>(&bars[kBarFull + st], (m / S) & 1, ab)) {
          ok = false;
          break;
        }
        const int rows = tile_rows(s, tt);
        if (rows < kBlk) {
          uint8_t* blk = sm + st * kBlkBytes;
          const int per_chunk = (kBlk - rows) * 8;  // 16-byte pieces per chunk
          for (int i = t; i < 8 * per_chunk; i += 64) {
            const int c = i / per_chunk, k = i % per_chunk;
            *reinterpret_cast<uint4*>(blk + c * kChunkBytes + (rows + (k >> 3)) * 128 + (k & 7) * 16) =
                make_uint4(0, 0, 0, 0);
          }
          tc::fence_async_smem();
          tc::mbar_arrive(&bars[kBarFix + st]);
        }
        tc::mbar_arrive(&bars[kBarEmpty + st]);
      }
    }
  } else if (warp == 7) {
    // -------------------------------------------------------------- zero query rows 96-127 of TMEM once
    const uint32_t lane_t = tb + ((uint32_t)((warp & 3) * 32) << 16);
    uint32_t z[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) z[i] = 0u;
#pragma unroll 1
    for (int c = 0; c < 9; ++c) tc::tmem_st32(lane_t + kColQ + 32 * c, z);
    tc::tmem_wait_st();
    tc::tc_fence_before();
    tc::mbar_arrive(&bars[kBarQzero]);
  }
  else if (warp == 1 || warp == 5) {
    if (warp == 5) {  // zero query rows 32-63 of TMEM once, then lane 0 issues the value MMAs
      uint32_t z[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) z[i] = 0u;
#pragma unroll 1
      for (int c = 0; c < 9; ++c) tc::tmem_st32(tb + (32u << 16) + kColQ + 32 * c, z);
      tc::tmem_wait_st();
      tc::tc_fence_before();
      tc::mbar_arrive(&bars[kBarQzero]);
    }
    if (lane == 0) {
      // ------------------------------------------------------------ MMA issue: warp 1 the scores,
      // warp 5 the values (two issuing threads, so a value product waiting for
      // its softmax never sits behind the next block's score in one thread's
      // blocking issue; each thread's commits track its own MMAs)
      constexpr uint32_t idS = tc::idesc_bf16(128, kBlk, 0, 0);  // Q (TMEM) x block rows (K-major)
      constexpr uint32_t idV = tc::idesc_bf16(128, kH, 1, 0);    // C^T (MN-major) x P^T (K-major)
      int ev = 0, oc = 0, ntail[kMaxSlots] = {0, 0, 0};
      bool ok = warp == 5 || tc::wait<false>(&bars[kBarQzero], 0, ab);
      auto post = [&](int type, int a0, int a1) -> bool {  // one event at a time
        evt_desc[0] = type;
        evt_desc[1] = a0;
        evt_desc[2] = a1;
        tc::mbar_arrive(&bars[kBarEvt]);
        ++ev;
        return type == kEvtExit || tc::wait<false>(&bars[kBarEvtDone], (ev - 1) & 1, ab);
      };
      auto drain = [&]() -> bool {
        tc::mma_commit(&bars[kBarOcomp]);
        return tc::wait<false>(&bars[kBarOcomp], (oc++) & 1, ab);
      };
      // score of block m (tile tt of segment s): S[m & 1] = Q . C^T over the 9 chunks
      auto score = [&](int m, const Seg& s, int tt) -> bool {
        const int st = m % S;
        if (m >= 2 && !tc::wait<false>(&bars[kBarSfree + (m & 1)], ((m >> 1) - 1) & 1, ab)) return false;
        if (!tc::wait<false>(&bars[kBarFull + st], (m / S) & 1, ab)) return false;
        if (tile_rows(s, tt) < kBlk) {
          if (!tc::wait<false>(&bars[kBarFix + st], ntail[st] & 1, ab)) return false;
          ++ntail[st];
        }
        tc::tc_fence_after();
        const uint32_t dS = tb + kColS + (m & 1) * kBlk, blk = ring + st * kBlkBytes;
#pragma unroll
        for (int c = 0; c < 9; ++c)
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            tc::mma_ts(dS, tb + kColQ + c * 32 + kk * 8, tc::smem_desc(blk + c * kChunkBytes + kk * 32, 16, 1024),
                       idS, (c | kk) != 0 ? 1u : 0u);
        tc::mma_commit(&bars[kBarSfull + (m & 1)]);
        return true;
      };
      // value of block m: O^T += C^T . P^T (four 128-row latent blocks)
      auto value = [&](int m, bool first) -> bool {
        const int st = m % S, pb = m & 1;
        if (!tc::wait<false>(&bars[kBarPfull + pb], (m >> 1) & 1, ab)) return false;
        const volatile int* fl = reinterpret_cast<const volatile int*>(sm + L.off_p + pb * kPBufBytes + kPMetaFlag);
        if (!first && *fl) {  // the reference maximum moved: rescale O first
          if (!drain() || !post(kEvtRescale, pb, 0)) return false;
        }
        tc::tc_fence_after();
        const uint32_t blk = ring + st * kBlkBytes, pa = pbuf + pb * kPBufBytes;
#pragma unroll
        for (int mb = 0; mb < 4; ++mb)
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            tc::mma_ss(tb + kColO + mb * kH, tc::smem_desc(blk + mb * 2 * kChunkBytes + kk * 2048, kChunkBytes, 1024),
                       tc::smem_desc(pa + kk * 32, 16, 1024), idV, (first && kk == 0) ? 0u : 1u);
        tc::mma_commit(&bars[kBarEmpty + st]);
        tc::mma_commit(&bars[kBarPfree + pb]);
        return true;
      };
      int m = 0, k = 0;
      if (warp == 1) {
        for (int64_t x = lo; x < hi && ok; ++k) {
          const Seg s = seg_at(pre, B, x, hi, p, cap);
          x += s.ntile;
          if (!tc::wait<false>(&bars[kBarQready + (k & 1)], (k >> 1) & 1, ab)) break;
          for (int j = 0; j < s.ntile && ok; ++j) ok = score(m + j, s, s.t_begin + j);
          m += s.ntile;
        }
        tc::mma_commit(&bars[kBarDrained]);
        tc::wait_drain<false>(&bars[kBarDrained], 0, ab);
      } else {
        for (int64_t x = lo; x < hi && ok; ++k) {
          const Seg s = seg_at(pre, B, x, hi, p, cap);
          x += s.ntile;
          for (int j = 0; j < s.ntile && ok; ++j) ok = value(m + j, j == 0);
          m += s.ntile;
          // segment end: the partial goes out before the next segment overwrites O
          if (!ok || !drain() || !post(kEvtEpilogue, k % kStatBufs, (int)(g + s.b))) break;
        }
        post(kEvtExit, 0, 0);
        tc::mma_commit(&bars[kBarDrainedV]);
        tc::wait_drain<false>(&bars[kBarDrainedV], 0, ab);
      }
    }
  } else if (warp == 4 || warp == 6) {
    // -------------------------------------------------------------- query loads and softmax (lane = head)
    // Even segments on warp 4 with their query in TMEM rows 0-15, odd ones on
    // warp 6 with rows 64-79 (rows 16-31 / 80-95 zero): the product's rows are
    // independent, so each warp loads its next query (segment k + 2) while the
    // other segment's scores run, and a segment change waits for no load.
    const int par = warp == 4 ? 0 : 1;
    const uint32_t lane_t = tb + ((uint32_t)((warp & 3) * 32) << 16);
    const int h = lane;
    auto load_q = [&](int b, int kq) {
      // nine rounds of 128 bytes per row, the loads of round c + 1 in flight
      // while round c is stored (one round at a time took ~1 us of latency each)
      const uint4* row = reinterpret_cast<const uint4*>(p.q + ((int64_t)b * kH + (h & (kH - 1))) * kD);
      uint4 v[2][8];
#pragma unroll
      for (int i = 0; i < 8; ++i) v[0][i] = h < kH ? __ldg(row + i) : make_uint4(0, 0, 0, 0);
#pragma unroll
      for (int c = 0; c < 9; ++c) {
        if (c + 1 < 9) {
#pragma unroll
          for (int i = 0; i < 8; ++i)
            v[(c + 1) & 1][i] = h < kH ? __ldg(row + (c + 1) * 8 + i) : make_uint4(0, 0, 0, 0);
        }
        uint32_t r[32];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          r[4 * i] = v[c & 1][i].x;
          r[4 * i + 1] = v[c & 1][i].y;
          r[4 * i + 2] = v[c & 1][i].z;
          r[4 * i + 3] = v[c & 1][i].w;
        }
        tc::tmem_st32(lane_t + kColQ + 32 * c, r);
      }
      tc::tmem_wait_st();
      tc::tc_fence_before();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&bars[kBarQready + (kq & 1)]);
    };
    {  // this warp's first segment (0 or 1)
      int64_t x = lo;
      if (par == 1 && x < hi) x += seg_at(pre, B, x, hi, p, cap).ntile;
      if (x < hi) load_q(seq_of_tile(pre, B, x), par);
    }
    // The two warps share the S and P barriers, whose parity waits are right
    // only for the next phase: a warp starts segment k once the other warp has
    // read the last S of segment k - 1 (then every earlier phase has completed).
    int m = 0, k = 0, nh = 0;
    bool ok = true;
    for (int64_t x = lo; x < hi && ok; ++k) {
      const Seg s = seg_at(pre, B, x, hi, p, cap);
      x += s.ntile;
      if ((k & 1) != par) {  // the other warp's segment
        m += s.ntile;
        continue;
      }
      if (k >= 1 && !tc::wait<false>(&bars[kBarHand + par], (nh++) & 1, ab)) break;
      // where segment k + 2 (this warp's next) starts; its query is warmed in L2 now
      int64_t x2 = x;
      if (x2 < hi) x2 += seg_at(pre, B, x2, hi, p, cap).ntile;
      if (x2 < hi && lane == 0)
        tc::prefetch_l2(p.q + (int64_t)seq_of_tile(pre, B, x2) * kH * kD, (uint32_t)(kH * kD * 2));
      float m_ref = -INFINITY, l = 0.f, lq = 0.f;
      for (int j = 0; j < s.ntile; ++j, ++m) {
        const int tt = s.t_begin + j;
        if (!tc::wait<false>(&bars[kBarSfull + (m & 1)], (m >> 1) & 1, ab)) {
          ok = false;
          break;
        }
        tc::tc_fence_after();
        uint32_t sa[32], sb[32];
        tc::tmem_ld32(lane_t + kColS + (m & 1) * kBlk, sa);
        tc::tmem_ld32(lane_t + kColS + (m & 1) * kBlk + 32, sb);
        tc::tmem_wait_ld();
        tc::tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          tc::mbar_arrive(&bars[kBarSfree + (m & 1)]);
          if (j + 1 == s.ntile && x < hi) tc::mbar_arrive(&bars[kBarHand + (par ^ 1)]);  // the next segment's warp may start
        }
        const int nvalid = tile_rows(s, tt);
        if (nvalid < kBlk) {  // tokens past the sequence end take no weight
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            if (c >= nvalid) sa[c] = __float_as_uint(-INFINITY);
            if (c + 32 >= nvalid) sb[c] = __float_as_uint(-INFINITY);
          }
        }
        float mx[16];
#pragma unroll
        for (int i = 0; i < 16; ++i)
          mx[i] = fmaxf(tc::max3(__uint_as_float(sa[i]), __uint_as_float(sa[i + 16]), __uint_as_float(sb[i])),
                        __uint_as_float(sb[i + 16]));
#pragma unroll
        for (int i = 0; i < 5; ++i) mx[i] = tc::max3(mx[i], mx[i + 5], mx[i + 10]);
        const float mt = fmaxf(tc::max3(mx[0], mx[1], mx[2]), tc::max3(mx[3], mx[4], mx[15])) * p.scale_log2;
        float alpha = 1.f;
        if (j == 0) {
          m_ref = mt;
        } else if (mt > m_ref + kRescaleThreshold) {
          alpha = exp2f(m_ref - mt);
          l *= alpha;
          lq *= alpha;
          m_ref = mt;
        }
        uint32_t pk[32];
        {
          const uint64_t c2 = tc::f2(p.scale_log2, p.scale_log2), nm2 = tc::f2(-m_ref, -m_ref);
          uint64_t la[2] = {tc::f2(0.f, 0.f), tc::f2(0.f, 0.f)}, qa[2] = {la[0], la[0]};
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const uint32_t u0 = i < 16 ? sa[2 * i] : sb[2 * i - 32], u1 = i < 16 ? sa[2 * i + 1] : sb[2 * i - 31];
            const float2 xv = tc::f2_split(tc::f2_fma(tc::f2u(u0, u1), c2, nm2));
            const float p0 = tc::ex2(xv.x), p1 = tc::ex2(xv.y);
            pk[i] = tc::cvt_bf16x2(p0, p1);
            la[i & 1] = tc::f2_add(la[i & 1], tc::f2(p0, p1));
            qa[i & 1] = tc::f2_add(qa[i & 1], tc::f2u(pk[i] << 16, pk[i] & 0xFFFF0000u));
          }
          const float2 ls = tc::f2_split(tc::f2_add(la[0], la[1])), lr = tc::f2_split(tc::f2_add(qa[0], qa[1]));
          l += ls.x + ls.y;
          lq += lr.x + lr.y;
        }
        // hand P over: buffer m & 1 is free once the value MMAs of block m - 2 are done
        if (m >= 2 && !tc::wait<false>(&bars[kBarPfree + (m & 1)], ((m >> 1) - 1) & 1, ab)) {
          ok = false;
          break;
        }
        uint8_t* pbp = sm + L.off_p + (m & 1) * kPBufBytes;
        const bool any = __any_sync(0xffffffffu, h < kH && alpha != 1.f);
        if (h < kH) {
#pragma unroll
          for (int c = 0; c < 8; ++c)
            *reinterpret_cast<uint4*>(pbp + h * 128 + ((c ^ (h & 7)) * 16)) =
                make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
          reinterpret_cast<float*>(pbp + kPMetaAlpha)[h] = alpha;
          if (j + 1 == s.ntile) {  // the segment's statistics for the epilogue
            float* st = stats + (k % kStatBufs) * 3 * kH;
            st[h] = m_ref;
            st[kH + h] = l;
            st[2 * kH + h] = lq;
          }
        }
        if (lane == 0) *reinterpret_cast<int*>(pbp + kPMetaFlag) = any ? 1 : 0;
        tc::fence_async_smem();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(&bars[kBarPfull + (m & 1)]);
      }
      // every score of segment k is done (this warp read its last S): the rows
      // can take segment k + 2's query
      if (ok && x2 < hi) load_q(seq_of_tile(pre, B, x2), k + 2);
    }
  }
  else if (warp >= 8) {
    // -------------------------------------------------------------- rescale / epilogue (thread = latent row)
    // O^T block mb holds latent rows 128 mb + (TMEM lane), columns = heads
    const int r = (warp & 3) * 32 + lane;
    const uint32_t lane_t = tb + ((uint32_t)((warp & 3) * 32) << 16);
    for (int e = 0;; ++e) {
      if (!tc::wait<false>(&bars[kBarEvt], e & 1, ab)) break;
      tc::tc_fence_after();
      const int type = evt_desc[0], a0 = evt_desc[1], a1 = evt_desc[2];
      if (type == kEvtExit) break;
      uint32_t o[2][32];  // O^T columns [0, 64): block mb = c / 16, head = c % 16
      tc::tmem_ld32(lane_t + kColO, o[0]);
      tc::tmem_ld32(lane_t + kColO + 32, o[1]);
      tc::tmem_wait_ld();
      if (type == kEvtRescale) {
        const float* alpha = reinterpret_cast<const float*>(sm + L.off_p + a0 * kPBufBytes + kPMetaAlpha);
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          o[0][i] = __float_as_uint(__uint_as_float(o[0][i]) * alpha[i & (kH - 1)]);
          o[1][i] = __float_as_uint(__uint_as_float(o[1][i]) * alpha[i & (kH - 1)]);
        }
        tc::tmem_st32(lane_t + kColO, o[0]);
        tc::tmem_st32(lane_t + kColO + 32, o[1]);
        tc::tmem_wait_st();
      } else {
        // partial of slot a1: o / lq and lse per head, in the shape-generic
        // layout.  The accumulator is in registers now, so the MMA thread may
        // start the next segment (overwriting it) while the stores go out.
        tc::tc_fence_before();
        tc::mbar_arrive(&bars[kBarEvtDone]);
        const float* st = stats + a0 * 3 * kH;
        // the 16 normalisers into registers first: read through the pointer
        // between the global stores they would be reloaded after every store
        float inv[kH];
#pragma unroll
        for (int hh = 0; hh < kH; ++hh) inv[hh] = 1.f / st[2 * kH + hh];
        float* dst = p.o_part + (int64_t)a1 * kH * kDC + r;
#pragma unroll
        for (int i = 0; i < 64; ++i) {
          const int mb = i >> 4, hh = i & (kH - 1);
          dst[hh * kDC + mb * 128] = __uint_as_float(o[i >> 5][i & 31]) * inv[hh];
        }
        if (warp == 8 && lane < kH) p.lse_part[(int64_t)a1 * kH + lane] = (st[lane] + log2f(st[kH + lane])) * kLn2;
        continue;
      }
      tc::tc_fence_before();
      tc::mbar_arrive(&bars[kBarEvtDone]);
    }
  }

  tc::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tb, 512);
  }
}

// ------------------------------------------------------------------ combine
// lse = log sum_s exp(lse_s);  z = sum_s exp(lse_s - lse) o_s over the partials
// of the workers first..last that the partial pass recorded for sequence b
// (workers without tiles in between wrote nothing).  Block = sequence, warp =
// head, lane = 16 latent columns.
template <bool ZF32>
__global__ void __launch_bounds__(512) combine_lh_kernel(const DecodeLaunch a) {
  // launched as a programmatic dependent of the partial pass: wait for it (and
  // its memory) before reading anything it wrote
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int b = blockIdx.x, h = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int T = a.plan_flag[1], G = a.plan_flag[2];
  const int g0 = a.seqplan[2 * b], g1 = a.seqplan[2 * b + 1];
  float* zf = static_cast<float*>(a.z_out) + ((int64_t)b * kH + h) * kDC + lane * 16;
  __nv_bfloat16* zb = static_cast<__nv_bfloat16*>(a.z_out) + ((int64_t)b * kH + h) * kDC + lane * 16;
  // a partial pass that gave up on a bounded wait left partials unwritten: the
  // outputs are NaN then, not stale numbers
  const bool failed = a.status != nullptr && *reinterpret_cast<volatile int32_t*>(a.status) == MLA_ERR_DEVICE_TIMEOUT;
  if (g1 < g0 || failed) {
    const float zv = failed ? __int_as_float(0x7fc00000) : 0.f;
    for (int d = 0; d < 16; ++d) {
      if (ZF32) zf[d] = zv; else zb[d] = __float2bfloat16_rn(zv);
    }
    if (lane == 0 && a.lse_out) a.lse_out[(int64_t)b * kH + h] = failed ? zv : -INFINITY;
    return;
  }
  auto live = [&](int g) { return worker_begin(g + 1, T, G) > worker_begin(g, T, G); };
  float mx = -INFINITY;
  for (int g = g0; g <= g1; ++g)
    if (live(g)) mx = fmaxf(mx, a.lse_part[((int64_t)g + b) * kH + h]);
  float sum = 0.f;
  for (int g = g0; g <= g1; ++g)
    if (live(g)) sum += expf(a.lse_part[((int64_t)g + b) * kH + h] - mx);
  const float lse = mx + logf(sum);
  float4 acc[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) acc[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int g = g0; g <= g1; ++g) {
    if (!live(g)) continue;
    const int64_t slot = (int64_t)g + b;
    const float w = expf(a.lse_part[slot * kH + h] - lse);
    const float4* src = reinterpret_cast<const float4*>(a.o_part + (slot * kH + h) * kDC + lane * 16);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float4 v = src[i];
      acc[i].x += w * v.x;
      acc[i].y += w * v.y;
      acc[i].z += w * v.z;
      acc[i].w += w * v.w;
    }
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    if (ZF32) {
      reinterpret_cast<float4*>(zf)[i] = acc[i];
    } else {
      reinterpret_cast<uint2*>(zb)[i] = make_uint2(pack_bf16x2(acc[i].x, acc[i].y), pack_bf16x2(acc[i].z, acc[i].w));
    }
  }
  if (lane == 0 && a.lse_out) a.lse_out[(int64_t)b * kH + h] = lse;
}

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

bool lh_supported(const DecodeLaunch& a) {
  return a.n_heads == kH && a.d_latent == kDC && a.d_rope == 64 && a.batch <= kMaxBatch;
}

cudaError_t launch_decode_lh(const DecodeLaunch& a, cudaStream_t s) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return cudaErrorNotSupported;
  // the cache as a 4-D tensor (64 columns, tokens, 9 column chunks, sequence or
  // block); one box = a whole 64-token block, chunk-major
  const bool paged = a.block_table != nullptr;
  const cuuint64_t row = (cuuint64_t)kD * 2;
  const cuuint64_t dims[4] = {64, paged ? (cuuint64_t)kBlk : (cuuint64_t)a.seq_stride, 9,
                              paged ? (cuuint64_t)a.num_blocks : (cuuint64_t)a.batch};
  const cuuint64_t strides[3] = {row, 128, (paged ? (cuuint64_t)kBlk : (cuuint64_t)a.seq_stride) * row};
  const cuuint32_t box[4] = {64, kBlk, 9, 1}, es[4] = {1, 1, 1, 1};
  CUtensorMap map;
  if (enc(&map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(a.pool), dims, strides, box, es,
          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  LhParams p;
  p.q = static_cast<const __nv_bfloat16*>(a.q);
  p.block_table = a.block_table;
  p.max_blocks = a.max_blocks;
  p.num_blocks = a.num_blocks;
  p.seq_stride = a.seq_stride;
  p.seqlens = a.seqlens;
  p.batch = a.batch;
  p.paged = paged ? 1 : 0;
  p.workers = a.workers;
  p.slots = lh_slots(a.batch);
  p.scale_log2 = a.scale * kLog2e;
  p.o_part = a.o_part;
  p.lse_part = a.lse_part;
  p.status = a.status;
  p.plan_hdr = a.plan_flag;
  p.seqplan = a.seqplan;
  const int smem = lh_layout(p.slots, a.batch).total;
  cudaError_t e = ensure_smem<decode_lh_kernel>(smem);
  if (e != cudaSuccess) return e;
  decode_lh_kernel<<<a.workers, kThreads, smem, s>>>(map, p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  // the combine as a programmatic dependent launch (see the 128-head path)
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.batch);
  cfg.blockDim = dim3(512);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return a.z_is_fp32 ? cudaLaunchKernelEx(&cfg, combine_lh_kernel<true>, a)
                     : cudaLaunchKernelEx(&cfg, combine_lh_kernel<false>, a);
}

}  // namespace mla

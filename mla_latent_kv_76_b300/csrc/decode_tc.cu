// Tensor-core split-KV decode for the DeepSeek-V3 head shape: n_h = 128,
// d_c = 512, d_R = 64 (576-wide cache rows), on tcgen05 / TMEM / TMA.
//
// What is computed ("结合 DeepSeek 推理代码看 MLA": score = (q^C W^UK).c^KV +
// q^R.k^R; worked example steps 4-5: scale, causal mask, softmax, z = A.kv):
// for every head i and visible token j of a sequence
//   s_j = scale * [q~_i ; q^R_i] . [c_j ; k^R_j],   z_i = sum_j softmax(s)_j c_j.
//
// Decomposition.  The fp32 accumulator O = 128 heads x 512 latent fills the
// whole tensor memory of one SM, so a pair of CTAs (a cluster of two, one
// per SM) shares every 64-token tile:
//   CTA r owns latent columns [256 r, 256 r + 256) of O and of the score
//   contraction; CTA 1 also owns the 64 RoPE columns.  Each CTA TMA-loads
//   only its columns of the tile (every cache byte leaves HBM once), computes
//   its partial score S_r = Q[:, cols_r] . C[:, cols_r]^T on the tensor core,
//   and the two partials are swapped through distributed shared memory, so
//   both CTAs hold the same S = S_0 + S_1 (fp32 addition commutes: the two
//   copies are bitwise equal) and run the same online softmax.  Each then
//   accumulates O[:, 256 r : 256 r + 256] += P . C[:, 256 r : 256 r + 256].
//
// Per CTA (256 threads):
//   warp 0      TMA producer: one 64x64 bf16 box per 64-column chunk, three
//               40 KB stages, 128-byte swizzle (the canonical K-major layout
//               of the score MMA and the MN-major layout of the value MMA)
//   warp 1      tcgen05.mma issuer (single thread) and TMEM owner
//   warps 2-3   zero the rows past the sequence end in the last tile (NaN
//               garbage in block slack must not meet a zero weight in the MMA);
//               they see every fill of every stage and release it too
//   warps 4-7   one thread per head: load Q, exchange the partial score,
//               online softmax, write P (bf16) for the value MMA, rescale O
//               when the running maximum grows, write the segment's partial
// Tensor memory (512 columns x 128 lanes): O [0, 256), S double buffer
// [256, 384), the CTA's Q columns as packed bf16 [384, 512) (A operand of
// the score MMA read straight from TMEM).
//
// Online softmax with a lazily updated reference maximum: P = 2^(x - m_ref)
// with x = s * scale * log2(e); m_ref moves (and O, l are rescaled) only when
// a tile's maximum exceeds m_ref by more than 8, so P <= 256 and O never
// overflows; the result is exact after the final division by l.
#include <cuda.h>
#include <mutex>

#include "common.cuh"
#include "kernels.h"
#include "plan.cuh"
#include "tc.cuh"

namespace mla {
namespace {

constexpr int kH = 128, kDC = 512, kD = 576;
constexpr int kStages = 3;
constexpr int kChunkBytes = 64 * 128;           // 64 tokens x 64 bf16, one 128-byte row per token
constexpr int kStageBytes = 5 * kChunkBytes;    // up to 5 chunks per CTA (CTA 1: 4 latent + RoPE)
constexpr int kQropeBytes = kH * 128;           // RoPE part of Q, 128 heads x 64 bf16
constexpr int kPBytes = kH * 128;               // P, 128 heads x 64 tokens bf16
constexpr int kRecvBytes = kH * 64 * 4;         // partial score from the peer, fp32
constexpr int kOffStage = 0;
constexpr int kOffQrope = kOffStage + kStages * kStageBytes;
constexpr int kOffP = kOffQrope + kQropeBytes;
constexpr int kOffRecv = kOffP + 2 * kPBytes;
constexpr int kOffBar = kOffRecv + kRecvBytes;
constexpr int kNumBars = 21;
constexpr int kOffMisc = kOffBar + kNumBars * 8;
constexpr int kOffPrefix = kOffMisc + 16;
constexpr int kTcMaxBatch = 1024;
constexpr int kThreads = 256;

// TMEM column map
constexpr uint32_t kColO = 0, kColS = 256, kColQ = 384;

constexpr float kRescaleThreshold = 8.f;  // log2 units

size_t tc_smem_bytes(int batch) { return (size_t)kOffPrefix + (size_t)(batch + 1) * 4 + 1024; }

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
  float* o_part;    // [(G + B)][128][512]
  float* lse_part;  // [(G + B)][128]
  int32_t* status;
};

// One segment of a worker's tile range: tiles [t_begin, t_begin + ntile) of sequence b.
struct Seg {
  int b, t_begin, ntile, len;
};

MLA_DEVI Seg seg_at(const int* pre, int B, int64_t x, int64_t hi, const TcParams& p, int64_t cap) {
  Seg s;
  s.b = seq_of_tile(pre, B, x);
  s.t_begin = (int)(x - pre[s.b]);
  const int64_t e = pre[s.b + 1] < hi ? pre[s.b + 1] : hi;
  s.ntile = (int)(e - x);
  s.len = effective_len(p.seqlens, s.b, cap, nullptr);
  return s;
}

// The last tile of a sequence whose length is not a multiple of 64 has rows
// past the end that must be zeroed before the value MMA.
MLA_DEVI bool is_tail(const Seg& s, int j) {
  return (s.len & 63) != 0 && s.t_begin + j == tiles_of(s.len) - 1;
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    decode_tc_kernel(const __grid_constant__ CUtensorMap cache_map, const TcParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + kOffBar);
  uint64_t* full = bars + 0;      // [3] TMA landed (count 1 + tx)
  // [3] stage free again: the value MMA's commit plus the 64 tail-zeroing
  // threads, which therefore see every fill of every stage in order
  uint64_t* empty = bars + 3;
  uint64_t* sfull = bars + 6;     // [2] score MMA done (commit)
  uint64_t* sfree = bars + 8;     // [2] score read out of TMEM (128)
  uint64_t* pfull = bars + 10;    // [2] P written (128)
  uint64_t* odone = bars + 12;    // value MMA of a tile done (commit)
  uint64_t* ofree = bars + 13;    // O read out at a segment end (128)
  uint64_t* qready = bars + 14;   // Q of the segment in TMEM / smem (128)
  uint64_t* recvfull = bars + 15; // the peer's partial score arrived (128 remote)
  uint64_t* peerfree = bars + 16; // the peer consumed what this CTA sent (128 remote)
  uint64_t* drained = bars + 17;  // all MMAs of this CTA done (commit, at exit)
  // [3] tail rows of the stage zeroed (64).  One per stage: a stage cannot be
  // refilled before the MMA has consumed its tail, so no phase is ever skipped.
  uint64_t* fixdone = bars + 18;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + kOffMisc);
  int* abort_flag = reinterpret_cast<int*>(sm + kOffMisc + 4);
  int* pre = reinterpret_cast<int*>(sm + kOffPrefix);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t rank = tc::cluster_rank(), peer = rank ^ 1u;
  const int g = (int)(blockIdx.x >> 1);
  const int64_t cap = p.paged ? (int64_t)p.max_blocks * kTileTokens : p.seq_stride;

  if (tid == 0) {
    for (int i = 0; i < 3; ++i) {
      tc::mbar_init(&full[i], 1);
      tc::mbar_init(&empty[i], 1 + 64);
    }
    for (int i = 0; i < 2; ++i) {
      tc::mbar_init(&sfull[i], 1);
      tc::mbar_init(&sfree[i], 128);
      tc::mbar_init(&pfull[i], 128);
    }
    tc::mbar_init(odone, 1);
    tc::mbar_init(ofree, 128);
    tc::mbar_init(qready, 128);
    for (int i = 0; i < 3; ++i) tc::mbar_init(&fixdone[i], 64);
    tc::mbar_init(recvfull, 128);
    tc::mbar_init(peerfree, 128);
    tc::mbar_init(drained, 1);
    *abort_flag = 0;
    tc::fence_mbar_init();
  }
  if (warp == 1) tc::tmem_alloc(tmem_slot, 512);
  tile_prefix(p.seqlens, p.batch, cap, p.status, pre);  // ends with __syncthreads
  tc::tc_fence_before();
  tc::cluster_sync();  // both CTAs' barriers initialised before any remote arrival
  tc::tc_fence_after();
  const uint32_t tb = *tmem_slot;
  const tc::Abort ab{abort_flag, p.status};

  const int B = p.batch, G = p.workers;
  const int64_t T = pre[B];
  const int64_t lo = worker_begin(g, T, G), hi = worker_begin(g + 1, T, G);
  const int chunk0 = (int)rank * 4;
  const int nchunk = rank ? 5 : 4;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      tc::prefetch_map(&cache_map);
      int n = 0;
      bool ok = true;
      for (int64_t x = lo; x < hi && ok;) {
        const Seg s = seg_at(pre, B, x, hi, p, cap);
        x += s.ntile;
        for (int j = 0; j < s.ntile; ++j, ++n) {
          const int st = n % kStages;
          if (n >= kStages && !tc::wait<false>(&empty[st], ((n / kStages) - 1) & 1, ab)) {
            ok = false;
            break;
          }
          uint8_t* dst = sm + kOffStage + st * kStageBytes;
          const int tt = s.t_begin + j;
          if (p.paged) {
            const int blk = p.block_table[(int64_t)s.b * p.max_blocks + tt];
            if (blk < 0 || blk >= p.num_blocks) {
              // unreadable block: its rows count as zeros
              report(p.status, MLA_ERR_DEVICE_BOUNDS);
              uint4* z = reinterpret_cast<uint4*>(dst);
              for (int i = 0; i < nchunk * kChunkBytes / 16; ++i) z[i] = make_uint4(0, 0, 0, 0);
              tc::fence_async_smem();
              tc::mbar_arrive(&full[st]);
              continue;
            }
            tc::mbar_expect_tx(&full[st], nchunk * kChunkBytes);
            for (int c = 0; c < nchunk; ++c)
              tc::tma_load_3d(dst + c * kChunkBytes, &cache_map, (chunk0 + c) * 64, 0, blk, &full[st]);
          } else {
            tc::mbar_expect_tx(&full[st], nchunk * kChunkBytes);
            for (int c = 0; c < nchunk; ++c)
              tc::tma_load_3d(dst + c * kChunkBytes, &cache_map, (chunk0 + c) * 64, tt * 64, s.b, &full[st]);
          }
        }
      }
      // never leave with a copy in flight: wait for the last use of every stage
      for (int k = 1; k <= kStages && k <= n; ++k) {
        const int m = n - k;
        tc::wait<false>(&full[m % kStages], (m / kStages) & 1, ab);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idS = tc::idesc_bf16(128, 64, 0, 0);
      constexpr uint32_t idO = tc::idesc_bf16(128, 256, 0, 1);
      const uint32_t sbase = smem_u32(sm + kOffStage);
      const uint32_t qrope = smem_u32(sm + kOffQrope);
      const uint32_t pbase = smem_u32(sm + kOffP);
      int n = 0, seg_i = 0;
      int ntail[kStages] = {0, 0, 0};
      bool ok = true;
      auto issue_o = [&](int m, bool first_in_seg) -> bool {
        if (!tc::wait<false>(&pfull[m & 1], (m >> 1) & 1, ab)) return false;
        if (first_in_seg && seg_i > 0 && !tc::wait<false>(ofree, (seg_i - 1) & 1, ab)) return false;
        tc::tc_fence_after();
        const uint32_t stg = sbase + (m % kStages) * kStageBytes;
        const uint32_t pb = pbase + (m & 1) * kPBytes;
#pragma unroll
        for (int k = 0; k < 4; ++k)
          tc::mma_ss(tb + kColO, tc::smem_desc(pb + k * 32, 16, 1024), tc::smem_desc(stg + k * 2048, kChunkBytes, 1024),
                     idO, (first_in_seg && k == 0) ? 0u : 1u);
        tc::mma_commit(&empty[m % kStages]);
        tc::mma_commit(odone);
        return true;
      };
      for (int64_t x = lo; x < hi && ok;) {
        const Seg s = seg_at(pre, B, x, hi, p, cap);
        x += s.ntile;
        if (!tc::wait<false>(qready, seg_i & 1, ab)) break;
        tc::tc_fence_after();
        for (int j = 0; j < s.ntile; ++j) {
          const int m = n + j;
          const int st = m % kStages;
          if (!tc::wait<false>(&full[st], (m / kStages) & 1, ab)) { ok = false; break; }
          if (is_tail(s, j)) {
            if (!tc::wait<false>(&fixdone[st], ntail[st] & 1, ab)) { ok = false; break; }
            ++ntail[st];
          }
          if (m >= 2 && !tc::wait<false>(&sfree[m & 1], ((m >> 1) - 1) & 1, ab)) { ok = false; break; }
          tc::tc_fence_after();
          const uint32_t stg = sbase + st * kStageBytes;
          const uint32_t dS = tb + kColS + (m & 1) * 64;
#pragma unroll
          for (int k = 0; k < 16; ++k)
            tc::mma_ts(dS, tb + kColQ + k * 8, tc::smem_desc(stg + (k >> 2) * kChunkBytes + (k & 3) * 32, 16, 1024),
                       idS, k > 0 ? 1u : 0u);
          if (rank == 1) {
#pragma unroll
            for (int k = 0; k < 4; ++k)
              tc::mma_ss(dS, tc::smem_desc(qrope + k * 32, 16, 1024),
                         tc::smem_desc(stg + 4 * kChunkBytes + k * 32, 16, 1024), idS, 1u);
          }
          tc::mma_commit(&sfull[m & 1]);
          if (j >= 1 && !issue_o(m - 1, j == 1)) { ok = false; break; }
        }
        if (!ok) break;
        if (!issue_o(n + s.ntile - 1, s.ntile == 1)) break;
        n += s.ntile;
        ++seg_i;
      }
      // drain: nothing may still read or write TMEM / shared memory at exit
      tc::mma_commit(drained);
      tc::wait<false>(drained, 0, ab);
    }
  } else if (warp < 4) {
    // ------------------------------------------------------------ tail zeroing
    const int t = tid - 64;  // 0..63
    int n = 0;
    bool ok = true;
    for (int64_t x = lo; x < hi && ok;) {
      const Seg s = seg_at(pre, B, x, hi, p, cap);
      x += s.ntile;
      for (int j = 0; j < s.ntile; ++j) {
        const int m = n + j;
        if (!tc::wait<false>(&full[m % kStages], (m / kStages) & 1, ab)) { ok = false; break; }
        if (is_tail(s, j)) {
          uint8_t* stg = sm + kOffStage + (m % kStages) * kStageBytes;
          const int r0 = s.len & 63;
          const int per_chunk = (64 - r0) * 8;  // 16-byte pieces per chunk
          for (int i = t; i < 4 * per_chunk; i += 64) {
            const int c = i / per_chunk, k = i % per_chunk;
            *reinterpret_cast<uint4*>(stg + c * kChunkBytes + (r0 + (k >> 3)) * 128 + (k & 7) * 16) =
                make_uint4(0, 0, 0, 0);
          }
          tc::fence_async_smem();
          tc::mbar_arrive(&fixdone[m % kStages]);
        }
        tc::mbar_arrive(&empty[m % kStages]);
      }
      n += s.ntile;
    }
  } else {
    // ------------------------------------------------------------ softmax (thread = head)
    const int h = tid - 128;
    const int wq = warp - 4;
    const uint32_t lane_t = tb + ((uint32_t)(wq * 32) << 16);
    const float4* recv = reinterpret_cast<const float4*>(sm + kOffRecv);
    const uint32_t peer_recv = tc::map_peer(sm + kOffRecv, peer) + (uint32_t)h * 16u;
    uint8_t* qrope_s = sm + kOffQrope;

    auto load_q = [&](int b) {
      const __nv_bfloat16* row = p.q + ((int64_t)b * kH + h) * kD;
      const uint4* src = reinterpret_cast<const uint4*>(row + rank * 256);
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t r[32];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const uint4 v = __ldg(src + c * 8 + i);
          r[4 * i] = v.x;
          r[4 * i + 1] = v.y;
          r[4 * i + 2] = v.z;
          r[4 * i + 3] = v.w;
        }
        tc::tmem_st32(lane_t + kColQ + c * 32, r);
      }
      if (rank == 1) {
        const uint4* srcr = reinterpret_cast<const uint4*>(row + kDC);
#pragma unroll
        for (int c = 0; c < 8; ++c)
          *reinterpret_cast<uint4*>(qrope_s + h * 128 + ((c ^ (h & 7)) * 16)) = __ldg(srcr + c);
      }
      tc::tmem_wait_st();
      tc::fence_async_smem();
      tc::tc_fence_before();
      tc::mbar_arrive(qready);
    };

    int n = 0;
    bool ok = true;
    bool first_seg = true;
    for (int64_t x = lo; x < hi && ok;) {
      const Seg s = seg_at(pre, B, x, hi, p, cap);
      x += s.ntile;
      if (first_seg) load_q(s.b);
      first_seg = false;
      float m_ref = -INFINITY, l = 0.f;
      for (int j = 0; j < s.ntile; ++j) {
        const int m = n + j;
        if (!tc::wait<false>(&sfull[m & 1], (m >> 1) & 1, ab)) { ok = false; break; }
        tc::tc_fence_after();
        uint32_t sa[32], sb[32];
        tc::tmem_ld32(lane_t + kColS + (m & 1) * 64, sa);
        tc::tmem_ld32(lane_t + kColS + (m & 1) * 64 + 32, sb);
        tc::tmem_wait_ld();
        tc::tc_fence_before();
        tc::mbar_arrive(&sfree[m & 1]);
        // ---- swap partial scores with the peer CTA
        if (m >= 1 && !tc::wait<true>(peerfree, (m - 1) & 1, ab)) { ok = false; break; }
#pragma unroll
        for (int c4 = 0; c4 < 8; ++c4)
          tc::st_cluster_v4(peer_recv + c4 * kH * 16, __uint_as_float(sa[4 * c4]), __uint_as_float(sa[4 * c4 + 1]),
                            __uint_as_float(sa[4 * c4 + 2]), __uint_as_float(sa[4 * c4 + 3]));
#pragma unroll
        for (int c4 = 0; c4 < 8; ++c4)
          tc::st_cluster_v4(peer_recv + (8 + c4) * kH * 16, __uint_as_float(sb[4 * c4]),
                            __uint_as_float(sb[4 * c4 + 1]), __uint_as_float(sb[4 * c4 + 2]),
                            __uint_as_float(sb[4 * c4 + 3]));
        tc::mbar_arrive_remote(recvfull, peer);
        if (!tc::wait<true>(recvfull, m & 1, ab)) { ok = false; break; }
        float x64[64];
#pragma unroll
        for (int c4 = 0; c4 < 16; ++c4) {
          const float4 v = recv[c4 * kH + h];
          const uint32_t* own = c4 < 8 ? &sa[4 * c4] : &sb[4 * (c4 - 8)];
          x64[4 * c4 + 0] = __uint_as_float(own[0]) + v.x;
          x64[4 * c4 + 1] = __uint_as_float(own[1]) + v.y;
          x64[4 * c4 + 2] = __uint_as_float(own[2]) + v.z;
          x64[4 * c4 + 3] = __uint_as_float(own[3]) + v.w;
        }
        tc::mbar_arrive_remote(peerfree, peer);
        // ---- scale, mask, tile maximum
        const int nvalid = s.len - (s.t_begin + j) * 64;  // >= 1
        float mt = -INFINITY;
#pragma unroll
        for (int c = 0; c < 64; ++c) {
          x64[c] = (c < nvalid) ? x64[c] * p.scale_log2 : -INFINITY;
          mt = fmaxf(mt, x64[c]);
        }
        if (j >= 1) {
          if (!tc::wait<false>(odone, (m - 1) & 1, ab)) { ok = false; break; }
          tc::tc_fence_after();
        }
        // TMEM loads / stores are warp-collective: the warp rescales together,
        // heads that keep their reference maximum multiply by exactly 1
        const bool grow = mt > m_ref + kRescaleThreshold;
        const bool rescaled = __any_sync(0xffffffffu, grow && j >= 1);
        if (rescaled) {
          const float f = (grow && j >= 1) ? exp2f(m_ref - mt) : 1.f;
          l *= f;
#pragma unroll 1
          for (int c = 0; c < 8; ++c) {
            uint32_t r[32];
            tc::tmem_ld32(lane_t + kColO + c * 32, r);
            tc::tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * f);
            tc::tmem_st32(lane_t + kColO + c * 32, r);
          }
        }
        if (grow) m_ref = mt;
        // ---- P = 2^(x - m_ref) in bf16; l sums the rounded weights
        uint8_t* prow = sm + kOffP + (m & 1) * kPBytes + h * 128;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          uint32_t pk[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float p0 = exp2f(x64[8 * c + 2 * i] - m_ref);
            const float p1 = exp2f(x64[8 * c + 2 * i + 1] - m_ref);
            pk[i] = pack_bf16x2(p0, p1);
            l += __uint_as_float(pk[i] << 16) + __uint_as_float(pk[i] & 0xFFFF0000u);
          }
          *reinterpret_cast<uint4*>(prow + ((c ^ (h & 7)) * 16)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
        }
        tc::fence_async_smem();
        if (rescaled) tc::tmem_wait_st();
        tc::tc_fence_before();
        tc::mbar_arrive(&pfull[m & 1]);
      }
      if (!ok) break;
      n += s.ntile;
      // the next segment's Q can go in as soon as this segment's last score is read
      if (x < hi) load_q(seq_of_tile(pre, B, x));
      // ---- segment result: O / l and the log-sum-exp
      if (!tc::wait<false>(odone, (n - 1) & 1, ab)) break;
      tc::tc_fence_after();
      const float inv = 1.f / l;
      float* dst = p.o_part + (((int64_t)g + s.b) * kH + h) * kDC + rank * 256;
#pragma unroll 1
      for (int c = 0; c < 8; ++c) {
        uint32_t r[32];
        tc::tmem_ld32(lane_t + kColO + c * 32, r);
        tc::tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 8; ++i)
          reinterpret_cast<float4*>(dst + c * 32)[i] =
              make_float4(__uint_as_float(r[4 * i]) * inv, __uint_as_float(r[4 * i + 1]) * inv,
                          __uint_as_float(r[4 * i + 2]) * inv, __uint_as_float(r[4 * i + 3]) * inv);
      }
      if (rank == 0) p.lse_part[((int64_t)g + s.b) * kH + h] = (m_ref + log2f(l)) * kLn2;
      tc::tc_fence_before();
      tc::mbar_arrive(ofree);
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
  CUtensorMap map;
  cuuint64_t dims[3], strides[2];
  const cuuint32_t box[3] = {64, 64, 1}, es[3] = {1, 1, 1};
  dims[0] = kD;
  strides[0] = (cuuint64_t)kD * 2;
  if (a.block_table) {
    dims[1] = kTileTokens;
    dims[2] = (cuuint64_t)a.num_blocks;
    strides[1] = (cuuint64_t)kTileTokens * kD * 2;
  } else {
    dims[1] = (cuuint64_t)a.seq_stride;
    dims[2] = (cuuint64_t)a.batch;
    strides[1] = (cuuint64_t)a.seq_stride * kD * 2;
  }
  if (enc(&map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(a.pool), dims, strides, box, es,
          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  TcParams p;
  p.q = static_cast<const __nv_bfloat16*>(a.q);
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
  p.lse_part = a.lse_part;
  p.status = a.status;
  const size_t smem = tc_smem_bytes(a.batch);
  cudaError_t e = cudaFuncSetAttribute(decode_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  decode_tc_kernel<<<2 * a.workers, kThreads, smem, s>>>(map, p);
  return cudaGetLastError();
}

}  // namespace mla

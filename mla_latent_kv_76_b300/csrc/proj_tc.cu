// Tensor-core weight projections around decode, for the DeepSeek-V3 head
// shape (d_h = d_v = 128, d_c = 512, d_R = 64):
//   absorb    q~[b][i][n] = sum_k q^C[b][i][k] W^UK_i[k][n]   ("为什么矩阵吸收很关键":
//             q^C.(W^UK c) = (q^C W^UK).c), plus q^R rotated into columns [512, 576)
//   out-proj  o[b][i][v]  = sum_c z[b][i][c] W^UV_i[v][c]     (W^UV applied after the sum)
// Both stream 16.8 MB of weights that are read exactly once; one CTA per head
// TMA-loads its 128 KB weight matrix in one go and keeps it in shared memory.
//
// The batch is the MMA's M dimension (padded to 128): the activations' TMA
// boxes hold only the real rows (a multiple of 8), packed back to back and
// followed by the weights, so the MMA rows past the batch read other
// operands' bytes and their results are simply not stored.  Operands use the
// 128-byte-swizzled K-major layout (activations, W^UV) and MN-major layout
// (W^UK, whose d_c columns are contiguous).
#include <cuda.h>

#include <mutex>

#include "common.cuh"
#include "kernels.h"
#include "tc.cuh"

namespace mla {
namespace {

constexpr int kThreads = 128;
constexpr int kBox = 128 * 128;  // 64 bf16 x 128 rows

struct ProjParams {
  int batch, n_heads;
  __nv_bfloat16* out;
  int64_t out_sb, out_sh;  // element strides of batch and head in the output
  // absorb only
  const __nv_bfloat16* q_r;
  const int32_t* pos;
  RopeTurns rope;
};

MLA_DEVI bool wait_done(uint64_t* b, uint32_t parity) {
  const long long t0 = clock64();
  while (!tc::mbar_test(b, parity))
    if (clock64() - t0 > tc::kWaitCycles) return false;
  return true;
}

// ---------------------------------------------------------------- absorb
// smem: q^C boxes [2][rows8 x 128 B] at 0, then W^UK boxes [8][128 k x 128 B].
__global__ void __launch_bounds__(kThreads, 1)
    absorb_tc_kernel(const __grid_constant__ CUtensorMap map_w, const __grid_constant__ CUtensorMap map_x,
                     const __grid_constant__ ProjParams p, int rows8, int32_t* status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ uint64_t bars[2];
  __shared__ uint32_t tmem_slot;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int h = blockIdx.x;
  const int xbytes = rows8 * 128;
  uint8_t* sx = sm;
  uint8_t* sw = sm + ((2 * xbytes + 1023) & ~1023);
  if (tid == 0) {
    tc::mbar_init(&bars[0], 10);  // one arrival per issuing lane
    tc::mbar_init(&bars[1], 1);
    tc::fence_mbar_init();
  }
  if (warp == 0) tc::tmem_alloc(&tmem_slot, 512);
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tb = tmem_slot;
  // the whole slice in one round: one box per issuing lane, all in flight together
  if (tid < 8) {
    tc::mbar_expect_tx(&bars[0], kBox);
    tc::tma_load_3d(sw + tid * kBox, &map_w, 64 * tid, 0, h, &bars[0]);
  } else if (tid < 10) {
    tc::mbar_expect_tx(&bars[0], xbytes);
    tc::tma_load_3d(sx + (tid - 8) * xbytes, &map_x, 64 * (tid - 8), h, 0, &bars[0]);
  }
  // ---- q^R part, RoPE(q^R, pos[b]) into columns [512, 576): independent of the
  // MMA, so warps 1-3 do it while warp 0 waits for the weights (six rotations
  // per thread per round, their loads issued together)
  if (warp >= 1) {
    constexpr int kU = 6;
    const int n = p.batch * 32;
    for (int base = tid - 32; base < n; base += 96 * kU) {
      float x0[kU], x1[kU];
      int ps[kU];
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const int idx = base + u * 96;
        x0[u] = x1[u] = 0.f;
        ps[u] = 0;
        if (idx < n) {
          const int bb = idx >> 5, i = idx & 31;
          const __nv_bfloat16* src = p.q_r + ((int64_t)bb * p.n_heads + h) * 64 + 2 * i;
          x0[u] = __bfloat162float(src[0]);
          x1[u] = __bfloat162float(src[1]);
          ps[u] = p.pos[bb];
        }
      }
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const int idx = base + u * 96;
        if (idx < n) {
          const int bb = idx >> 5, i = idx & 31;
          float c, sn;
          rope_cos_sin(ps[u], p.rope.hi[i], p.rope.lo[i], &c, &sn);
          __nv_bfloat16* dst = p.out + (int64_t)bb * p.out_sb + (int64_t)h * p.out_sh + 512 + 2 * i;
          *reinterpret_cast<uint32_t*>(dst) = pack_bf16x2(x0[u] * c - x1[u] * sn, x0[u] * sn + x1[u] * c);
        }
      }
    }
  }
  bool ok = true;
  if (tid == 0) {
    ok = wait_done(&bars[0], 0);
    if (ok) {
      tc::tc_fence_after();
      constexpr uint32_t id = tc::idesc_bf16(128, 256, 0, 1);
      const uint32_t xa = smem_u32(sx), wa = smem_u32(sw);
#pragma unroll
      for (int nh = 0; nh < 2; ++nh)
#pragma unroll
        for (int ks = 0; ks < 8; ++ks)
          tc::mma_ss(tb + nh * 256, tc::smem_desc(xa + (ks >> 2) * xbytes + (ks & 3) * 32, 16, 1024),
                     tc::smem_desc(wa + nh * 4 * kBox + ks * 2048, kBox, 1024), id, ks > 0 ? 1u : 0u);
      tc::mma_commit(&bars[1]);
      ok = wait_done(&bars[1], 0);
    }
    if (!ok) report(status, MLA_ERR_DEVICE_TIMEOUT);
  }
  __syncthreads();
  tc::tc_fence_after();
  // ---- epilogue: thread = batch row; 512 accumulator columns -> bf16
  const int b = warp * 32 + lane;
  if (warp * 32 < p.batch) {
    const uint32_t lane_t = tb + ((uint32_t)(warp * 32) << 16);
    __nv_bfloat16* dst = p.out + (int64_t)b * p.out_sb + (int64_t)h * p.out_sh;
#pragma unroll 1
    for (int c = 0; c < 16; c += 2) {  // two loads per wait
      uint32_t r[2][32];
      tc::tmem_ld32(lane_t + c * 32, r[0]);
      tc::tmem_ld32(lane_t + (c + 1) * 32, r[1]);
      tc::tmem_wait_ld();
      if (b < p.batch) {
#pragma unroll
        for (int k = 0; k < 2; ++k) {
          uint4* d4 = reinterpret_cast<uint4*>(dst + (c + k) * 32);
#pragma unroll
          for (int i = 0; i < 4; ++i)
            d4[i] = make_uint4(pack_bf16x2(__uint_as_float(r[k][8 * i]), __uint_as_float(r[k][8 * i + 1])),
                               pack_bf16x2(__uint_as_float(r[k][8 * i + 2]), __uint_as_float(r[k][8 * i + 3])),
                               pack_bf16x2(__uint_as_float(r[k][8 * i + 4]), __uint_as_float(r[k][8 * i + 5])),
                               pack_bf16x2(__uint_as_float(r[k][8 * i + 6]), __uint_as_float(r[k][8 * i + 7])));
        }
      }
    }
  }
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tb, 512);
  }
}

// ---------------------------------------------------------------- out-projection
// smem: z boxes [8][rows8 x 128 B] at 0, then W^UV boxes [8][128 v x 128 B].
__global__ void __launch_bounds__(kThreads, 1)
    out_proj_tc_kernel(const __grid_constant__ CUtensorMap map_w, const __grid_constant__ CUtensorMap map_x,
                       const __grid_constant__ ProjParams p, int rows8, int32_t* status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ uint64_t bars[2];
  __shared__ uint32_t tmem_slot;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int h = blockIdx.x;
  const int xbytes = rows8 * 128;
  uint8_t* sx = sm;
  uint8_t* sw = sm + ((8 * xbytes + 1023) & ~1023);
  if (tid == 0) {
    tc::mbar_init(&bars[0], 16);  // one arrival per issuing lane
    tc::mbar_init(&bars[1], 1);
    tc::fence_mbar_init();
  }
  if (warp == 0) tc::tmem_alloc(&tmem_slot, 128);
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tb = tmem_slot;
  if (tid < 8) {
    tc::mbar_expect_tx(&bars[0], kBox);
    tc::tma_load_3d(sw + tid * kBox, &map_w, 64 * tid, 0, h, &bars[0]);
  } else if (tid < 16) {
    tc::mbar_expect_tx(&bars[0], xbytes);
    tc::tma_load_3d(sx + (tid - 8) * xbytes, &map_x, 64 * (tid - 8), h, 0, &bars[0]);
  }
  if (tid == 0) {
    bool ok = wait_done(&bars[0], 0);
    if (ok) {
      tc::tc_fence_after();
      constexpr uint32_t id = tc::idesc_bf16(128, 128, 0, 0);
      const uint32_t xa = smem_u32(sx), wa = smem_u32(sw);
#pragma unroll
      for (int ks = 0; ks < 32; ++ks)
        tc::mma_ss(tb, tc::smem_desc(xa + (ks >> 2) * xbytes + (ks & 3) * 32, 16, 1024),
                   tc::smem_desc(wa + (ks >> 2) * kBox + (ks & 3) * 32, 16, 1024), id, ks > 0 ? 1u : 0u);
      tc::mma_commit(&bars[1]);
      ok = wait_done(&bars[1], 0);
    }
    if (!ok) report(status, MLA_ERR_DEVICE_TIMEOUT);
  }
  __syncthreads();
  tc::tc_fence_after();
  const int b = warp * 32 + lane;
  if (warp * 32 < p.batch) {
    const uint32_t lane_t = tb + ((uint32_t)(warp * 32) << 16);
    __nv_bfloat16* dst = p.out + (int64_t)b * p.out_sb + (int64_t)h * p.out_sh;
#pragma unroll 1
    for (int c = 0; c < 4; ++c) {
      uint32_t r[32];
      tc::tmem_ld32(lane_t + c * 32, r);
      tc::tmem_wait_ld();
      if (b < p.batch) {
        uint4* d4 = reinterpret_cast<uint4*>(dst + c * 32);
#pragma unroll
        for (int i = 0; i < 4; ++i)
          d4[i] = make_uint4(pack_bf16x2(__uint_as_float(r[8 * i]), __uint_as_float(r[8 * i + 1])),
                             pack_bf16x2(__uint_as_float(r[8 * i + 2]), __uint_as_float(r[8 * i + 3])),
                             pack_bf16x2(__uint_as_float(r[8 * i + 4]), __uint_as_float(r[8 * i + 5])),
                             pack_bf16x2(__uint_as_float(r[8 * i + 6]), __uint_as_float(r[8 * i + 7])));
      }
    }
  }
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tb, 128);
  }
}


// ---------------------------------------------------------------- cache append
// [c; k^R] = [W^DKV; W^KR] h for the new tokens ("MLA 的核心结构": c^KV =
// W^DKV h; "RoPE 为什么要解耦": k^R = RoPE(W^KR h)), tokens as M.
// A cluster of kAppendSplit CTAs shares one 96-column slice of the 576 outputs,
// each CTA one 448-deep slice of d_model (7 boxes of 64): 6 x 16 = 96 CTAs
// stream the 8.3 MB weight once, all of it in flight at the same time, and
// keep their weight slice in shared memory for every token tile.  Tokens come
// in tiles of `rows` (up to 32 tokens: one tile of the count rounded up to 8;
// more: tiles of 128, the last one padded with zero rows by the TMA fill).
// Per tile, the fp32 partials are summed in rank order through distributed
// shared memory, each rank finishing 6 of the 96 columns: RoPE on the k^R
// pairs, bf16 rounding, and the write into the cache slot of (sequence,
// position).
constexpr int kAppendSplit = 16;
MLA_DEVI float ld_cluster_f32(uint32_t a) {
  float x;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(x) : "r"(a) : "memory");
  return x;
}
constexpr int kAppendN = 96;
constexpr int kAppendKBoxes = 7;
constexpr int kAppendBigRows = 128;

struct AppendParams {
  int n_tokens, d_model;
  const int32_t* seq_idx;
  const int32_t* pos;
  int n_seqs;
  const int32_t* block_table;
  int max_blocks, num_blocks, block_tokens;
  int64_t seq_stride;
  __nv_bfloat16* pool;
  RopeTurns rope;
  int32_t* status;
};

__global__ void __launch_bounds__(kThreads, 1)
    append_tc_kernel(const __grid_constant__ CUtensorMap map_w, const __grid_constant__ CUtensorMap map_h,
                     const __grid_constant__ AppendParams p, int rows) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ uint64_t bars[3];  // weight slice, token tile, MMAs done
  __shared__ uint32_t tmem_slot;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t rank = tc::cluster_rank();
  const int ntile = (int)(blockIdx.x / kAppendSplit);
  const int n0 = ntile * kAppendN;
  const int k0 = (int)rank * kAppendKBoxes * 64;
  const int hbytes = rows * 128;
  const int wbytes = kAppendN * 128;
  const int mtiles = (p.n_tokens + rows - 1) / rows;
  uint8_t* sh = sm;                                                    // [7][rows x 128 B]
  uint8_t* sw = sm + ((kAppendKBoxes * hbytes + 1023) & ~1023);        // [7][96 x 128 B]
  // once a tile's MMAs are done its token boxes hold this CTA's fp32 partial
  // tile, [column][token] (96 x rows floats fit in 7 x rows x 128 bytes)
  float* red = reinterpret_cast<float*>(sh);
  if (tid == 0) {
    tc::mbar_init(&bars[0], kAppendKBoxes);  // one arrival per issuing thread
    tc::mbar_init(&bars[1], kAppendKBoxes);
    tc::mbar_init(&bars[2], 1);
    tc::fence_mbar_init();
  }
  if (warp == 0) tc::tmem_alloc(&tmem_slot, 128);
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tb = tmem_slot;
  if (tid < kAppendKBoxes) {
    tc::mbar_expect_tx(&bars[0], wbytes);
    tc::tma_load_2d(sw + tid * wbytes, &map_w, k0 + 64 * tid, n0, &bars[0]);
  }
  constexpr int kCols = kAppendN / kAppendSplit;
  for (int mt = 0; mt < mtiles; ++mt) {
    if (tid < kAppendKBoxes) {
      tc::mbar_expect_tx(&bars[1], hbytes);
      tc::tma_load_2d(sh + tid * hbytes, &map_h, k0 + 64 * tid, mt * rows, &bars[1]);
    }
    if (tid == 0) {
      bool ok = (mt > 0 || wait_done(&bars[0], 0)) && wait_done(&bars[1], mt & 1);
      if (ok) {
        tc::tc_fence_after();
        constexpr uint32_t id = tc::idesc_bf16(128, kAppendN, 0, 0);
        const uint32_t ha = smem_u32(sh), wa = smem_u32(sw);
        // M = 128 token rows; with rows < 128 the rows past the tile read other
        // operands' bytes and their results are not used
#pragma unroll
        for (int ks = 0; ks < 4 * kAppendKBoxes; ++ks)
          tc::mma_ss(tb, tc::smem_desc(ha + (ks >> 2) * hbytes + (ks & 3) * 32, 16, 1024),
                     tc::smem_desc(wa + (ks >> 2) * wbytes + (ks & 3) * 32, 16, 1024), id, ks > 0 ? 1u : 0u);
        tc::mma_commit(&bars[2]);
        ok = wait_done(&bars[2], mt & 1);
      }
      if (!ok) report(p.status, MLA_ERR_DEVICE_TIMEOUT);
    }
    __syncthreads();
    tc::tc_fence_after();
    if (32 * warp < rows) {  // token rows 32 w .. 32 w + 31 live in TMEM lanes of warp w
      const int t = 32 * warp + lane;
      uint32_t r[32];
#pragma unroll
      for (int c = 0; c < kAppendN / 32; ++c) {
        tc::tmem_ld32(tb + ((uint32_t)(32 * warp) << 16) + c * 32, r);
        tc::tmem_wait_ld();
        if (t < rows)
#pragma unroll
          for (int i = 0; i < 32; ++i) red[(c * 32 + i) * rows + t] = __uint_as_float(r[i]);
      }
    }
    tc::tc_fence_before();
    __syncthreads();
    tc::cluster_sync();
    // rank r finishes columns [n0 + 6 r, n0 + 6 r + 6) of the tile's tokens: sum
    // the 16 partials in rank order, RoPE the k^R pairs, round, scatter into the cache
    const int nt = min(rows, p.n_tokens - mt * rows);
    for (int idx = tid; idx < nt * (kCols / 2); idx += kThreads) {
      const int t = idx / (kCols / 2), cp = idx % (kCols / 2);
      const int cl = (int)rank * kCols + 2 * cp;  // local column (even)
      float v0 = 0.f, v1 = 0.f;
#pragma unroll
      for (int q = 0; q < kAppendSplit; ++q) {
        v0 += ld_cluster_f32(tc::map_peer(&red[cl * rows + t], (uint32_t)q));
        v1 += ld_cluster_f32(tc::map_peer(&red[(cl + 1) * rows + t], (uint32_t)q));
      }
      const int n = n0 + cl;
      const int tok = mt * rows + t;
      const int s = p.seq_idx[tok], ps = p.pos[tok];
      bool ok = (s >= 0) && (s < p.n_seqs) && (ps >= 0);
      int64_t row = 0;
      if (ok) {
        if (p.block_table) {
          const int lb = ps / p.block_tokens;
          ok = lb < p.max_blocks;
          if (ok) {
            const int blk = p.block_table[(int64_t)s * p.max_blocks + lb];
            ok = (blk >= 0) && (blk < p.num_blocks);
            row = (int64_t)blk * p.block_tokens + ps % p.block_tokens;
          }
        } else {
          ok = ps < p.seq_stride;
          row = (int64_t)s * p.seq_stride + ps;
        }
      }
      if (!ok) {
        report(p.status, MLA_ERR_DEVICE_BOUNDS);
        continue;
      }
      if (n >= 512) {
        float c, sn;
        const int i = (n - 512) >> 1;
        rope_cos_sin(ps, p.rope.hi[i], p.rope.lo[i], &c, &sn);
        const float r0 = v0 * c - v1 * sn, r1 = v0 * sn + v1 * c;
        v0 = r0;
        v1 = r1;
      }
      *reinterpret_cast<uint32_t*>(p.pool + row * 576 + n) = pack_bf16x2(v0, v1);
    }
    tc::cluster_sync();  // peers keep their partials until every rank has read them
  }
  if (warp == 0) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tb, 128);
  }
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

// 3-D bf16 tensor map, 128-byte swizzle, box {64, box1, box2}.
bool make_map(CUtensorMap* m, const void* base, uint64_t d0, uint64_t d1, uint64_t d2, uint64_t s1_bytes,
              uint64_t s2_bytes, uint32_t box1, uint32_t box2) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  const cuuint64_t dims[3] = {d0, d1, d2};
  const cuuint64_t strides[2] = {s1_bytes, s2_bytes};
  const cuuint32_t box[3] = {64, box1, box2}, es[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2-D bf16 tensor map, 128-byte swizzle, box {64, box1}.
bool make_map2(CUtensorMap* m, const void* base, uint64_t d0, uint64_t d1, uint64_t s1_bytes, uint32_t box1) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  const cuuint64_t dims[2] = {d0, d1};
  const cuuint64_t strides[1] = {s1_bytes};
  const cuuint32_t box[2] = {64, box1}, es[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

int append_smem_bytes(int rows) {
  return ((kAppendKBoxes * rows * 128 + 1023) & ~1023) + kAppendKBoxes * kAppendN * 128 + 1024;
}
int append_rows(int n_tokens) { return n_tokens <= 32 ? (n_tokens + 7) & ~7 : kAppendBigRows; }

// True when a cluster of 16 CTAs of the append kernel with the shared memory
// of `rows`-token tiles can be resident on this device (a non-portable
// cluster size: it needs 16 free SMs in one GPC).  Decided once per device
// for each of the two tile sizes; also sets the kernel's attributes there.
bool append_cluster_fits(int rows) {
  static int fits_dev[64][2];  // 0 unknown, 1 no, 2 yes; [small tiles, 128-token tiles]
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
  std::lock_guard<std::mutex> lk(mu);
  const bool big = rows > 32;
  int& fits = fits_dev[dev][big ? 1 : 0];
  if (fits) return fits == 2;
  fits = 1;
  const int smem = append_smem_bytes(big ? kAppendBigRows : 32);
  if (cudaFuncSetAttribute(append_tc_kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess ||
      cudaFuncSetAttribute(append_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           append_smem_bytes(kAppendBigRows)) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((576 / kAppendN) * kAppendSplit);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kAppendSplit;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, append_tc_kernel, &cfg) != cudaSuccess) {
    cudaGetLastError();
    n = 0;
  }
  fits = n >= 1 ? 2 : 1;
  return fits == 2;
}

bool append_tc_supported(const mla_dims& d, int n_tokens, int d_model) {
  return d.d_latent == 512 && d.d_rope == 64 && n_tokens >= 1 && d_model == kAppendSplit * kAppendKBoxes * 64 &&
         append_cluster_fits(append_rows(n_tokens));
}

cudaError_t launch_append_tc(const mla_dims& d, int n_tokens, int d_model, const void* h, const void* w,
                             const int32_t* seq_idx, const int32_t* pos, int n_seqs, const int32_t* block_table,
                             int max_blocks, int num_blocks, int64_t seq_stride, void* pool, int32_t* status,
                             cudaStream_t s) {
  const int rows = append_rows(n_tokens);
  CUtensorMap mw, mh;
  if (!make_map2(&mw, w, (uint64_t)d_model, 576, (uint64_t)d_model * 2, kAppendN) ||
      !make_map2(&mh, h, (uint64_t)d_model, (uint64_t)n_tokens, (uint64_t)d_model * 2, rows))
    return cudaErrorInvalidValue;
  AppendParams p;
  p.n_tokens = n_tokens;
  p.d_model = d_model;
  p.seq_idx = seq_idx;
  p.pos = pos;
  p.n_seqs = n_seqs;
  p.block_table = block_table;
  p.max_blocks = max_blocks;
  p.num_blocks = num_blocks;
  p.block_tokens = d.block_tokens;
  p.seq_stride = seq_stride;
  p.pool = static_cast<__nv_bfloat16*>(pool);
  rope_turns_host(d.rope_base, 64, &p.rope);
  p.status = status;
  const int smem = append_smem_bytes(rows);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((576 / kAppendN) * kAppendSplit);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kAppendSplit;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, append_tc_kernel, mw, mh, p, rows);
}

bool proj_tc_supported(const mla_dims& d, int batch, bool absorb) {
  if (d.d_latent != 512 || batch < 1) return false;
  if (absorb) return d.d_head == 128 && d.d_rope == 64 && batch <= 128;
  return d.d_v == 128 && batch <= 64;
}

cudaError_t launch_absorb_tc(const mla_dims& d, int batch, const void* q_c, const void* q_r, const int32_t* pos,
                             const void* w_uk, void* q_out, int32_t* status, cudaStream_t s) {
  const int rows8 = (batch + 7) & ~7;
  CUtensorMap mw, mx;
  // W^UK [h][k][n]: dims {n 512, k 128, h}
  if (!make_map(&mw, w_uk, 512, 128, (uint64_t)d.n_heads, 512 * 2, (uint64_t)128 * 512 * 2, 128, 1) ||
      // q^C [b][h][k]: dims {k 128, h, b}
      !make_map(&mx, q_c, 128, (uint64_t)d.n_heads, (uint64_t)batch, 128 * 2, (uint64_t)d.n_heads * 128 * 2, 1,
                rows8))
    return cudaErrorInvalidValue;
  ProjParams p;
  p.batch = batch;
  p.n_heads = d.n_heads;
  p.out = static_cast<__nv_bfloat16*>(q_out);
  p.out_sb = (int64_t)d.n_heads * 576;
  p.out_sh = 576;
  p.q_r = static_cast<const __nv_bfloat16*>(q_r);
  p.pos = pos;
  rope_turns_host(d.rope_base, 64, &p.rope);
  const int smem = ((2 * rows8 * 128 + 1023) & ~1023) + 8 * kBox + 1024;
  cudaError_t e = ensure_smem<absorb_tc_kernel>(smem);
  if (e != cudaSuccess) return e;
  absorb_tc_kernel<<<d.n_heads, kThreads, smem, s>>>(mw, mx, p, rows8, status);
  return cudaGetLastError();
}

cudaError_t launch_out_proj_tc(const mla_dims& d, int batch, const void* z, const void* w_uv, void* o_out,
                               int32_t* status, cudaStream_t s) {
  const int rows8 = (batch + 7) & ~7;
  CUtensorMap mw, mx;
  // W^UV [h][v][c]: dims {c 512, v 128, h}
  if (!make_map(&mw, w_uv, 512, 128, (uint64_t)d.n_heads, 512 * 2, (uint64_t)128 * 512 * 2, 128, 1) ||
      // z [b][h][c]: dims {c 512, h, b}
      !make_map(&mx, z, 512, (uint64_t)d.n_heads, (uint64_t)batch, 512 * 2, (uint64_t)d.n_heads * 512 * 2, 1,
                rows8))
    return cudaErrorInvalidValue;
  ProjParams p = {};
  p.batch = batch;
  p.n_heads = d.n_heads;
  p.out = static_cast<__nv_bfloat16*>(o_out);
  p.out_sb = (int64_t)d.n_heads * 128;
  p.out_sh = 128;
  const int smem = ((8 * rows8 * 128 + 1023) & ~1023) + 8 * kBox + 1024;
  cudaError_t e = ensure_smem<out_proj_tc_kernel>(smem);
  if (e != cudaSuccess) return e;
  out_proj_tc_kernel<<<d.n_heads, kThreads, smem, s>>>(mw, mx, p, rows8, status);
  return cudaGetLastError();
}

}  // namespace mla

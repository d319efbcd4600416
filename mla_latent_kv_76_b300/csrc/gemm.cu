// Small batched GEMMs around decode: query absorption (q^C W^UK, plus RoPE on
// q^R), the value up-projection (W^UV z) and the cache-append projection
// ([W^DKV; W^KR] h, RoPE on the k^R part, scatter into the paged cache).
//
// All three are Y[g][m][n] = sum_k X[g][m][k] * W[g](k, n) with a small M
// (batch or new tokens) and a weight matrix read once; bf16 tensor-core
// mma.sync tiles (64 n x 32 k per stage, cp.async double buffering) with
// an fp32 accumulator and a per-use epilogue.
#include "common.cuh"
#include "kernels.h"

namespace mla {

enum class WLayout { KN, NK };  // KN: W[g][k][n] (n contiguous); NK: W[g][n][k] (k contiguous)
enum class Epi { ABSORB, OUT, APPEND };

struct GemmArgs {
  int M, N, K;
  const __nv_bfloat16* X;
  int64_t x_sm, x_sg;  // X + g*x_sg + m*x_sm + k
  const __nv_bfloat16* W;
  int64_t w_sr, w_sg;  // KN: W + g*w_sg + k*w_sr + n ; NK: W + g*w_sg + n*w_sr + k
  __nv_bfloat16* Y;
  int64_t y_sm, y_sg;  // Y + g*y_sg + m*y_sm + n
  // absorb: RoPE of q^R into Y[.., N : N + d_rope]
  const __nv_bfloat16* q_r;
  const int32_t* pos;
  int n_heads, d_rope, d_latent;
  float rope_base;
  // append
  const int32_t* seq_idx;
  int n_seqs;
  const int32_t* block_table;
  int max_blocks, num_blocks, block_tokens;
  int64_t seq_stride;
  int32_t* status;
};

constexpr int kBN = 64, kBK = 32;
constexpr int kARow = kBK * 2 + 16;   // 80 B: 5 chunks (odd) per staged row
constexpr int kWRowNK = kBK * 2 + 16; // [BN][BK]
constexpr int kWRowKN = kBN * 2 + 16; // [BK][BN], 144 B: 9 chunks

template <int BM, WLayout WL, Epi EP>
__global__ void __launch_bounds__(128) gemm_kernel(const GemmArgs a) {
  constexpr int W_BYTES = (WL == WLayout::NK) ? kBN * kWRowNK : kBK * kWRowKN;
  __shared__ __align__(16) uint8_t sA[2][BM * kARow];
  __shared__ __align__(16) uint8_t sW[2][W_BYTES];
  __shared__ double s_theta[64];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = blockIdx.z, m0 = blockIdx.y * BM, n0 = blockIdx.x * kBN;
  const __nv_bfloat16* X = a.X + g * a.x_sg;
  const __nv_bfloat16* W = a.W + g * a.w_sg;

  float acc[BM / 16][2][4];
#pragma unroll
  for (int i = 0; i < BM / 16; ++i)
#pragma unroll
    for (int j = 0; j < 2; ++j)
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[i][j][e] = 0.f;

  auto load = [&](int stage, int kt) {
    const int k0 = kt * kBK;
    for (int c = tid; c < BM * 4; c += 128) {
      const int r = c >> 2, ch = c & 3, m = m0 + r, k = k0 + ch * 8;
      const bool ok = (m < a.M) && (k < a.K);
      cp_async16(sA[stage] + r * kARow + ch * 16, ok ? X + m * a.x_sm + k : a.X, ok);
    }
    if (WL == WLayout::NK) {
      for (int c = tid; c < kBN * 4; c += 128) {
        const int r = c >> 2, ch = c & 3, n = n0 + r, k = k0 + ch * 8;
        const bool ok = (n < a.N) && (k < a.K);
        cp_async16(sW[stage] + r * kWRowNK + ch * 16, ok ? W + n * a.w_sr + k : a.W, ok);
      }
    } else {
      for (int c = tid; c < kBK * 8; c += 128) {
        const int r = c >> 3, ch = c & 7, k = k0 + r, n = n0 + ch * 8;
        const bool ok = (k < a.K) && (n < a.N);
        cp_async16(sW[stage] + r * kWRowKN + ch * 16, ok ? W + k * a.w_sr + n : a.W, ok);
      }
    }
  };

  const int ktiles = (a.K + kBK - 1) / kBK;
  load(0, 0);
  cp_async_commit();
  for (int kt = 0; kt < ktiles; ++kt) {
    if (kt + 1 < ktiles) {
      load((kt + 1) & 1, kt + 1);
      cp_async_commit();
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();
    const uint8_t* A = sA[kt & 1];
    const uint8_t* Ws = sW[kt & 1];
#pragma unroll
    for (int kk = 0; kk < kBK / 16; ++kk) {
      uint32_t b[4];
      if (WL == WLayout::NK) {
        ldsm_x4(b, Ws + (warp * 16 + (lane & 7) + (lane >> 4) * 8) * kWRowNK +
                       (kk * 16 + ((lane >> 3) & 1) * 8) * 2);
      } else {
        ldsm_x4_t(b, Ws + (kk * 16 + (lane & 7) + ((lane >> 3) & 1) * 8) * kWRowKN +
                         (warp * 16 + (lane >> 4) * 8) * 2);
      }
#pragma unroll
      for (int mb = 0; mb < BM / 16; ++mb) {
        uint32_t af[4];
        ldsm_x4(af, A + (mb * 16 + (lane & 15)) * kARow + (kk * 16 + (lane >> 4) * 8) * 2);
        mma_bf16(acc[mb][0], af, b[0], b[1]);
        mma_bf16(acc[mb][1], af, b[2], b[3]);
      }
    }
    __syncthreads();
  }

  // ------------------------------------------------------------ epilogue
  if (EP == Epi::APPEND) {
    // RoPE frequencies, once per CTA, in fp64
    for (int i = tid; i < a.d_rope / 2 && i < 64; i += 128)
      s_theta[i] = pow((double)a.rope_base, -2.0 * (double)i / (double)a.d_rope);
    __syncthreads();
  }
#pragma unroll
  for (int mb = 0; mb < BM / 16; ++mb) {
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      const int m = m0 + mb * 16 + (lane >> 2) + half * 8;
      if (m >= a.M) continue;
      __nv_bfloat16* dst_row = nullptr;
      int p = 0;
      if (EP == Epi::APPEND) {
        const int s = a.seq_idx[m];
        p = a.pos[m];
        bool ok = (s >= 0) && (s < a.n_seqs) && (p >= 0);
        int64_t row = 0;
        if (ok) {
          if (a.block_table) {
            const int lb = p / a.block_tokens;
            ok = lb < a.max_blocks;
            if (ok) {
              const int blk = a.block_table[(int64_t)s * a.max_blocks + lb];
              ok = (blk >= 0) && (blk < a.num_blocks);
              row = (int64_t)blk * a.block_tokens + p % a.block_tokens;
            }
          } else {
            ok = p < a.seq_stride;
            row = (int64_t)s * a.seq_stride + p;
          }
        }
        if (!ok) {
          report(a.status, MLA_ERR_DEVICE_BOUNDS);
          continue;
        }
        dst_row = a.Y + row * a.y_sm;
      } else {
        dst_row = a.Y + g * a.y_sg + m * a.y_sm;
      }
#pragma unroll
      for (int nb = 0; nb < 2; ++nb) {
        const int n = n0 + warp * 16 + nb * 8 + (lane & 3) * 2;
        if (n >= a.N) continue;
        float v0 = acc[mb][nb][half * 2 + 0], v1 = acc[mb][nb][half * 2 + 1];
        if (EP == Epi::APPEND && n >= a.d_latent) {
          const int i = (n - a.d_latent) >> 1;
          float c, sn;
          rope_cos_sin_theta(p, s_theta[i], &c, &sn);
          const float r0 = v0 * c - v1 * sn, r1 = v0 * sn + v1 * c;
          v0 = r0;
          v1 = r1;
        }
        *reinterpret_cast<uint32_t*>(dst_row + n) = pack_bf16x2(v0, v1);
      }
    }
  }

  if (EP == Epi::ABSORB && blockIdx.x == 0) {
    // q^R part of the latent query: RoPE(q^R, pos[b]) into columns [d_c, d_c + d_R)
    const int half_r = a.d_rope / 2;
    for (int i = tid; i < half_r && i < 64; i += 128)
      s_theta[i] = pow((double)a.rope_base, -2.0 * (double)i / (double)a.d_rope);
    __syncthreads();
    for (int idx = tid; idx < BM * half_r; idx += 128) {
      const int m = m0 + idx / half_r, i = idx % half_r;
      if (m >= a.M) continue;
      const __nv_bfloat16* src = a.q_r + ((int64_t)m * a.n_heads + g) * a.d_rope + 2 * i;
      const float x0 = __bfloat162float(src[0]), x1 = __bfloat162float(src[1]);
      float c, sn;
      rope_cos_sin_theta(a.pos[m], s_theta[i], &c, &sn);
      __nv_bfloat16* dst = a.Y + g * a.y_sg + m * a.y_sm + a.d_latent + 2 * i;
      *reinterpret_cast<uint32_t*>(dst) = pack_bf16x2(x0 * c - x1 * sn, x0 * sn + x1 * c);
    }
  }
}

template <int BM, WLayout WL, Epi EP>
static cudaError_t run(const GemmArgs& a, int groups, cudaStream_t s) {
  dim3 grid((a.N + kBN - 1) / kBN, (a.M + BM - 1) / BM, groups);
  gemm_kernel<BM, WL, EP><<<grid, 128, 0, s>>>(a);
  return cudaGetLastError();
}

template <WLayout WL, Epi EP>
static cudaError_t run_bm(const GemmArgs& a, int groups, cudaStream_t s) {
  if (a.M <= 16) return run<16, WL, EP>(a, groups, s);
  if (a.M <= 32) return run<32, WL, EP>(a, groups, s);
  return run<64, WL, EP>(a, groups, s);
}

cudaError_t launch_absorb(const mla_dims& d, int batch, const void* q_c, const void* q_r,
                          const int32_t* pos, const void* w_uk, void* q_out, cudaStream_t s) {
  GemmArgs a = {};
  const int D = d.d_latent + d.d_rope;
  a.M = batch;
  a.N = d.d_latent;
  a.K = d.d_head;
  a.X = static_cast<const __nv_bfloat16*>(q_c);
  a.x_sm = (int64_t)d.n_heads * d.d_head;
  a.x_sg = d.d_head;
  a.W = static_cast<const __nv_bfloat16*>(w_uk);
  a.w_sr = d.d_latent;
  a.w_sg = (int64_t)d.d_head * d.d_latent;
  a.Y = static_cast<__nv_bfloat16*>(q_out);
  a.y_sm = (int64_t)d.n_heads * D;
  a.y_sg = D;
  a.q_r = static_cast<const __nv_bfloat16*>(q_r);
  a.pos = pos;
  a.n_heads = d.n_heads;
  a.d_rope = d.d_rope;
  a.d_latent = d.d_latent;
  a.rope_base = d.rope_base;
  return run_bm<WLayout::KN, Epi::ABSORB>(a, d.n_heads, s);
}

cudaError_t launch_out_proj(const mla_dims& d, int batch, const void* z, const void* w_uv,
                            void* o_out, cudaStream_t s) {
  GemmArgs a = {};
  a.M = batch;
  a.N = d.d_v;
  a.K = d.d_latent;
  a.X = static_cast<const __nv_bfloat16*>(z);
  a.x_sm = (int64_t)d.n_heads * d.d_latent;
  a.x_sg = d.d_latent;
  a.W = static_cast<const __nv_bfloat16*>(w_uv);
  a.w_sr = d.d_latent;
  a.w_sg = (int64_t)d.d_v * d.d_latent;
  a.Y = static_cast<__nv_bfloat16*>(o_out);
  a.y_sm = (int64_t)d.n_heads * d.d_v;
  a.y_sg = d.d_v;
  return run_bm<WLayout::NK, Epi::OUT>(a, d.n_heads, s);
}

cudaError_t launch_append(const mla_dims& d, int n_tokens, int d_model, const void* h,
                          const void* w, const int32_t* seq_idx, const int32_t* pos, int n_seqs,
                          const int32_t* block_table, int max_blocks, int num_blocks,
                          int64_t seq_stride, void* pool, int32_t* status, cudaStream_t s) {
  GemmArgs a = {};
  const int D = d.d_latent + d.d_rope;
  a.M = n_tokens;
  a.N = D;
  a.K = d_model;
  a.X = static_cast<const __nv_bfloat16*>(h);
  a.x_sm = d_model;
  a.x_sg = 0;
  a.W = static_cast<const __nv_bfloat16*>(w);
  a.w_sr = d_model;
  a.w_sg = 0;
  a.Y = static_cast<__nv_bfloat16*>(pool);
  a.y_sm = D;
  a.y_sg = 0;
  a.pos = pos;
  a.d_rope = d.d_rope;
  a.d_latent = d.d_latent;
  a.rope_base = d.rope_base;
  a.seq_idx = seq_idx;
  a.n_seqs = n_seqs;
  a.block_table = block_table;
  a.max_blocks = max_blocks;
  a.num_blocks = num_blocks;
  a.block_tokens = d.block_tokens;
  a.seq_stride = seq_stride;
  a.status = status;
  return run_bm<WLayout::NK, Epi::APPEND>(a, 1, s);
}

}  // namespace mla

// Weight-streaming GEMMs around decode: query absorption (q^C W^UK, plus
// RoPE on q^R), the value up-projection (W^UV z) and the cache-append
// projection ([W^DKV; W^KR] h, RoPE on the k^R part, scatter into the cache).
//
// All three are Y[g][m][n] = sum_k X[g][m][k] W[g](k, n) with a small M (the
// batch, or the new tokens) and a weight matrix that is read exactly once, so
// they are bound by HBM bandwidth, not by arithmetic.  What matters is the
// number of weight bytes in flight: every CTA issues all (or most) of its
// weight tile as 16-byte cp.async copies up front, in a multi-stage ring of
// BK-wide K chunks.  The arithmetic is bf16 mma.sync with fp32 accumulation
// (M is 16..64: a tensor-memory MMA would not shorten an HBM-bound kernel).
//
// A long K (the append's d_model = 7168) is split across a cluster of up to 8
// CTAs along grid x; their fp32 partial tiles are summed in rank order by
// rank 0 through distributed shared memory (deterministic), which then runs
// the epilogue.
#include "common.cuh"
#include "kernels.h"
#include "tc.cuh"

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
  int ksplit;          // CTAs of a cluster along x sharing one output tile
  // absorb: RoPE of q^R into Y[.., N : N + d_rope]
  const __nv_bfloat16* q_r;
  const int32_t* pos;
  int n_heads, d_rope, d_latent;
  RopeTurns rope;
  // append
  const int32_t* seq_idx;
  int n_seqs;
  const int32_t* block_table;
  int max_blocks, num_blocks, block_tokens;
  int64_t seq_stride;
  int32_t* status;
};

MLA_DEVI void ldsm_x2(uint32_t (&r)[2], const void* smem) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0,%1}, [%2];\n"
               : "=r"(r[0]), "=r"(r[1])
               : "r"(smem_u32(smem)));
}

template <int BM, int BN, int BK, int STAGES, WLayout WL>
struct GemmCfg {
  static constexpr int RA = BK * 2 + 16;                                   // staged X row (odd # of 16 B)
  static constexpr int RW = (WL == WLayout::NK) ? BK * 2 + 16 : BN * 2 + 16;
  static constexpr int WROWS = (WL == WLayout::NK) ? BN : BK;
  static constexpr int A_BYTES = BM * RA;
  static constexpr int STAGE = A_BYTES + WROWS * RW;
  static constexpr int CROW = BN + 4;                                      // fp32 result tile row
  static constexpr int C_BYTES = BM * CROW * 4;
  static constexpr int SMEM = (STAGES * STAGE > C_BYTES ? STAGES * STAGE : C_BYTES);
};

template <int BM, int BN, int BK, int STAGES, WLayout WL, Epi EP>
__global__ void __launch_bounds__(128) sgemm_kernel(const __grid_constant__ GemmArgs a) {
  using C = GemmCfg<BM, BN, BK, STAGES, WL>;
  constexpr int WN = BN / 4;  // output columns per warp
  constexpr int NB = WN / 8;  // n8 blocks per warp
  static_assert(WN % 8 == 0, "BN must be a multiple of 32");
  extern __shared__ __align__(16) uint8_t smem[];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int ks = a.ksplit;
  const int kr = (int)(blockIdx.x % ks);
  const int n0 = (int)(blockIdx.x / ks) * BN, m0 = blockIdx.y * BM, g = blockIdx.z;
  const __nv_bfloat16* X = a.X + g * a.x_sg;
  const __nv_bfloat16* W = a.W + g * a.w_sg;

  // this CTA's K range
  const int kc = ((a.K + ks - 1) / ks + BK - 1) / BK * BK;
  const int kbeg = kr * kc;
  const int kend = min(a.K, kbeg + kc);
  const int nk = kend > kbeg ? (kend - kbeg + BK - 1) / BK : 0;

  float acc[BM / 16][NB][4];
#pragma unroll
  for (int i = 0; i < BM / 16; ++i)
#pragma unroll
    for (int j = 0; j < NB; ++j)
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[i][j][e] = 0.f;

  auto load = [&](int slot, int kt) {
    uint8_t* sA = smem + slot * C::STAGE;
    uint8_t* sW = sA + C::A_BYTES;
    const int k0 = kbeg + kt * BK;
    for (int c = tid; c < BM * (BK / 8); c += 128) {
      const int r = c / (BK / 8), ch = c % (BK / 8), m = m0 + r, k = k0 + ch * 8;
      const bool ok = (m < a.M) && (k < kend);
      cp_async16(sA + r * C::RA + ch * 16, ok ? X + m * a.x_sm + k : a.X, ok);
    }
    if (WL == WLayout::NK) {
      for (int c = tid; c < BN * (BK / 8); c += 128) {
        const int r = c / (BK / 8), ch = c % (BK / 8), n = n0 + r, k = k0 + ch * 8;
        const bool ok = (n < a.N) && (k < kend);
        cp_async16(sW + r * C::RW + ch * 16, ok ? W + n * a.w_sr + k : a.W, ok);
      }
    } else {
      for (int c = tid; c < BK * (BN / 8); c += 128) {
        const int r = c / (BN / 8), ch = c % (BN / 8), k = k0 + r, n = n0 + ch * 8;
        const bool ok = (k < kend) && (n < a.N);
        cp_async16(sW + r * C::RW + ch * 16, ok ? W + k * a.w_sr + n : a.W, ok);
      }
    }
  };

  auto compute = [&](int slot) {
    const uint8_t* sA = smem + slot * C::STAGE;
    const uint8_t* sW = sA + C::A_BYTES;
#pragma unroll
    for (int kk = 0; kk < BK / 16; ++kk) {
      uint32_t bf[NB][2];
      if (WL == WLayout::NK) {
#pragma unroll
        for (int nb = 0; nb < NB; ++nb) {
          uint32_t r2[2];
          ldsm_x2(r2, sW + (warp * WN + nb * 8 + (lane & 7)) * C::RW + (kk * 16 + ((lane >> 3) & 1) * 8) * 2);
          bf[nb][0] = r2[0];
          bf[nb][1] = r2[1];
        }
      } else {
#pragma unroll
        for (int nb = 0; nb < NB; nb += 2) {
          uint32_t r4[4];
          ldsm_x4_t(r4, sW + (kk * 16 + (lane & 7) + ((lane >> 3) & 1) * 8) * C::RW +
                            (warp * WN + nb * 8 + (lane >> 4) * 8) * 2);
          bf[nb][0] = r4[0];
          bf[nb][1] = r4[1];
          bf[nb + 1][0] = r4[2];
          bf[nb + 1][1] = r4[3];
        }
      }
#pragma unroll
      for (int mb = 0; mb < BM / 16; ++mb) {
        uint32_t af[4];
        ldsm_x4(af, sA + (mb * 16 + (lane & 15)) * C::RA + (kk * 16 + (lane >> 4) * 8) * 2);
#pragma unroll
        for (int nb = 0; nb < NB; ++nb) mma_bf16(acc[mb][nb], af, bf[nb][0], bf[nb][1]);
      }
    }
  };

  if (nk <= STAGES) {
    // everything in flight at once
    for (int kt = 0; kt < nk; ++kt) load(kt, kt);
    cp_async_commit();
    cp_async_wait<0>();
    __syncthreads();
    for (int kt = 0; kt < nk; ++kt) compute(kt);
  } else {
#pragma unroll
    for (int kt = 0; kt < STAGES - 1; ++kt) {
      load(kt, kt);
      cp_async_commit();
    }
    for (int kt = 0; kt < nk; ++kt) {
      cp_async_wait<STAGES - 2>();
      __syncthreads();
      const int nxt = kt + STAGES - 1;
      if (nxt < nk) load(nxt % STAGES, nxt);
      cp_async_commit();
      compute(kt % STAGES);
    }
    cp_async_wait<0>();
  }
  __syncthreads();  // stages are reused as the fp32 result tile

  // ------------------------------------------------------------ partial tile -> shared memory
  float* Cs = reinterpret_cast<float*>(smem);
#pragma unroll
  for (int mb = 0; mb < BM / 16; ++mb)
#pragma unroll
    for (int nb = 0; nb < NB; ++nb)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int r = mb * 16 + (lane >> 2) + (e >> 1) * 8;
        const int c = warp * WN + nb * 8 + (lane & 3) * 2 + (e & 1);
        Cs[r * C::CROW + c] = acc[mb][nb][e];
      }
  if (ks > 1) {
    tc::cluster_sync();
    if (kr == 0) {
      for (int i = tid; i < BM * BN; i += 128) {
        const int r = i / BN, c = i % BN;
        float v = Cs[r * C::CROW + c];
        for (int q = 1; q < ks; ++q) {
          const uint32_t ra = tc::map_peer(&Cs[r * C::CROW + c], (uint32_t)q);
          float pv;
          asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(pv) : "r"(ra) : "memory");
          v += pv;
        }
        Cs[r * C::CROW + c] = v;
      }
    }
    tc::cluster_sync();  // peers keep their shared memory until rank 0 has read it
    if (kr != 0) return;
  } else {
    __syncthreads();
  }

  // ------------------------------------------------------------ epilogue
  for (int i = tid; i < BM * (BN / 2); i += 128) {
    const int r = i / (BN / 2), cp = i % (BN / 2);
    const int m = m0 + r, n = n0 + 2 * cp;
    if (m >= a.M || n >= a.N) continue;
    float v0 = Cs[r * C::CROW + 2 * cp], v1 = Cs[r * C::CROW + 2 * cp + 1];
    __nv_bfloat16* dst_row;
    if (EP == Epi::APPEND) {
      const int s = a.seq_idx[m];
      const int p = a.pos[m];
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
      if (n >= a.d_latent) {
        float c, sn;
        const int fi = (n - a.d_latent) >> 1;
        rope_cos_sin(p, a.rope.hi[fi], a.rope.lo[fi], &c, &sn);
        const float r0 = v0 * c - v1 * sn, r1 = v0 * sn + v1 * c;
        v0 = r0;
        v1 = r1;
      }
    } else {
      dst_row = a.Y + g * a.y_sg + m * a.y_sm;
    }
    *reinterpret_cast<uint32_t*>(dst_row + n) = pack_bf16x2(v0, v1);
  }

  if (EP == Epi::ABSORB && blockIdx.x == 0) {
    // q^R part of the latent query: RoPE(q^R, pos[b]) into columns [d_c, d_c + d_R)
    const int half_r = a.d_rope / 2;
    for (int idx = tid; idx < BM * half_r; idx += 128) {
      const int m = m0 + idx / half_r, i = idx % half_r;
      if (m >= a.M) continue;
      const __nv_bfloat16* src = a.q_r + ((int64_t)m * a.n_heads + g) * a.d_rope + 2 * i;
      const float x0 = __bfloat162float(src[0]), x1 = __bfloat162float(src[1]);
      float c, sn;
      rope_cos_sin(a.pos[m], a.rope.hi[i], a.rope.lo[i], &c, &sn);
      __nv_bfloat16* dst = a.Y + g * a.y_sg + m * a.y_sm + a.d_latent + 2 * i;
      *reinterpret_cast<uint32_t*>(dst) = pack_bf16x2(x0 * c - x1 * sn, x0 * sn + x1 * c);
    }
  }
}

template <int BM, int BN, int BK, int STAGES, WLayout WL, Epi EP>
static cudaError_t run(GemmArgs a, int groups, int ksplit, cudaStream_t s) {
  using C = GemmCfg<BM, BN, BK, STAGES, WL>;
  auto kern = sgemm_kernel<BM, BN, BK, STAGES, WL, EP>;
  cudaError_t e = ensure_smem<sgemm_kernel<BM, BN, BK, STAGES, WL, EP>>(C::SMEM);
  if (e != cudaSuccess) return e;
  a.ksplit = ksplit;
  const int ntiles = (a.N + BN - 1) / BN;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(ntiles * ksplit, (a.M + BM - 1) / BM, groups);
  cfg.blockDim = dim3(128);
  cfg.dynamicSmemBytes = C::SMEM;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = ksplit;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, a);
}

cudaError_t launch_absorb(const mla_dims& d, int batch, const void* q_c, const void* q_r,
                          const int32_t* pos, const void* w_uk, void* q_out, cudaStream_t s) {
  if (proj_tc_supported(d, batch, true)) return launch_absorb_tc(d, batch, q_c, q_r, pos, w_uk, q_out, nullptr, s);
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
  rope_turns_host(d.rope_base, d.d_rope, &a.rope);
  // K = d_h is short: one CTA per (head, 128 latent columns) holds all of its weight tile
  if (batch <= 16) return run<16, 128, 64, 2, WLayout::KN, Epi::ABSORB>(a, d.n_heads, 1, s);
  if (batch <= 32) return run<32, 128, 64, 2, WLayout::KN, Epi::ABSORB>(a, d.n_heads, 1, s);
  return run<64, 128, 64, 2, WLayout::KN, Epi::ABSORB>(a, d.n_heads, 1, s);
}

cudaError_t launch_out_proj(const mla_dims& d, int batch, const void* z, const void* w_uv,
                            void* o_out, cudaStream_t s) {
  if (proj_tc_supported(d, batch, false)) return launch_out_proj_tc(d, batch, z, w_uv, o_out, nullptr, s);
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
  // one CTA per (head, 32 output columns) streams a 32 x d_c weight slice
  if (batch <= 16) return run<16, 32, 128, 4, WLayout::NK, Epi::OUT>(a, d.n_heads, 1, s);
  if (batch <= 32) return run<32, 32, 128, 4, WLayout::NK, Epi::OUT>(a, d.n_heads, 1, s);
  return run<64, 32, 128, 4, WLayout::NK, Epi::OUT>(a, d.n_heads, 1, s);
}

cudaError_t launch_append(const mla_dims& d, int n_tokens, int d_model, const void* h,
                          const void* w, const int32_t* seq_idx, const int32_t* pos, int n_seqs,
                          const int32_t* block_table, int max_blocks, int num_blocks,
                          int64_t seq_stride, void* pool, int32_t* status, cudaStream_t s) {
  if (append_tc_supported(d, n_tokens, d_model))
    return launch_append_tc(d, n_tokens, d_model, h, w, seq_idx, pos, n_seqs, block_table, max_blocks, num_blocks,
                            seq_stride, pool, status, s);
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
  rope_turns_host(d.rope_base, d.d_rope, &a.rope);
  a.seq_idx = seq_idx;
  a.n_seqs = n_seqs;
  a.block_table = block_table;
  a.max_blocks = max_blocks;
  a.num_blocks = num_blocks;
  a.block_tokens = d.block_tokens;
  a.seq_stride = seq_stride;
  a.status = status;
  // split K over a cluster so that about one CTA per SM streams the weights,
  // with (for 16 tokens) the CTA's whole K slice in flight at once; every
  // cluster of the launch must be co-resident (about 15 clusters of 8 fit at
  // one ~126 KB CTA per SM, so larger tiles use clusters of at most 4)
  const int ntiles = (D + 31) / 32;
  auto split = [&](int bm, int bk, int kmax_cluster) {
    const int mt = (n_tokens + bm - 1) / bm;
    int ks = (148 + ntiles * mt - 1) / (ntiles * mt);
    const int kmax = (d_model + bk - 1) / bk;
    ks = ks < 1 ? 1 : (ks > kmax_cluster ? kmax_cluster : ks);
    return ks > kmax ? kmax : ks;
  };
  if (n_tokens <= 16) return run<16, 32, 128, 7, WLayout::NK, Epi::APPEND>(a, 1, split(16, 128, 8), s);
  if (n_tokens <= 32) return run<32, 32, 256, 4, WLayout::NK, Epi::APPEND>(a, 1, split(32, 256, 4), s);
  return run<64, 32, 128, 5, WLayout::NK, Epi::APPEND>(a, 1, split(64, 128, 4), s);
}

}  // namespace mla

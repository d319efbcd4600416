// Shape-generic split-KV decode in latent space on bf16 mma.sync tiles.
//
// One CTA = one split-KV worker x one group of 16 heads.  Per 64-token tile
// (staged with cp.async, double buffered):
//   S = Q[16 x D] . C[64 x D]^T                   (score, D = d_c + d_R)
//   online softmax over the tile (fp32, base 2)
//   O[16 x d_c] = alpha O + P[16 x 64] . C[64 x d_c]   (latent weighted sum)
// The score contracts the whole cache row, so q~.c and q^R.k^R are summed in
// the same accumulator ("结合 DeepSeek 推理代码看 MLA": score = (q^C W^UK).c^KV +
// q^R.k^R).  Rows past the sequence end are zero-filled in shared memory, so
// NaN garbage in block slack never reaches the MMA.  Each segment writes a
// normalised partial o and its lse; the combine kernel merges the partials.
#include "common.cuh"
#include "kernels.h"
#include "plan.cuh"

namespace mla {

constexpr int kHG = 16;          // heads per CTA (one m16 block)
constexpr int kMaxWarps = 8;     // warps per CTA: 8 for d_c >= 128, 4 for d_c = 64
constexpr int kPRow = 64 * 2 + 16;  // staged P row: 144 B (9 chunks)

struct GenericSmem {
  int row_bytes;   // staged cache / query row
  int off_q, off_kv0, off_kv1, off_p, off_red, off_prefix, total;
};

__host__ __device__ inline GenericSmem generic_smem(int D, int batch) {
  GenericSmem s;
  s.row_bytes = ldsm_row_bytes(D);
  s.off_q = 0;
  s.off_kv0 = s.off_q + kHG * s.row_bytes;
  s.off_kv1 = s.off_kv0 + kTileTokens * s.row_bytes;
  s.off_p = s.off_kv1 + kTileTokens * s.row_bytes;
  s.off_red = s.off_p + kHG * kPRow;
  s.off_prefix = s.off_red + 3 * kMaxWarps * kHG * 4;
  s.total = s.off_prefix + ((batch + 1) * 4 + 15) / 16 * 16;
  return s;
}

int generic_head_groups(int n_heads) { return (n_heads + kHG - 1) / kHG; }

MLA_DEVI void ldsm_x2_b(uint32_t (&r)[2], const void* smem_ptr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0,%1}, [%2];\n" : "=r"(r[0]), "=r"(r[1]) : "r"(smem_u32(smem_ptr)));
}

// NW warps: in the score each warp takes 64 / NW tokens of the tile, in the
// weighted sum DC / NW latent columns.  Eight warps halve the serial chain of
// mma.sync / ldmatrix / softmax steps each warp issues per tile (with four, a
// 16-head batch ran issue-bound at a third of DRAM peak).
template <int DC, int NW>
__global__ void __launch_bounds__(NW * 32) decode_generic_kernel(const DecodeLaunch a) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int D = DC + a.d_rope;
  const GenericSmem L = generic_smem(D, a.batch);
  const int RS = L.row_bytes;
  uint8_t* sQ = smem + L.off_q;
  uint8_t* sKV[2] = {smem + L.off_kv0, smem + L.off_kv1};
  uint8_t* sP = smem + L.off_p;
  float* sMax = reinterpret_cast<float*>(smem + L.off_red);  // [NW][16]
  float* sSum = sMax + NW * kHG;                               // [NW][16]
  float* sSumQ = sSum + NW * kHG;                              // [NW][16]
  constexpr int TPW = kTileTokens / NW;  // score tokens per warp
  constexpr int SB = TPW / 8;            // n8 blocks per warp in the score
  static_assert(SB == 1 || SB == 2, "4 or 8 warps");
  int* pre = reinterpret_cast<int*>(smem + L.off_prefix);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int gq = lane >> 2, tq = lane & 3;  // mma fragment row / column-pair index
  const int G = a.workers, wk = blockIdx.x, hg = blockIdx.y;
  const int64_t cap = a.block_table ? (int64_t)a.max_blocks * kTileTokens : a.seq_stride;
  const __nv_bfloat16* pool = static_cast<const __nv_bfloat16*>(a.pool);
  const __nv_bfloat16* qg = static_cast<const __nv_bfloat16*>(a.q);
  const float sl2 = a.scale * kLog2e;

  tile_prefix(a.seqlens, a.batch, cap, a.status, pre);
  const int64_t T = pre[a.batch];
  const int64_t lo = worker_begin(wk, T, G), hi = worker_begin(wk + 1, T, G);
  const int chunks = D / 8;

  for (int64_t x = lo; x < hi;) {
    // sequence owning tile x: largest b with pre[b] <= x
    int bl = 0, bh = a.batch - 1;
    while (bl < bh) {
      const int mid = (bl + bh + 1) >> 1;
      if (pre[mid] <= x) bl = mid; else bh = mid - 1;
    }
    const int b = bl;
    const int Lb = effective_len(a.seqlens, b, cap, nullptr);
    const int t_begin = (int)(x - pre[b]);
    const int64_t e1 = pre[b + 1];
    const int64_t seg_end = e1 < hi ? e1 : hi;
    const int ntile = (int)(seg_end - x);
    x = seg_end;

    __syncthreads();  // previous segment finished with sQ / sKV
    // query rows of this head group (rows past n_heads are zero)
    for (int c = tid; c < kHG * chunks; c += NW * 32) {
      const int r = c / chunks, ch = c % chunks, h = hg * kHG + r;
      const bool ok = h < a.n_heads;
      cp_async16(sQ + r * RS + ch * 16, ok ? qg + ((int64_t)b * a.n_heads + h) * D + ch * 8 : qg, ok);
    }
    auto load_tile = [&](int j, int buf) {
      const int tt = t_begin + j;
      const int t0 = tt * kTileTokens;
      const __nv_bfloat16* base = pool;
      bool blk_ok = true;
      if (a.block_table) {
        const int blk = a.block_table[(int64_t)b * a.max_blocks + tt];
        blk_ok = (blk >= 0) && (blk < a.num_blocks);
        if (!blk_ok) report(a.status, MLA_ERR_DEVICE_BOUNDS);
        else base = pool + (int64_t)blk * kTileTokens * D;
      } else {
        base = pool + ((int64_t)b * a.seq_stride + t0) * D;
      }
      for (int r = warp; r < kTileTokens; r += NW) {
        const bool ok = blk_ok && (t0 + r < Lb);
        for (int ch = lane; ch < chunks; ch += 32)
          cp_async16(sKV[buf] + r * RS + ch * 16, ok ? base + (int64_t)r * D + ch * 8 : pool, ok);
      }
    };
    load_tile(0, 0);
    cp_async_commit();

    float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f}, lq_run[2] = {0.f, 0.f};
    constexpr int NB = DC / (8 * NW);  // n8 blocks of the latent per warp
    static_assert(NB >= 2 && NB % 2 == 0, "value columns are loaded two n8 blocks at a time");
    float o[NB][4];
#pragma unroll
    for (int i = 0; i < NB; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;

    for (int j = 0; j < ntile; ++j) {
      const int buf = j & 1;
      if (j + 1 < ntile) {
        load_tile(j + 1, buf ^ 1);
        cp_async_commit();
        cp_async_wait<1>();
      } else {
        cp_async_wait<0>();
      }
      __syncthreads();
      const uint8_t* kv = sKV[buf];
      const int t0 = (t_begin + j) * kTileTokens;

      // ---- score: warp owns tokens [TPW warp, TPW warp + TPW) of the tile
      float s[SB][4];
#pragma unroll
      for (int nb = 0; nb < SB; ++nb) s[nb][0] = s[nb][1] = s[nb][2] = s[nb][3] = 0.f;
      const uint8_t* qa = sQ + (lane & 15) * RS + (lane >> 4) * 16;
      if (SB == 2) {
        const uint8_t* kb = kv + (warp * 16 + (lane & 7) + (lane >> 4) * 8) * RS + ((lane >> 3) & 1) * 16;
        for (int kk = 0; kk < D / 16; ++kk) {
          uint32_t af[4], bf[4];
          ldsm_x4(af, qa + kk * 32);
          ldsm_x4(bf, kb + kk * 32);
          mma_bf16(s[0], af, bf[0], bf[1]);
          mma_bf16(s[SB - 1], af, bf[2], bf[3]);
        }
      } else {
        const uint8_t* kb = kv + (warp * 8 + (lane & 7)) * RS + ((lane >> 3) & 1) * 16;
        for (int kk = 0; kk < D / 16; ++kk) {
          uint32_t af[4], bf[2];
          ldsm_x4(af, qa + kk * 32);
          ldsm_x2_b(bf, kb + kk * 32);
          mma_bf16(s[0], af, bf[0], bf[1]);
        }
      }
      // ---- scale, mask, tile row max
      float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
      for (int nb = 0; nb < SB; ++nb)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int tok = t0 + warp * TPW + nb * 8 + tq * 2 + (e & 1);
          const float v = (tok < Lb) ? s[nb][e] * sl2 : -INFINITY;
          s[nb][e] = v;
          mx[e >> 1] = fmaxf(mx[e >> 1], v);
        }
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 1));
        mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 2));
      }
      if (tq == 0) {
        sMax[warp * kHG + gq] = mx[0];
        sMax[warp * kHG + gq + 8] = mx[1];
      }
      __syncthreads();
      float alpha[2];
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        float tm = sMax[gq + 8 * r];
#pragma unroll
        for (int w = 1; w < NW; ++w) tm = fmaxf(tm, sMax[w * kHG + gq + 8 * r]);
        const float mn = fmaxf(m_run[r], tm);
        alpha[r] = exp2f(m_run[r] - mn);
        m_run[r] = mn;
        l_run[r] *= alpha[r];
        lq_run[r] *= alpha[r];
      }
      // ---- P = 2^(x - m), rounded to bf16 for the value MMA; l sums the fp32
      // weights (for lse), lq the rounded ones (it normalises o, so o is an exact
      // convex combination of the weights the MMA multiplied)
#pragma unroll
      for (int nb = 0; nb < SB; ++nb)
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          const float p0 = exp2f(s[nb][2 * r] - m_run[r]);
          const float p1 = exp2f(s[nb][2 * r + 1] - m_run[r]);
          const uint32_t pk = pack_bf16x2(p0, p1);
          l_run[r] += p0 + p1;
          lq_run[r] += __uint_as_float(pk << 16) + __uint_as_float(pk & 0xFFFF0000u);
          *reinterpret_cast<uint32_t*>(sP + (gq + 8 * r) * kPRow + (warp * TPW + nb * 8 + tq * 2) * 2) = pk;
        }
      __syncthreads();
      // ---- O = alpha O + P . C[:, warp's latent columns]
#pragma unroll
      for (int i = 0; i < NB; ++i) {
        o[i][0] *= alpha[0];
        o[i][1] *= alpha[0];
        o[i][2] *= alpha[1];
        o[i][3] *= alpha[1];
      }
      const int d_warp = warp * (DC / NW);
#pragma unroll
      for (int kk = 0; kk < kTileTokens / 16; ++kk) {
        uint32_t af[4];
        ldsm_x4(af, sP + (lane & 15) * kPRow + (kk * 16 + (lane >> 4) * 8) * 2);
        const uint8_t* vb = kv + (kk * 16 + (lane & 7) + ((lane >> 3) & 1) * 8) * RS + (d_warp + (lane >> 4) * 8) * 2;
#pragma unroll
        for (int nb2 = 0; nb2 < NB / 2; ++nb2) {
          uint32_t bf[4];
          ldsm_x4_t(bf, vb + nb2 * 32);
          mma_bf16(o[2 * nb2], af, bf[0], bf[1]);
          mma_bf16(o[2 * nb2 + 1], af, bf[2], bf[3]);
        }
      }
      __syncthreads();  // tile buffer and sP/sMax free for the next tile
    }

    // ---- segment result: o / l and lse, one partial slot per (worker, sequence)
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      l_run[r] += __shfl_xor_sync(0xffffffffu, l_run[r], 1);
      l_run[r] += __shfl_xor_sync(0xffffffffu, l_run[r], 2);
      lq_run[r] += __shfl_xor_sync(0xffffffffu, lq_run[r], 1);
      lq_run[r] += __shfl_xor_sync(0xffffffffu, lq_run[r], 2);
    }
    if (tq == 0) {
      sSum[warp * kHG + gq] = l_run[0];
      sSum[warp * kHG + gq + 8] = l_run[1];
      sSumQ[warp * kHG + gq] = lq_run[0];
      sSumQ[warp * kHG + gq + 8] = lq_run[1];
    }
    __syncthreads();
    const int64_t slot = (int64_t)wk + b;
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      const int h = hg * kHG + gq + 8 * r;
      float l = 0.f, lq = 0.f;
#pragma unroll
      for (int w = 0; w < NW; ++w) {
        l += sSum[w * kHG + gq + 8 * r];
        lq += sSumQ[w * kHG + gq + 8 * r];
      }
      if (h >= a.n_heads) continue;
      const float inv = 1.f / lq;
      float* op = a.o_part + (slot * a.n_heads + h) * DC + warp * (DC / NW) + tq * 2;
#pragma unroll
      for (int i = 0; i < NB; ++i)
        *reinterpret_cast<float2*>(op + i * 8) = make_float2(o[i][2 * r] * inv, o[i][2 * r + 1] * inv);
      if (warp == 0 && tq == 0) a.lse_part[slot * a.n_heads + h] = (m_run[r] + log2f(l)) * kLn2;
    }
  }
}

// ------------------------------------------------------------------ combine
// lse = log sum_s exp(lse_s);  z = sum_s exp(lse_s - lse) o_s   (one warp per head)
template <bool ZF32>
__global__ void __launch_bounds__(128) combine_kernel(const DecodeLaunch a) {
  const int b = blockIdx.y, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = blockIdx.x * 4 + warp;
  const int DC = a.d_latent, G = a.workers;
  const int64_t cap = a.block_table ? (int64_t)a.max_blocks * kTileTokens : a.seq_stride;

  // T (all tiles) and S_b (tiles before b): two block reductions
  long long before = 0, total = 0;
  for (int i = threadIdx.x; i < a.batch; i += blockDim.x) {
    const int t = tiles_of(effective_len(a.seqlens, i, cap, nullptr));
    total += t;
    if (i < b) before += t;
  }
  __shared__ long long red[2][4];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    before += __shfl_xor_sync(0xffffffffu, before, o);
    total += __shfl_xor_sync(0xffffffffu, total, o);
  }
  if (lane == 0) {
    red[0][warp] = before;
    red[1][warp] = total;
  }
  __syncthreads();
  const int64_t Sb = red[0][0] + red[0][1] + red[0][2] + red[0][3];
  const int64_t T = red[1][0] + red[1][1] + red[1][2] + red[1][3];
  if (h >= a.n_heads) return;
  const int nb = tiles_of(effective_len(a.seqlens, b, cap, nullptr));
  float* zf = static_cast<float*>(a.z_out) + ((int64_t)b * a.n_heads + h) * DC;
  __nv_bfloat16* zb = static_cast<__nv_bfloat16*>(a.z_out) + ((int64_t)b * a.n_heads + h) * DC;
  if (nb == 0) {
    for (int d = lane; d < DC; d += 32) {
      if (ZF32) zf[d] = 0.f; else zb[d] = __float2bfloat16_rn(0.f);
    }
    if (lane == 0 && a.lse_out) a.lse_out[(int64_t)b * a.n_heads + h] = -INFINITY;
    return;
  }
  const int g0 = worker_of(Sb, T, G), g1 = worker_of(Sb + nb - 1, T, G);
  auto live = [&](int g) {  // worker g's range meets sequence b's tiles
    return worker_begin(g, T, G) < Sb + nb && worker_begin(g + 1, T, G) > Sb &&
           worker_begin(g + 1, T, G) > worker_begin(g, T, G);
  };
  float mx = -INFINITY;
  for (int g = g0 + lane; g <= g1; g += 32)
    if (live(g)) mx = fmaxf(mx, a.lse_part[((int64_t)g + b) * a.n_heads + h]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  float sum = 0.f;
  for (int g = g0 + lane; g <= g1; g += 32)
    if (live(g)) sum += expf(a.lse_part[((int64_t)g + b) * a.n_heads + h] - mx);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
  const float lse = mx + logf(sum);
  for (int d = lane * 4; d < DC; d += 128) {
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int g = g0; g <= g1; ++g) {
      if (!live(g)) continue;
      const int64_t slot = (int64_t)g + b;
      const float w = expf(a.lse_part[slot * a.n_heads + h] - lse);
      const float4 v = *reinterpret_cast<const float4*>(a.o_part + (slot * a.n_heads + h) * DC + d);
      acc.x += w * v.x;
      acc.y += w * v.y;
      acc.z += w * v.z;
      acc.w += w * v.w;
    }
    if (ZF32) {
      *reinterpret_cast<float4*>(zf + d) = acc;
    } else {
      uint2 pk = make_uint2(pack_bf16x2(acc.x, acc.y), pack_bf16x2(acc.z, acc.w));
      *reinterpret_cast<uint2*>(zb + d) = pk;
    }
  }
  if (lane == 0 && a.lse_out) a.lse_out[(int64_t)b * a.n_heads + h] = lse;
}

template <int DC>
static cudaError_t launch_generic_dc(const DecodeLaunch& a, cudaStream_t s) {
  constexpr int NW = DC >= 128 ? 8 : 4;
  const GenericSmem L = generic_smem(DC + a.d_rope, a.batch);
  cudaError_t e = ensure_smem<decode_generic_kernel<DC, NW>>(L.total);
  if (e != cudaSuccess) return e;
  dim3 grid(a.workers, generic_head_groups(a.n_heads));
  decode_generic_kernel<DC, NW><<<grid, NW * 32, L.total, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_decode_generic(const DecodeLaunch& a, int, cudaStream_t s) {
  switch (a.d_latent) {
    case 64: return launch_generic_dc<64>(a, s);
    case 128: return launch_generic_dc<128>(a, s);
    case 256: return launch_generic_dc<256>(a, s);
    case 512: return launch_generic_dc<512>(a, s);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_combine(const DecodeLaunch& a, cudaStream_t s) {
  dim3 grid((a.n_heads + 3) / 4, a.batch);
  if (a.z_is_fp32) combine_kernel<true><<<grid, 128, 0, s>>>(a);
  else combine_kernel<false><<<grid, 128, 0, s>>>(a);
  return cudaGetLastError();
}

size_t generic_smem_bytes(int D, int batch) { return (size_t)generic_smem(D, batch).total; }

}  // namespace mla

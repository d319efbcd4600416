// Shared device helpers: cp.async staging, ldmatrix, bf16 mma.sync, RoPE angle.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <cmath>

#include "../../include/mla.h"

#define MLA_DEVI __device__ __forceinline__
#define MLA_HD __host__ __device__ __forceinline__  // plain integer helpers, also checked on the host

namespace mla {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// ---------------------------------------------------------------- status word
MLA_DEVI void report(int32_t* status, int code) {
  if (status) atomicCAS(reinterpret_cast<int*>(status), 0, code);
}

// ---------------------------------------------------------------- cp.async
MLA_DEVI uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// 16-byte async copy; when `full` is false the destination is zero-filled and
// nothing is read (the source pointer must still be a valid address).
MLA_DEVI void cp_async16(void* smem, const void* gmem, bool full) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(smem_u32(smem)), "l"(gmem),
               "r"(full ? 16 : 0));
}
MLA_DEVI void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::); }
template <int N>
MLA_DEVI void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N));
}

// ---------------------------------------------------------------- ldmatrix / mma
MLA_DEVI void ldsm_x4(uint32_t (&r)[4], const void* smem) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(smem_u32(smem)));
}
MLA_DEVI void ldsm_x4_t(uint32_t (&r)[4], const void* smem) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(smem_u32(smem)));
}

// D(16x8, fp32) += A(16x16, bf16, row) * B(16x8, bf16, col)
MLA_DEVI void mma_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

MLA_DEVI uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);  // round-to-nearest-even
  return *reinterpret_cast<uint32_t*>(&v);
}

// ---------------------------------------------------------------- RoPE
// Frequency i of the rotary embedding as turns per position,
// u_i = base^(-2i/d_R) / (2 pi), held as an fp32 pair hi + lo (about 48 bits).
// It is computed on the host in fp64: this part runs fp64 arithmetic at a tiny
// fraction of its fp32 rate (one device pow() cost ~4 us per CTA).
struct RopeTurns {
  float hi[64];
  float lo[64];
};

inline void rope_turns_host(float base, int d_rope, RopeTurns* t) {
  const double two_pi = 6.283185307179586476925286766559;
  for (int i = 0; i < 64; ++i) {
    const double u = (2 * i < d_rope) ? std::pow((double)base, -2.0 * i / d_rope) / two_pi : 0.0;
    t->hi[i] = (float)u;
    t->lo[i] = (float)(u - (double)t->hi[i]);
  }
}

// frac(x * (a_hi + a_lo)) for an integer-valued x < 2^24, in fp32: the product's
// rounding error is recovered exactly with an fma, and p - floor(p) is exact.
MLA_DEVI float turns_frac(float x, float a_hi, float a_lo) {
  const float p = x * a_hi;
  const float e = fmaf(x, a_hi, -p);
  const float f = p - floorf(p);
  const float g = f + fmaf(x, a_lo, e);
  return g - floorf(g);
}

// cos/sin of pos * theta_i.  The angle is reduced in turns (positions are split
// as pos = 4096 ph + pl so both factors are exact in fp32); the angle error stays
// below 1e-5 rad for every int32 position, far under a bf16 step, where a plain
// fp32 pos * theta would be off by ~1e-2 rad at pos ~ 1e5.
MLA_DEVI void rope_cos_sin(int pos, float u_hi, float u_lo, float* c, float* s) {
  const float ph = (float)(pos >> 12), pl = (float)(pos & 4095);
  float t = turns_frac(ph, u_hi * 4096.f, u_lo * 4096.f) + turns_frac(pl, u_hi, u_lo);
  t -= floorf(t);
  sincospif(2.f * t, s, c);
}

// Row stride in bytes for a bf16 row of `elems` values staged for ldmatrix:
// an odd number of 16-byte chunks keeps the 8 rows of one 8x8 matrix on
// distinct bank groups.
__host__ __device__ inline int ldsm_row_bytes(int elems) {
  int chunks = (elems * 2 + 15) / 16;
  if ((chunks & 1) == 0) chunks += 1;
  return chunks * 16;
}

}  // namespace mla

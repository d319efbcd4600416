// Shared device helpers: cp.async staging, ldmatrix, bf16 mma.sync, RoPE angle.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/mla.h"

#define MLA_DEVI __device__ __forceinline__

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
// cos/sin of pos * theta with theta = base^(-2i/d_R) given in fp64.  The
// angle is formed and reduced modulo 2*pi in fp64 (positions reach 1e5 and
// more, where an fp32 angle would be off by ~1e-2 rad), then evaluated with
// the fp32 sincosf on [0, 2*pi).
MLA_DEVI void rope_cos_sin_theta(int pos, double theta, float* c, float* s) {
  const double two_pi = 6.283185307179586476925286766559;
  const double inv_two_pi = 0.15915494309189533576888376337251;
  const double ang = (double)pos * theta;
  const double k = floor(ang * inv_two_pi);
  const double r = fma(-k, two_pi, ang);
  sincosf((float)r, s, c);
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

// Host-side launch wrappers shared by the C ABI (api.cu) and the kernel files.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <mutex>

#include "../../include/mla.h"

namespace mla {

// Raise a kernel's dynamic shared-memory limit to at least `bytes` on the
// current device.  Done once per (kernel, device) and size increase, so that
// steady-state launches make no host API call besides the launch itself.
// The slow path runs under a lock and only ever raises the limit, so host
// threads racing with different sizes cannot record a size above the one set.
template <auto Kernel>
cudaError_t ensure_smem(int bytes) {
  static std::atomic<int> set_bytes[64];
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return cudaErrorInvalidDevice;
  const bool cached = dev >= 0 && dev < 64;
  if (cached && bytes <= set_bytes[dev].load(std::memory_order_acquire)) return cudaSuccess;
  std::lock_guard<std::mutex> lk(mu);
  const int have = cached ? set_bytes[dev].load(std::memory_order_relaxed) : 0;
  if (bytes <= have) return cudaSuccess;
  const cudaError_t e = cudaFuncSetAttribute(Kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && cached) set_bytes[dev].store(bytes, std::memory_order_release);
  return e;
}

// Tokens per split-KV tile; equal to the paged block size so a tile never
// straddles two blocks.
constexpr int kTileTokens = 64;
constexpr int kMaxBatch = 4096;     // decode: per-CTA prefix table lives in shared memory
constexpr int kMaxWorkers = 4096;

struct DecodeLaunch {
  const void* q;
  const void* pool;
  const int32_t* block_table;
  int32_t max_blocks;
  int32_t num_blocks;
  int64_t seq_stride;
  const int32_t* seqlens;
  int32_t batch;
  int32_t n_heads;
  int32_t d_latent;
  int32_t d_rope;
  float scale;
  int32_t workers;        // G
  float* o_part;          // [(G + B)][n_h][d_c]
  float* lse_part;        // [(G + B)][n_h]  generic: lse; tensor-core: reference maximum (log2)
  float* l_part;          // [(G + B)][n_h]  tensor-core: fp32 weight sum relative to the maximum
  float* lq_part;         // [(G + B)][n_h]  tensor-core: bf16-rounded weight sum relative to the maximum
  int32_t* plan_flag;     // tensor-core: workspace header words [plan kind (1 = sequence-aligned), tiles, workers]
  int32_t* seqplan;       // tensor-core: [B][2] partials of sequence b: slots (aligned) or workers (even split) first..last
  void* z_out;
  int32_t z_is_fp32;
  float* lse_out;
  int32_t* status;
};

// Generic (mma.sync) decode partial pass + combine.
cudaError_t launch_decode_generic(const DecodeLaunch& a, int num_sms, cudaStream_t s);
cudaError_t launch_combine(const DecodeLaunch& a, cudaStream_t s);
int generic_head_groups(int n_heads);

// Tensor-core (tcgen05) decode for n_h = 128, d_c = 512, d_R = 64, partial pass
// and its combine: `workers` is the number of CTA pairs (clusters of two).
bool tc_supported(const DecodeLaunch& a);
// Tensor-core decode for 16 heads (d_c = 512, d_R = 64): one CTA per SM, the
// shape-generic partial layout and combine.
cudaError_t launch_decode_lh(const DecodeLaunch& a, cudaStream_t s);
bool lh_supported(const DecodeLaunch& a);

// Split-KV workers a decode call uses (num_workers, else the automatic count
// for its path on a device with `sms` SMs), and the workspace bytes it needs
// (0 for arguments mla_decode_attn rejects).
int decode_workers(const mla_dims& d, int batch, int num_workers, int flags, int sms);
size_t decode_workspace_bytes(const mla_dims* dims, int batch, int num_workers, int flags);
cudaError_t launch_decode_tc(const DecodeLaunch& a, cudaStream_t s);
size_t generic_smem_bytes(int D, int batch);

// Tensor-core absorb / out-projection for d_h = d_v = 128, d_c = 512, d_R = 64
// (absorb: batch <= 128, out-projection: batch <= 64).
bool proj_tc_supported(const mla_dims& d, int batch, bool absorb);
cudaError_t launch_absorb_tc(const mla_dims& d, int batch, const void* q_c, const void* q_r, const int32_t* pos,
                             const void* w_uk, void* q_out, int32_t* status, cudaStream_t s);
cudaError_t launch_out_proj_tc(const mla_dims& d, int batch, const void* z, const void* w_uv, void* o_out,
                               int32_t* status, cudaStream_t s);

// Tensor-core cache append for d_c = 512, d_R = 64, up to 32 tokens, d_model = 7168.
bool append_tc_supported(const mla_dims& d, int n_tokens, int d_model);
cudaError_t launch_append_tc(const mla_dims& d, int n_tokens, int d_model, const void* h, const void* w,
                             const int32_t* seq_idx, const int32_t* pos, int n_seqs, const int32_t* block_table,
                             int max_blocks, int num_blocks, int64_t seq_stride, void* pool, int32_t* status,
                             cudaStream_t s);

cudaError_t launch_absorb(const mla_dims& d, int batch, const void* q_c, const void* q_r,
                          const int32_t* pos, const void* w_uk, void* q_out, cudaStream_t s);
cudaError_t launch_out_proj(const mla_dims& d, int batch, const void* z, const void* w_uv,
                            void* o_out, cudaStream_t s);
cudaError_t launch_append(const mla_dims& d, int n_tokens, int d_model, const void* h,
                          const void* w, const int32_t* seq_idx, const int32_t* pos, int n_seqs,
                          const int32_t* block_table, int max_blocks, int num_blocks,
                          int64_t seq_stride, void* pool, int32_t* status, cudaStream_t s);

}  // namespace mla

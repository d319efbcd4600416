// mla_decode_attn_noalloc: decode for callers that cannot allocate device
// memory.  It runs the regular decode entry point with its workspace placed in
// a file-scope device array, so the caller passes only inputs and outputs.
#include "../../include/mla.h"
#include "kernels.h"

namespace {

// The split-KV partials live here.  Every GPU that loads the library holds
// this array until the process exits.
static __device__ __align__(256) unsigned char g_noalloc_scratch[MLA_NOALLOC_SCRATCH_BYTES];

// Device address of the array on the current device, looked up on every call
// (cheap), so that a context re-created after a device reset gets its own
// array rather than a stale address.  Host code must not use the array's name
// as an address: on the host it is only a stand-in symbol.
int scratch_address(void** out) {
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return MLA_ERR_CUDA;
  *out = p;
  return MLA_OK;
}

}  // namespace

extern "C" int mla_decode_attn_noalloc(const mla_dims* dims, int32_t batch, const void* q, const void* pool,
                                       const int32_t* block_table, int32_t max_blocks_per_seq,
                                       int32_t num_blocks, int64_t seq_stride_tokens, const int32_t* seqlens,
                                       float scale, int32_t num_workers, int32_t flags, void* z_out,
                                       int32_t z_is_fp32, float* lse_out, int32_t* dev_status, void* stream) {
  if (!dims || batch < 0) return MLA_ERR_INVALID_ARG;
  if (batch == 0) return MLA_OK;
  // sized for the worker count this call will use
  const size_t need = mla::decode_workspace_bytes(dims, batch, num_workers, flags);
  if (need == 0) {
    // invalid or unsupported arguments: let the regular entry point name the error
    return mla_decode_attn(dims, batch, q, pool, block_table, max_blocks_per_seq, num_blocks,
                           seq_stride_tokens, seqlens, scale, num_workers, flags, nullptr, 0, z_out,
                           z_is_fp32, lse_out, dev_status, stream);
  }
  if (need > (size_t)MLA_NOALLOC_SCRATCH_BYTES) return MLA_ERR_WORKSPACE;
  void* scratch = nullptr;
  const int st = scratch_address(&scratch);
  if (st != MLA_OK) return st;
  return mla_decode_attn(dims, batch, q, pool, block_table, max_blocks_per_seq, num_blocks, seq_stride_tokens,
                         seqlens, scale, num_workers, flags, scratch, (size_t)MLA_NOALLOC_SCRATCH_BYTES, z_out,
                         z_is_fp32, lse_out, dev_status, stream);
}

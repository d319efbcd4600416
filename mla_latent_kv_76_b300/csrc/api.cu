// C ABI of libmla.so: argument validation, workspace sizing and launches.
// Nothing here computes a value of the method; every numeric step runs in
// the kernels of the other files.
#include <math.h>
#include <stdint.h>

#include <atomic>

#include "../../include/mla.h"
#include "kernels.h"

namespace {

using mla::DecodeLaunch;

constexpr int kMaxDevices = 64;
std::atomic<int> g_sm_count[kMaxDevices];

int device_sm_count() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return -1;
  if (dev < kMaxDevices) {
    const int cached = g_sm_count[dev].load(std::memory_order_relaxed);
    if (cached > 0) return cached;
  }
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return -1;
  if (dev < kMaxDevices) g_sm_count[dev].store(n, std::memory_order_relaxed);
  return n;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

cudaStream_t as_stream(void* s) { return static_cast<cudaStream_t>(s); }

int from_cuda(cudaError_t e) { return e == cudaSuccess ? MLA_OK : MLA_ERR_CUDA; }

bool dims_basic_ok(const mla_dims* d) {
  if (!d) return false;
  if (d->n_heads < 1 || d->d_head < 1 || d->d_v < 1 || d->d_latent < 1 || d->d_rope < 0) return false;
  if (d->d_rope % 2 != 0) return false;
  if (!(d->rope_base > 0.f) || !isfinite(d->rope_base)) return false;
  return true;
}

size_t align256(size_t x) { return (x + 255) / 256 * 256; }

struct WsLayout {
  size_t off_plan, off_o, off_lse, off_l, off_lq, total;
};

// Workspace: a header (64 bytes of plan scalars, then two int32 per sequence:
// the partial slots the combine reads), then per split-KV partial slot (worker
// g + sequence b) the latent vector o [n_h][d_c] and three per-head scalars.
WsLayout ws_layout(const mla_dims& d, int batch, int workers) {
  WsLayout w;
  const size_t slots = (size_t)workers + (size_t)batch;
  w.off_plan = 64;
  w.off_o = align256(w.off_plan + 8 * (size_t)batch);
  w.off_lse = w.off_o + align256(slots * d.n_heads * d.d_latent * sizeof(float));
  w.off_l = w.off_lse + align256(slots * d.n_heads * sizeof(float));
  w.off_lq = w.off_l + align256(slots * d.n_heads * sizeof(float));
  w.total = w.off_lq + align256(slots * d.n_heads * sizeof(float));
  return w;
}

bool decode_dims_ok(const mla_dims* d, int* why) {
  *why = MLA_ERR_INVALID_ARG;
  if (!dims_basic_ok(d)) return false;
  *why = MLA_ERR_UNSUPPORTED;
  if (d->n_heads > 128) return false;
  if (d->d_latent != 64 && d->d_latent != 128 && d->d_latent != 256 && d->d_latent != 512) return false;
  const int D = d->d_latent + d->d_rope;
  if (D % 16 != 0 || d->d_rope > 128) return false;
  return true;
}

int auto_workers(const mla_dims& d, int num_sms) {
  const int hg = mla::generic_head_groups(d.n_heads);
  int g = num_sms / hg;
  return g < 1 ? 1 : g;
}

}  // namespace

extern "C" {

int mla_version(void) { return 10000; }

const char* mla_status_string(int s) {
  switch (s) {
    case MLA_OK: return "ok";
    case MLA_ERR_INVALID_ARG: return "invalid argument";
    case MLA_ERR_UNSUPPORTED: return "unsupported shape";
    case MLA_ERR_WORKSPACE: return "workspace missing or too small";
    case MLA_ERR_CUDA: return "CUDA error";
    case MLA_ERR_DEVICE_TIMEOUT: return "device wait timed out";
    case MLA_ERR_DEVICE_BOUNDS: return "device index out of range";
    default: return "unknown status";
  }
}

int mla_absorb_q(const mla_dims* dims, int32_t batch, const void* q_c, const void* q_r,
                 const int32_t* pos, const void* w_uk, void* q_out, void* stream) {
  if (!dims_basic_ok(dims) || batch < 0) return MLA_ERR_INVALID_ARG;
  if (dims->d_head % 8 || dims->d_latent % 8 || dims->d_rope > 128) return MLA_ERR_UNSUPPORTED;
  if (batch == 0) return MLA_OK;
  if (!q_c || !pos || !w_uk || !q_out || (dims->d_rope > 0 && !q_r)) return MLA_ERR_INVALID_ARG;
  if (!aligned16(q_c) || !aligned16(w_uk) || !aligned16(q_out) || (q_r && ((uintptr_t)q_r & 3)))
    return MLA_ERR_INVALID_ARG;
  return from_cuda(mla::launch_absorb(*dims, batch, q_c, q_r, pos, w_uk, q_out, as_stream(stream)));
}

int mla_append_cache(const mla_dims* dims, int32_t n_tokens, int32_t d_model, const void* h,
                     const void* w_dkv_kr, const int32_t* seq_idx, const int32_t* pos,
                     int32_t n_seqs, const int32_t* block_table, int32_t max_blocks_per_seq,
                     int32_t num_blocks, int64_t seq_stride_tokens, void* pool,
                     int32_t* dev_status, void* stream) {
  if (!dims_basic_ok(dims) || n_tokens < 0 || d_model < 1 || n_seqs < 0) return MLA_ERR_INVALID_ARG;
  if (d_model % 8 || (dims->d_latent + dims->d_rope) % 8 || dims->d_latent % 2 || dims->d_rope > 128)
    return MLA_ERR_UNSUPPORTED;
  if (n_tokens == 0) return MLA_OK;
  if (!h || !w_dkv_kr || !seq_idx || !pos || !pool || n_seqs < 1) return MLA_ERR_INVALID_ARG;
  if (!aligned16(h) || !aligned16(w_dkv_kr) || !aligned16(pool)) return MLA_ERR_INVALID_ARG;
  if (block_table) {
    if (max_blocks_per_seq < 1 || num_blocks < 1 || dims->block_tokens < 1) return MLA_ERR_INVALID_ARG;
  } else if (seq_stride_tokens < 1) {
    return MLA_ERR_INVALID_ARG;
  }
  return from_cuda(mla::launch_append(*dims, n_tokens, d_model, h, w_dkv_kr, seq_idx, pos, n_seqs,
                                      block_table, max_blocks_per_seq, num_blocks, seq_stride_tokens,
                                      pool, dev_status, as_stream(stream)));
}

}  // extern "C"

namespace mla {

// The split-KV worker count a decode call uses: the caller's, else one per SM
// pair on the tensor-core path and auto_workers on the shape-generic path.
int decode_workers(const mla_dims& d, int batch, int num_workers, int flags, int sms) {
  if (num_workers > 0) return num_workers;
  DecodeLaunch a;
  a.n_heads = d.n_heads;
  a.d_latent = d.d_latent;
  a.d_rope = d.d_rope;
  a.batch = batch;
  const bool native = !(flags & MLA_DECODE_FORCE_GENERIC);
  if (native && tc_supported(a)) return sms / 2 > 0 ? sms / 2 : 1;  // one per SM pair
  if (native && lh_supported(a)) return sms;                         // one per SM
  return auto_workers(d, sms);
}

size_t decode_workspace_bytes(const mla_dims* dims, int batch, int num_workers, int flags) {
  int why = 0;
  if (!decode_dims_ok(dims, &why) || batch < 0 || batch > kMaxBatch || num_workers < 0 ||
      num_workers > kMaxWorkers || (flags & ~MLA_DECODE_FORCE_GENERIC))
    return 0;
  const int sms = num_workers > 0 ? 1 : device_sm_count();
  if (sms <= 0) return 0;
  return ws_layout(*dims, batch, decode_workers(*dims, batch, num_workers, flags, sms)).total;
}

}  // namespace mla

extern "C" {

size_t mla_decode_workspace_size(const mla_dims* dims, int32_t batch, int32_t num_workers) {
  int why = 0;
  if (!decode_dims_ok(dims, &why) || batch < 0 || batch > mla::kMaxBatch || num_workers < 0 ||
      num_workers > mla::kMaxWorkers)
    return 0;
  int G = num_workers;
  if (G == 0) {
    const int sms = device_sm_count();
    if (sms <= 0) return 0;
    G = sms;  // upper bound of every automatic worker count
  }
  return ws_layout(*dims, batch, G).total;
}

int mla_decode_attn(const mla_dims* dims, int32_t batch, const void* q, const void* pool,
                    const int32_t* block_table, int32_t max_blocks_per_seq, int32_t num_blocks,
                    int64_t seq_stride_tokens, const int32_t* seqlens, float scale,
                    int32_t num_workers, int32_t flags, void* workspace, size_t workspace_bytes,
                    void* z_out, int32_t z_is_fp32, float* lse_out, int32_t* dev_status,
                    void* stream) {
  int why = 0;
  if (!decode_dims_ok(dims, &why)) return why;
  if (batch < 0 || num_workers < 0 || num_workers > mla::kMaxWorkers || !isfinite(scale))
    return MLA_ERR_INVALID_ARG;
  if (batch > mla::kMaxBatch) return MLA_ERR_UNSUPPORTED;
  if (flags & ~MLA_DECODE_FORCE_GENERIC) return MLA_ERR_INVALID_ARG;
  if (batch == 0) return MLA_OK;
  if (!q || !pool || !seqlens || !z_out) return MLA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(pool) || !aligned16(z_out)) return MLA_ERR_INVALID_ARG;
  if (block_table) {
    if (max_blocks_per_seq < 1 || num_blocks < 1) return MLA_ERR_INVALID_ARG;
    if (dims->block_tokens != mla::kTileTokens) return MLA_ERR_UNSUPPORTED;
  } else if (seq_stride_tokens < 1) {
    return MLA_ERR_INVALID_ARG;
  }
  const int sms = device_sm_count();
  if (sms <= 0) return MLA_ERR_CUDA;
  DecodeLaunch a;
  a.n_heads = dims->n_heads;
  a.d_latent = dims->d_latent;
  a.d_rope = dims->d_rope;
  a.batch = batch;
  const bool use_tc = !(flags & MLA_DECODE_FORCE_GENERIC) && mla::tc_supported(a);
  const int G = mla::decode_workers(*dims, batch, num_workers, flags, sms);
  const WsLayout w = ws_layout(*dims, batch, G);
  if (!workspace || !aligned16(workspace)) return MLA_ERR_WORKSPACE;
  if (workspace_bytes < w.total) return MLA_ERR_WORKSPACE;

  a.q = q;
  a.pool = pool;
  a.block_table = block_table;
  a.max_blocks = max_blocks_per_seq;
  a.num_blocks = num_blocks;
  a.seq_stride = seq_stride_tokens;
  a.seqlens = seqlens;
  a.scale = scale;
  a.workers = G;
  a.o_part = reinterpret_cast<float*>(static_cast<char*>(workspace) + w.off_o);
  a.plan_flag = static_cast<int32_t*>(workspace);  // header words: plan kind, tiles, workers
  a.seqplan = reinterpret_cast<int32_t*>(static_cast<char*>(workspace) + w.off_plan);
  a.lse_part = reinterpret_cast<float*>(static_cast<char*>(workspace) + w.off_lse);
  a.l_part = reinterpret_cast<float*>(static_cast<char*>(workspace) + w.off_l);
  a.lq_part = reinterpret_cast<float*>(static_cast<char*>(workspace) + w.off_lq);
  a.z_out = z_out;
  a.z_is_fp32 = z_is_fp32 ? 1 : 0;
  a.lse_out = lse_out;
  a.status = dev_status;
  cudaStream_t s = as_stream(stream);
  if (use_tc) return from_cuda(mla::launch_decode_tc(a, s));  // partial pass + its combine
  if (!(flags & MLA_DECODE_FORCE_GENERIC) && mla::lh_supported(a)) return from_cuda(mla::launch_decode_lh(a, s));
  cudaError_t e = mla::launch_decode_generic(a, sms, s);
  if (e != cudaSuccess) return MLA_ERR_CUDA;
  return from_cuda(mla::launch_combine(a, s));
}

int mla_out_proj(const mla_dims* dims, int32_t batch, const void* z, const void* w_uv,
                 void* o_out, void* stream) {
  if (!dims_basic_ok(dims) || batch < 0) return MLA_ERR_INVALID_ARG;
  if (dims->d_latent % 8 || dims->d_v % 8) return MLA_ERR_UNSUPPORTED;
  if (batch == 0) return MLA_OK;
  if (!z || !w_uv || !o_out) return MLA_ERR_INVALID_ARG;
  if (!aligned16(z) || !aligned16(w_uv) || !aligned16(o_out)) return MLA_ERR_INVALID_ARG;
  return from_cuda(mla::launch_out_proj(*dims, batch, z, w_uv, o_out, as_stream(stream)));
}

int mla_read_status(const int32_t* dev_status, int32_t* host_status, void* stream) {
  if (!dev_status || !host_status) return MLA_ERR_INVALID_ARG;
  cudaStream_t s = as_stream(stream);
  if (cudaMemcpyAsync(host_status, dev_status, sizeof(int32_t), cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return MLA_ERR_CUDA;
  return from_cuda(cudaStreamSynchronize(s));
}

}  // extern "C"

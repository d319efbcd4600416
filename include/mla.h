/*
 * mla.h - C ABI of the MLA latent-space decode library (libmla.so, sm_103a).
 *
 * Multi-head Latent Attention (MLA) caches, per token and layer, one joint
 * key/value latent c^KV (d_c values) plus one decoupled RoPE key k^R (d_R
 * values) that every head shares.  Decode attends directly in latent space:
 * W^UK is folded into the query, W^UV is applied after the weighted sum.
 * Sources: "MLA模型结构详解：从公式到推理代码" (gentlecold.top), sections
 * MLA 的核心结构, RoPE 为什么要解耦, 结合 DeepSeek 推理代码看 MLA and the worked
 * example 一个实际推理示例; "DeepSeek-V2 MLA visual reading" (syt-nju.github.io),
 * sections on joint compression, absorption and decoupled RoPE.
 *
 * Conventions shared by every entry point
 *  - bf16 tensors are passed as void* holding __nv_bfloat16 values; all data
 *    pointers are DEVICE pointers owned by the caller.  The library allocates
 *    no device memory (mla_decode_attn_noalloc's static scratch aside), keeps
 *    no state between calls beyond per-device launch attributes and never
 *    synchronises the stream (except mla_read_status).
 *  - `stream` is a cudaStream_t (NULL = legacy default stream).  Work is
 *    enqueued asynchronously; the int return value is the result of host-side
 *    argument validation and of the launch itself.
 *  - A cache row is [c^KV (d_c) | RoPE(k^R) (d_R)], D = d_c + d_R bf16 values
 *    (576 at d_c = 512, d_R = 64: 1152 bytes).  The cache is either
 *      paged:      pool [num_blocks][block_tokens][D], token t of sequence b at
 *                  block block_table[b * max_blocks_per_seq + t / block_tokens],
 *                  slot t % block_tokens;
 *      contiguous: block_table == NULL, pool [batch][seq_stride_tokens][D].
 *  - Positions are 0-based.  seqlens[b] counts the visible tokens of sequence
 *    b including the token appended at this step (the worked example writes
 *    slot start_pos and then attends to start_pos + 1 tokens).
 *  - RoPE rotates pairs (x[2i], x[2i+1]) by pos * rope_base^(-2i / d_R).
 *  - `dev_status` (where present) is an optional device int32, zeroed by the
 *    caller; a kernel that meets an out-of-range block id, position or
 *    sequence length skips that access and stores the first such error code
 *    there.  Read it with mla_read_status.
 *
 * Error behaviour: every entry point returns MLA_OK or one of the codes
 * below and never aborts, prints or throws.  On a non-OK return nothing was
 * enqueued, except MLA_ERR_CUDA from a failed launch.
 */
#ifndef MLA_H_
#define MLA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum {
  MLA_OK = 0,
  MLA_ERR_INVALID_ARG = 1,    /* null pointer, negative or inconsistent size */
  MLA_ERR_UNSUPPORTED = 2,    /* shape outside what the kernels implement */
  MLA_ERR_WORKSPACE = 3,      /* workspace missing or smaller than required */
  MLA_ERR_CUDA = 4,           /* a CUDA runtime call or launch failed */
  MLA_ERR_DEVICE_TIMEOUT = 5, /* device-side bounded wait gave up (dev_status) */
  MLA_ERR_DEVICE_BOUNDS = 6   /* device-side index check failed (dev_status) */
};

/* Model dimensions (host struct, read during the call only). */
typedef struct mla_dims {
  int32_t n_heads;      /* n_h: attention heads */
  int32_t d_head;       /* d_h: per-head content query/key dim (q^C, k^C) */
  int32_t d_v;          /* per-head value dim (v^C) */
  int32_t d_latent;     /* d_c: joint KV latent dim (kv_lora_rank) */
  int32_t d_rope;       /* d_R: decoupled RoPE dim (qk_rope_head_dim), even */
  int32_t block_tokens; /* tokens per cache block; 64 */
  float rope_base;      /* RoPE base, 10000 */
} mla_dims;

/*
 * Query absorption ("为什么矩阵吸收很关键": q^C.(W^UK c) = (q^C W^UK).c; worked
 * example step 4).  For every sequence b and head i:
 *   q_out[b][i][0:d_c]      = W^UK_i^T q^C_{b,i}          (bf16, fp32 accumulate)
 *   q_out[b][i][d_c:d_c+d_R] = RoPE(q^R_{b,i}, pos[b])
 *   q_c   [batch][n_h][d_h]   bf16
 *   q_r   [batch][n_h][d_R]   bf16, before RoPE
 *   pos   [batch]             int32, position of the decode token
 *   w_uk  [n_h][d_h][d_c]     bf16 (k^C_i = W^UK_i c)
 *   q_out [batch][n_h][d_c + d_R] bf16
 * Requires d_h, d_c multiples of 8 and d_R even and <= 128
 * (MLA_ERR_UNSUPPORTED otherwise).  batch == 0 is a no-op.
 */
int mla_absorb_q(const mla_dims* dims, int32_t batch, const void* q_c, const void* q_r,
                 const int32_t* pos, const void* w_uk, void* q_out, void* stream);

/*
 * Cache append ("MLA 的核心结构": c^KV = W^DKV h; "RoPE 为什么要解耦":
 * k^R = RoPE(W^KR h); worked example steps 2-3: the new rows are written at
 * start_pos).  For each new token t:
 *   row = [W^DKV h_t | RoPE(W^KR h_t, pos[t])]  rounded to bf16 (RNE)
 *   written to the cache slot of (seq_idx[t], pos[t]).
 *   h        [n_tokens][d_model]          bf16
 *   w_dkv_kr [d_c + d_R][d_model]         bf16 (W^DKV rows, then W^KR rows)
 *   seq_idx  [n_tokens], pos [n_tokens]   int32 device arrays
 *   paged:      block_table [n_seqs][max_blocks_per_seq], pool of num_blocks blocks
 *   contiguous: block_table NULL, pool [n_seqs][seq_stride_tokens][D]
 * A token whose sequence, position or block id is out of range is skipped
 * and MLA_ERR_DEVICE_BOUNDS is stored in *dev_status.  Two tokens that map
 * to the same slot race.  Requires d_model and d_c + d_R multiples of 8, d_c
 * even and d_R <= 128 (MLA_ERR_UNSUPPORTED otherwise).  n_tokens == 0 is a
 * no-op.
 */
int mla_append_cache(const mla_dims* dims, int32_t n_tokens, int32_t d_model, const void* h,
                     const void* w_dkv_kr, const int32_t* seq_idx, const int32_t* pos,
                     int32_t n_seqs, const int32_t* block_table, int32_t max_blocks_per_seq,
                     int32_t num_blocks, int64_t seq_stride_tokens, void* pool,
                     int32_t* dev_status, void* stream);

/*
 * Bytes of device workspace mla_decode_attn needs for `batch` sequences with
 * `num_workers` split-KV workers (0 = the automatic count for the current
 * device).  Returns 0 on invalid arguments.
 */
size_t mla_decode_workspace_size(const mla_dims* dims, int32_t batch, int32_t num_workers);

/* flags for mla_decode_attn */
enum {
  MLA_DECODE_DEFAULT = 0,
  MLA_DECODE_FORCE_GENERIC = 1 /* use the shape-generic kernel even where a specialised one exists */
};

/*
 * Latent-space decode attention ("结合 DeepSeek 推理代码看 MLA": score =
 * (q^C W^UK).c^KV + q^R.k^R; worked example steps 4-5: scale, causal mask,
 * softmax, z = A . kv_cache).  For every sequence b and head i over the
 * visible tokens j < seqlens[b]:
 *   s_j   = scale * (q[b][i][0:d_c] . c_j + q[b][i][d_c:] . k^R_j)
 *   lse   = log sum_j exp(s_j)
 *   z     = sum_j exp(s_j - lse) c_j
 * computed as split-KV partial passes (online softmax over 64-token tiles, or
 * 128-token tiles on the tensor-core path for n_h = 128, d_c = 512, d_R = 64)
 * followed by a log-sum-exp combine.  A sequence with seqlens[b] == 0 gives
 * z = 0, lse = -inf.
 *   q        [batch][n_h][d_c + d_R] bf16 (output of mla_absorb_q)
 *   pool / block_table / max_blocks_per_seq / num_blocks / seq_stride_tokens:
 *            cache layout as above (read only)
 *   seqlens  [batch] int32 device array
 *   scale    softmax scale, normally 1/sqrt(d_h + d_R)
 *   num_workers  split-KV workers (0 = automatic: one per SM pair on the
 *            tensor-core path); the result is the same for every value up to
 *            floating-point rounding.  The shape-generic path gives worker g
 *            tiles [floor(g T / G), floor((g + 1) T / G)) of the batch's tile
 *            list (T tiles, G workers).  The tensor-core path chooses, per
 *            call and on the device, between that even split and cutting
 *            sequence b into w_b = min(t_b, 1 + floor((G - n) t_b / T))
 *            pieces (t_b its 128-token tiles, n non-empty sequences; one
 *            piece per sequence when G <= n), which keeps each worker inside
 *            one sequence while the pieces fit the workers; it takes the
 *            pieces unless their longest exceeds the even split's bound
 *            Q + 3 ceil(Q / t_min) (Q = ceil(T / G), t_min the fewest tiles
 *            of a non-empty sequence).
 *   workspace / workspace_bytes: device scratch of at least
 *            mla_decode_workspace_size(dims, batch, num_workers) bytes; its
 *            contents on entry do not matter
 *   z_out    [batch][n_h][d_c], fp32 if z_is_fp32 else bf16
 *   lse_out  [batch][n_h] fp32, natural log; may be NULL
 * Sequence lengths above the cache capacity, or block ids outside
 * [0, num_blocks), are treated as empty / zero rows and reported through
 * dev_status.  If a bounded device-side wait gives up (MLA_ERR_DEVICE_TIMEOUT
 * in dev_status), the tensor-core path writes NaN to z_out and lse_out; the
 * outputs of a call whose dev_status is non-zero are otherwise not defined
 * beyond the rules above.  Requires n_h <= 128, d_c in {64, 128, 256, 512},
 * (d_c + d_R) a multiple of 16, block_tokens == 64 for a paged cache.
 */
int mla_decode_attn(const mla_dims* dims, int32_t batch, const void* q, const void* pool,
                    const int32_t* block_table, int32_t max_blocks_per_seq, int32_t num_blocks,
                    int64_t seq_stride_tokens, const int32_t* seqlens, float scale,
                    int32_t num_workers, int32_t flags, void* workspace, size_t workspace_bytes,
                    void* z_out, int32_t z_is_fp32, float* lse_out, int32_t* dev_status,
                    void* stream);

/*
 * Decode without a caller-provided workspace.  The pages have no counterpart
 * to this entry point; it exists for callers that cannot allocate device
 * memory when they call decode: a plugin inside an inference server that is
 * handed only its input and output buffers and has no allocator of its own,
 * or a latency-critical serving loop that forbids cudaMalloc after start-up
 * because an allocation can synchronise the device or fail under memory
 * pressure.  It runs the same kernels as mla_decode_attn, with the split-KV
 * partials in a file-scope device array of MLA_NOALLOC_SCRATCH_BYTES (64 MiB)
 * that every GPU which loads the library holds until the process exits.
 *  - Arguments are those of mla_decode_attn without workspace/workspace_bytes.
 *  - If the workspace this call needs (mla_decode_workspace_size for the
 *    worker count the call uses: num_workers, else the automatic count of
 *    its path, one per SM pair on the tensor-core path) is larger than
 *    MLA_NOALLOC_SCRATCH_BYTES the call returns MLA_ERR_WORKSPACE and
 *    enqueues nothing.  (On a 148-SM B300 with 128 heads, d_c = 512 and
 *    automatic workers this allows up to 180 sequences; passing an explicit,
 *    smaller num_workers allows more.)
 *  - It allocates nothing: no cudaMalloc, cudaFree or allocating library call.
 *  - Every call looks up the array's device address (cudaGetSymbolAddress)
 *    on the current device, so a context re-created after a device reset
 *    gets its own array.  The first lookup on a device loads the library's
 *    device code there; make that first call before any stream capture.
 *  - All calls share the one array, which keeps the last call's contents.
 *    Nothing in it has to start at zero: each call writes every partial it
 *    reads back.  Calls whose GPU work overlaps (other streams, or threads
 *    without ordering between them) race on the array and return wrong
 *    results; serialise them, for example on one stream.
 */
#define MLA_NOALLOC_SCRATCH_BYTES (64u << 20)
int mla_decode_attn_noalloc(const mla_dims* dims, int32_t batch, const void* q, const void* pool,
                            const int32_t* block_table, int32_t max_blocks_per_seq, int32_t num_blocks,
                            int64_t seq_stride_tokens, const int32_t* seqlens, float scale,
                            int32_t num_workers, int32_t flags, void* z_out, int32_t z_is_fp32,
                            float* lse_out, int32_t* dev_status, void* stream);

/*
 * Value up-projection after the latent sum ("为什么矩阵吸收很关键":
 * sum_j A_j W^UV c_j = W^UV sum_j A_j c_j; worked example step 5).
 *   o[b][i] = W^UV_i z[b][i]           (bf16 out, fp32 accumulate)
 *   z     [batch][n_h][d_c]  bf16
 *   w_uv  [n_h][d_v][d_c]    bf16
 *   o_out [batch][n_h][d_v]  bf16
 * Requires d_c and d_v multiples of 8 (MLA_ERR_UNSUPPORTED otherwise).
 */
int mla_out_proj(const mla_dims* dims, int32_t batch, const void* z, const void* w_uv,
                 void* o_out, void* stream);

/*
 * Self-test of the device-side bounded wait every kernel uses on its
 * mbarriers.  Launches one CTA of 64 threads on `stream`: thread 0 waits on a
 * barrier that nothing arrives on, giving up after `budget_cycles` SM cycles
 * (1 .. 4e9); it then raises the CTA's abort flag and stores
 * MLA_ERR_DEVICE_TIMEOUT in *dev_status (may be NULL), and thread 32, which
 * waits with the full ~2 s budget on another such barrier, leaves on the
 * flag.  dev_out (device, 2 int32) receives 1 per wait that succeeded, 0 per
 * wait that gave up.  With `arrive` non-zero both barriers are completed
 * first (control case: dev_out = {1, 1}, nothing reported).  Nothing faults or
 * hangs: the kernel returns within about budget_cycles.
 */
int mla_selftest_bounded_wait(int64_t budget_cycles, int32_t arrive, int32_t* dev_status, int32_t* dev_out,
                              void* stream);

/* Synchronise `stream`, copy *dev_status to *host_status and return MLA_OK
 * (or MLA_ERR_CUDA if the copy failed). */
int mla_read_status(const int32_t* dev_status, int32_t* host_status, void* stream);

/* Static, human-readable name of a status code. */
const char* mla_status_string(int status);

/* Library version, e.g. 10000 for 1.0.0. */
int mla_version(void);

#ifdef __cplusplus
}
#endif

#endif /* MLA_H_ */

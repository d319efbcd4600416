"""ctypes binding of libmla.so.  Same entry-point names as include/mla.h.

Each wrapper takes torch CUDA tensors, checks dtype / device / contiguity,
passes raw pointers and the current stream, and raises MlaError on a non-OK
status.  bf16 tensors may be torch.bfloat16 or int16/uint16 holding bf16 bits.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libmla.so")

MLA_OK = 0
MLA_ERR_INVALID_ARG = 1
MLA_ERR_UNSUPPORTED = 2
MLA_ERR_WORKSPACE = 3
MLA_ERR_CUDA = 4
MLA_ERR_DEVICE_TIMEOUT = 5
MLA_ERR_DEVICE_BOUNDS = 6
MLA_DECODE_FORCE_GENERIC = 1
MLA_NOALLOC_SCRATCH_BYTES = 64 << 20

if not os.path.exists(LIB_PATH):
    raise ImportError(f"{LIB_PATH} is missing: build it with `python mla_latent_kv_76_b300/build.py` "
                      "(there is no fallback implementation)")

lib = ctypes.CDLL(LIB_PATH)


class Dims(ctypes.Structure):
    """mla_dims: n_heads, d_head, d_v, d_latent, d_rope, block_tokens, rope_base."""
    _fields_ = [("n_heads", ctypes.c_int32), ("d_head", ctypes.c_int32), ("d_v", ctypes.c_int32),
                ("d_latent", ctypes.c_int32), ("d_rope", ctypes.c_int32),
                ("block_tokens", ctypes.c_int32), ("rope_base", ctypes.c_float)]

    @classmethod
    def of(cls, wl) -> "Dims":
        return cls(wl.n_heads, wl.d_head, wl.d_v, wl.d_latent, wl.d_rope, wl.block_tokens, wl.rope_base)


class MlaError(RuntimeError):
    def __init__(self, fn: str, code: int):
        super().__init__(f"{fn} failed: {code} ({mla_status_string(code)})")
        self.code = code


_P = ctypes.c_void_p
_I32 = ctypes.c_int32
_I64 = ctypes.c_int64
_DP = ctypes.POINTER(Dims)

lib.mla_absorb_q.argtypes = [_DP, _I32, _P, _P, _P, _P, _P, _P]
lib.mla_append_cache.argtypes = [_DP, _I32, _I32, _P, _P, _P, _P, _I32, _P, _I32, _I32, _I64, _P, _P, _P]
lib.mla_decode_workspace_size.argtypes = [_DP, _I32, _I32]
lib.mla_decode_workspace_size.restype = ctypes.c_size_t
lib.mla_decode_attn.argtypes = [_DP, _I32, _P, _P, _P, _I32, _I32, _I64, _P, ctypes.c_float, _I32, _I32,
                                _P, ctypes.c_size_t, _P, _I32, _P, _P, _P]
lib.mla_out_proj.argtypes = [_DP, _I32, _P, _P, _P, _P]
lib.mla_decode_attn_noalloc.argtypes = [_DP, _I32, _P, _P, _P, _I32, _I32, _I64, _P, ctypes.c_float, _I32, _I32,
                                        _P, _I32, _P, _P, _P]
lib.mla_read_status.argtypes = [_P, _P, _P]
lib.mla_selftest_bounded_wait.argtypes = [_I64, _I32, _P, _P, _P]
lib.mla_status_string.argtypes = [ctypes.c_int]
lib.mla_status_string.restype = ctypes.c_char_p
lib.mla_version.argtypes = []
for _fn in ("mla_absorb_q", "mla_append_cache", "mla_decode_attn", "mla_out_proj", "mla_read_status",
            "mla_version", "mla_decode_attn_noalloc", "mla_selftest_bounded_wait"):
    getattr(lib, _fn).restype = ctypes.c_int


def mla_status_string(code: int) -> str:
    return lib.mla_status_string(int(code)).decode()


def mla_version() -> int:
    return lib.mla_version()


_BF16_LIKE = (torch.bfloat16, torch.int16, torch.uint16)


def _ptr(t: Optional[torch.Tensor], name: str, dtypes=None) -> Optional[int]:
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor (the library has no CPU path)")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtypes is not None and t.dtype not in dtypes:
        raise TypeError(f"{name} has dtype {t.dtype}, expected one of {dtypes}")
    return t.data_ptr()


def _need(t: Optional[torch.Tensor], n: int, name: str) -> None:
    """The library sees only pointers: refuse a buffer smaller than the call
    will read or write through it."""
    if t is not None and isinstance(t, torch.Tensor) and t.numel() < n:
        raise ValueError(f"{name} holds {t.numel()} elements, the call needs at least {n}")


_Z_DTYPES = (torch.float32,) + _BF16_LIKE


def _stream(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _check(fn: str, code: int):
    if code != MLA_OK:
        raise MlaError(fn, code)


def mla_absorb_q(dims: Dims, q_c, q_r, pos, w_uk, q_out=None, stream=None):
    """q_out[b, i] = [W^UK_i^T q^C_{b,i} | RoPE(q^R_{b,i}, pos[b])] (bf16)."""
    B = q_c.shape[0]
    if q_out is None:
        q_out = torch.empty((B, dims.n_heads, dims.d_latent + dims.d_rope), dtype=torch.bfloat16,
                            device=q_c.device)
    H = B * dims.n_heads
    _need(q_c, H * dims.d_head, "q_c")
    _need(q_r, H * dims.d_rope, "q_r")
    _need(pos, B, "pos")
    _need(w_uk, dims.n_heads * dims.d_head * dims.d_latent, "w_uk")
    _need(q_out, H * (dims.d_latent + dims.d_rope), "q_out")
    code = lib.mla_absorb_q(ctypes.byref(dims), B, _ptr(q_c, "q_c", _BF16_LIKE), _ptr(q_r, "q_r", _BF16_LIKE),
                            _ptr(pos, "pos", (torch.int32,)), _ptr(w_uk, "w_uk", _BF16_LIKE),
                            _ptr(q_out, "q_out", _BF16_LIKE), _stream(stream))
    _check("mla_absorb_q", code)
    return q_out


def mla_append_cache(dims: Dims, h, w_dkv_kr, seq_idx, pos, pool, n_seqs: int, block_table=None,
                     num_blocks: int = 0, seq_stride: int = 0, dev_status=None, stream=None):
    """Project h through [W^DKV; W^KR], RoPE the k^R part, write bf16 rows into `pool` in place."""
    T, d_model = h.shape
    max_blocks = 0 if block_table is None else block_table.shape[1]
    D = dims.d_latent + dims.d_rope
    _need(w_dkv_kr, D * d_model, "w_dkv_kr")
    _need(seq_idx, T, "seq_idx")
    _need(pos, T, "pos")
    if block_table is not None:
        _need(block_table, n_seqs * max_blocks, "block_table")
        _need(pool, num_blocks * dims.block_tokens * D, "pool")
    else:
        _need(pool, n_seqs * seq_stride * D, "pool")
    code = lib.mla_append_cache(ctypes.byref(dims), T, d_model, _ptr(h, "h", _BF16_LIKE),
                                _ptr(w_dkv_kr, "w_dkv_kr", _BF16_LIKE), _ptr(seq_idx, "seq_idx", (torch.int32,)),
                                _ptr(pos, "pos", (torch.int32,)), n_seqs,
                                _ptr(block_table, "block_table", (torch.int32,)), max_blocks, num_blocks,
                                seq_stride, _ptr(pool, "pool", _BF16_LIKE),
                                _ptr(dev_status, "dev_status", (torch.int32,)), _stream(stream))
    _check("mla_append_cache", code)
    return pool


def mla_decode_workspace_size(dims: Dims, batch: int, num_workers: int = 0) -> int:
    return int(lib.mla_decode_workspace_size(ctypes.byref(dims), batch, num_workers))


def _check_decode_buffers(dims, B, q, pool, seqlens, block_table, max_blocks, num_blocks, seq_stride, z_out,
                          lse_out) -> None:
    D = dims.d_latent + dims.d_rope
    H = B * dims.n_heads
    _need(q, H * D, "q")
    _need(seqlens, B, "seqlens")
    if block_table is not None:
        _need(block_table, B * max_blocks, "block_table")
        _need(pool, num_blocks * dims.block_tokens * D, "pool")
    else:
        _need(pool, B * seq_stride * D, "pool")
    if z_out is not None and z_out.dtype not in _Z_DTYPES:
        raise TypeError(f"z_out has dtype {z_out.dtype}, expected float32 or bf16")
    _need(z_out, H * dims.d_latent, "z_out")
    _need(lse_out, H, "lse_out")


def mla_decode_attn(dims: Dims, q, pool, seqlens, scale: float, block_table=None, num_blocks: int = 0,
                    seq_stride: int = 0, num_workers: int = 0, flags: int = 0, workspace=None,
                    z_out=None, z_is_fp32: bool = True, lse_out=None, dev_status=None, stream=None,
                    want_lse: bool = True):
    """Latent-space decode attention; returns (z, lse)."""
    B = q.shape[0]
    dev = q.device
    if workspace is None:
        nbytes = mla_decode_workspace_size(dims, B, num_workers)
        if nbytes == 0 and B > 0:
            raise MlaError("mla_decode_workspace_size", MLA_ERR_INVALID_ARG)
        workspace = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=dev)
    if z_out is None:
        z_out = torch.empty((B, dims.n_heads, dims.d_latent),
                            dtype=torch.float32 if z_is_fp32 else torch.bfloat16, device=dev)
    if lse_out is None and want_lse:
        lse_out = torch.empty((B, dims.n_heads), dtype=torch.float32, device=dev)
    max_blocks = 0 if block_table is None else block_table.shape[1]
    _check_decode_buffers(dims, B, q, pool, seqlens, block_table, max_blocks, num_blocks, seq_stride, z_out, lse_out)
    code = lib.mla_decode_attn(
        ctypes.byref(dims), B, _ptr(q, "q", _BF16_LIKE), _ptr(pool, "pool", _BF16_LIKE),
        _ptr(block_table, "block_table", (torch.int32,)), max_blocks, num_blocks, seq_stride,
        _ptr(seqlens, "seqlens", (torch.int32,)), float(scale), num_workers, flags,
        _ptr(workspace, "workspace"), workspace.numel() * workspace.element_size(),
        _ptr(z_out, "z_out"), 1 if z_out.dtype == torch.float32 else 0,
        _ptr(lse_out, "lse_out", (torch.float32,)), _ptr(dev_status, "dev_status", (torch.int32,)),
        _stream(stream))
    _check("mla_decode_attn", code)
    return z_out, lse_out


def mla_decode_attn_noalloc(dims: Dims, q, pool, seqlens, scale: float, block_table=None, num_blocks: int = 0,
                            seq_stride: int = 0, num_workers: int = 0, flags: int = 0, z_out=None,
                            z_is_fp32: bool = True, lse_out=None, dev_status=None, stream=None,
                            want_lse: bool = True):
    """Decode with the library's built-in scratch instead of a workspace, for
    callers that cannot allocate device memory at call time.  Outputs must be
    passed in for the call itself to allocate nothing.  Returns (z, lse)."""
    B = q.shape[0]
    dev = q.device
    if z_out is None:
        z_out = torch.empty((B, dims.n_heads, dims.d_latent),
                            dtype=torch.float32 if z_is_fp32 else torch.bfloat16, device=dev)
    if lse_out is None and want_lse:
        lse_out = torch.empty((B, dims.n_heads), dtype=torch.float32, device=dev)
    max_blocks = 0 if block_table is None else block_table.shape[1]
    _check_decode_buffers(dims, B, q, pool, seqlens, block_table, max_blocks, num_blocks, seq_stride, z_out, lse_out)
    code = lib.mla_decode_attn_noalloc(
        ctypes.byref(dims), B, _ptr(q, "q", _BF16_LIKE), _ptr(pool, "pool", _BF16_LIKE),
        _ptr(block_table, "block_table", (torch.int32,)), max_blocks, num_blocks, seq_stride,
        _ptr(seqlens, "seqlens", (torch.int32,)), float(scale), num_workers, flags,
        _ptr(z_out, "z_out"), 1 if z_out.dtype == torch.float32 else 0,
        _ptr(lse_out, "lse_out", (torch.float32,)), _ptr(dev_status, "dev_status", (torch.int32,)),
        _stream(stream))
    _check("mla_decode_attn_noalloc", code)
    return z_out, lse_out


def mla_out_proj(dims: Dims, z, w_uv, o_out=None, stream=None):
    """o[b, i] = W^UV_i z[b, i] (bf16 in, bf16 out)."""
    B = z.shape[0]
    if o_out is None:
        o_out = torch.empty((B, dims.n_heads, dims.d_v), dtype=torch.bfloat16, device=z.device)
    _need(z, B * dims.n_heads * dims.d_latent, "z")
    _need(w_uv, dims.n_heads * dims.d_v * dims.d_latent, "w_uv")
    _need(o_out, B * dims.n_heads * dims.d_v, "o_out")
    code = lib.mla_out_proj(ctypes.byref(dims), B, _ptr(z, "z", _BF16_LIKE), _ptr(w_uv, "w_uv", _BF16_LIKE),
                            _ptr(o_out, "o_out", _BF16_LIKE), _stream(stream))
    _check("mla_out_proj", code)
    return o_out


def mla_read_status(dev_status, stream=None) -> int:
    host = ctypes.c_int32(0)
    code = lib.mla_read_status(_ptr(dev_status, "dev_status", (torch.int32,)), ctypes.addressof(host),
                               _stream(stream))
    _check("mla_read_status", code)
    return int(host.value)


def mla_selftest_bounded_wait(budget_cycles: int, arrive: bool, dev_status, dev_out, stream=None):
    """Run the device bounded-wait self-test (include/mla.h); returns nothing,
    results land in dev_status / dev_out on the device."""
    _need(dev_out, 2, "dev_out")
    code = lib.mla_selftest_bounded_wait(int(budget_cycles), 1 if arrive else 0,
                                         _ptr(dev_status, "dev_status", (torch.int32,)),
                                         _ptr(dev_out, "dev_out", (torch.int32,)), _stream(stream))
    _check("mla_selftest_bounded_wait", code)

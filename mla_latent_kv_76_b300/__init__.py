"""MLA latent-space decode on B300: Python binding of libmla.so.

The binding only marshals arguments (tensor pointers, sizes, the current CUDA
stream) into the C ABI declared in include/mla.h; every numeric step runs in
the library's CUDA kernels.  Importing the package fails loudly when
libmla.so has not been built (``python mla_latent_kv_76_b300/build.py``).
"""
from ._binding import (  # noqa: F401
    Dims, MlaError, LIB_PATH, lib,
    MLA_OK, MLA_ERR_INVALID_ARG, MLA_ERR_UNSUPPORTED, MLA_ERR_WORKSPACE, MLA_ERR_CUDA,
    MLA_ERR_DEVICE_TIMEOUT, MLA_ERR_DEVICE_BOUNDS, MLA_DECODE_FORCE_GENERIC, MLA_NOALLOC_SCRATCH_BYTES,
    mla_absorb_q, mla_append_cache, mla_decode_workspace_size, mla_decode_attn, mla_decode_attn_noalloc,
    mla_out_proj,
    mla_read_status, mla_status_string, mla_version, mla_selftest_bounded_wait,
)

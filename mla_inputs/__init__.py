"""Seeded synthetic workloads for MLA latent-space decode.

This module only draws random numbers and lays them out; it holds none of the
attention arithmetic.  Both the CPU oracle (``oracle/``) and the CUDA path
(tests, ``bench.py``) consume the arrays it returns, so the two sides always
see bit-identical bf16 inputs.

Every array that stands for a bf16 tensor is returned as ``uint16`` bit
patterns.  Values are drawn as float32 from ``np.random.default_rng(seed)``
and rounded to bf16 with round-to-nearest-even (NaN kept as a quiet NaN).

Workload shapes follow the DeepSeek-V3 MLA configuration the pages use
(page "MLA模型结构详解", section 结合 DeepSeek 推理代码看 MLA: kv_lora_rank 512,
qk_rope_head_dim 64, qk_nope_head_dim 128, v_head_dim 128; page
"ai.saiita.com.cn", 128 heads per layer) and the five benchmark cases:

* ``tiny``     d=256, n_h=4, d_h=32, d_c=64, d_R=16; fp32 weights N(0, 1/fan_in);
               B=1, 128 context tokens + 1 decode token at position 128.
* ``v3``       n_h=128, d_c=512, d_R=64, B=16, seqlen 4096, contiguous cache.
* ``paged``    v3 heads, B=64, seqlen ~ U{1024..8192}, 64-token blocks,
               pool 1.25x the needed blocks, permuted block table.
* ``long``     v3 heads, B=4, seqlen 131072, paged as above.
* ``lowhead``  n_h=16, B=256, seqlen ~ U{512..4096}, paged, plus one appended
               token per sequence (d=7168) before attention.

Draw order (per seed) is fixed and documented in each builder below.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np

BF16_QNAN = np.uint16(0x7FC0)

CONFIG_NAMES = ("tiny", "v3", "paged", "long", "lowhead")
CONFIG_SEEDS = {"tiny": 0, "v3": 1, "paged": 2, "long": 3, "lowhead": 4}


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (round-to-nearest-even); returns uint16 bits."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32)
    bias = ((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    with np.errstate(over="ignore"):
        r = ((u + bias) >> np.uint32(16)).astype(np.uint16)
    nan = np.isnan(x)
    if nan.any():
        r[nan] = BF16_QNAN
    return r


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to float32."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def _normal_bf16(rng: np.random.Generator, shape, std: float = 1.0, chunk: int = 1 << 24) -> np.ndarray:
    """N(0, std^2) drawn as float32, rounded to bf16 bits; drawn in row-major chunks."""
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.uint16)
    for s in range(0, n, chunk):
        e = min(n, s + chunk)
        v = rng.standard_normal(e - s, dtype=np.float32)
        if std != 1.0:
            v *= np.float32(std)
        out[s:e] = f32_to_bf16_bits(v)
    return out.reshape(shape)


def _normal_f32_to_bf16(rng: np.random.Generator, shape, std: float) -> np.ndarray:
    """Tiny-case weights: drawn as float64, cast to float32, then rounded to bf16."""
    v = rng.standard_normal(shape) * std
    return f32_to_bf16_bits(v.astype(np.float32))


@dataclasses.dataclass
class Workload:
    name: str
    seed: int
    # model dimensions
    n_heads: int
    d_head: int
    d_v: int
    d_latent: int
    d_rope: int
    rope_base: float
    scale: float
    # batch and cache layout
    batch: int
    seqlens: np.ndarray            # int32 [B]: visible tokens incl. the decode token
    block_tokens: int
    paged: bool
    block_table: Optional[np.ndarray]   # int32 [B, max_blocks] (paged) else None
    num_blocks: int                # paged pool capacity in blocks
    seq_stride: int                # contiguous: tokens between sequences
    pool: np.ndarray               # uint16: [num_blocks, block_tokens, D] or [B, seq_stride, D]
    # decode query in latent space (absorbed content part | roped part)
    q: Optional[np.ndarray]        # uint16 [B, n_h, D]
    # inputs of the steps around decode
    q_c: Optional[np.ndarray] = None      # uint16 [B, n_h, d_h]
    q_r: Optional[np.ndarray] = None      # uint16 [B, n_h, d_R] (before RoPE)
    q_pos: Optional[np.ndarray] = None    # int32 [B] position of the decode token
    w_uk: Optional[np.ndarray] = None     # uint16 [n_h, d_h, d_c]
    w_uv: Optional[np.ndarray] = None     # uint16 [n_h, d_v, d_c]
    d_model: int = 0
    h: Optional[np.ndarray] = None        # uint16 [T, d]
    w_dkv_kr: Optional[np.ndarray] = None  # uint16 [d_c + d_R, d]
    app_seq: Optional[np.ndarray] = None  # int32 [T]
    app_pos: Optional[np.ndarray] = None  # int32 [T]
    w_q: Optional[np.ndarray] = None      # uint16 [n_h, d_h + d_R, d] (tiny case only)
    poisoned: bool = False

    @property
    def row_dim(self) -> int:
        return self.d_latent + self.d_rope

    @property
    def max_blocks(self) -> int:
        return 0 if self.block_table is None else int(self.block_table.shape[1])

    @property
    def total_tokens(self) -> int:
        return int(np.asarray(self.seqlens, dtype=np.int64).sum())


def _paged_layout(rng: np.random.Generator, seqlens: np.ndarray, block_tokens: int, factor: float = 1.25):
    """Random permuted block table over a pool `factor` times the needed size."""
    need = [(int(L) + block_tokens - 1) // block_tokens for L in seqlens]
    total_need = int(sum(need))
    num_blocks = int(math.ceil(factor * total_need))
    perm = rng.permutation(num_blocks).astype(np.int32)
    max_blocks = max(1, max(need))
    bt = np.full((len(seqlens), max_blocks), -1, dtype=np.int32)
    k = 0
    for b, n in enumerate(need):
        bt[b, :n] = perm[k:k + n]
        k += n
    return bt, num_blocks


def _poison_paged(pool: np.ndarray, bt: np.ndarray, seqlens: np.ndarray, block_tokens: int) -> None:
    """NaN every pool slot that no sequence can see (unused blocks, tail slack)."""
    used = np.zeros(pool.shape[0], dtype=bool)
    for b, L in enumerate(seqlens):
        n = (int(L) + block_tokens - 1) // block_tokens
        used[bt[b, :n]] = True
        if n and int(L) % block_tokens:
            pool[bt[b, n - 1], int(L) % block_tokens:, :] = BF16_QNAN
    pool[~used] = BF16_QNAN


def make_tiny(seed: int = 0, poison: bool = True) -> Workload:
    """Tiny case.  Draw order: W^DKV, W^UK, W^UV, W^KR, W^Q, then H [129 x 256]."""
    rng = np.random.default_rng(seed)
    d, n_h, d_h, d_c, d_R = 256, 4, 32, 64, 16
    w_dkv = _normal_f32_to_bf16(rng, (d_c, d), 1.0 / math.sqrt(d))
    w_uk = _normal_f32_to_bf16(rng, (n_h, d_h, d_c), 1.0 / math.sqrt(d_c))
    w_uv = _normal_f32_to_bf16(rng, (n_h, d_h, d_c), 1.0 / math.sqrt(d_c))
    w_kr = _normal_f32_to_bf16(rng, (d_R, d), 1.0 / math.sqrt(d))
    w_q = _normal_f32_to_bf16(rng, (n_h, d_h + d_R, d), 1.0 / math.sqrt(d))
    h = _normal_f32_to_bf16(rng, (129, d), 1.0)
    seq_stride = 192
    D = d_c + d_R
    pool = np.full((1, seq_stride, D), BF16_QNAN if poison else np.uint16(0), dtype=np.uint16)
    return Workload(
        name="tiny", seed=seed, n_heads=n_h, d_head=d_h, d_v=d_h, d_latent=d_c, d_rope=d_R,
        rope_base=10000.0, scale=1.0 / math.sqrt(d_h + d_R), batch=1,
        seqlens=np.array([129], dtype=np.int32), block_tokens=64, paged=False, block_table=None,
        num_blocks=0, seq_stride=seq_stride, pool=pool, q=None,
        q_pos=np.array([128], dtype=np.int32), w_uk=w_uk, w_uv=w_uv, d_model=d, h=h,
        w_dkv_kr=np.concatenate([w_dkv, w_kr], axis=0),
        app_seq=np.zeros(129, dtype=np.int32), app_pos=np.arange(129, dtype=np.int32),
        w_q=w_q, poisoned=poison)


def _v3_common(rng, B, n_h, seqlens, paged, poison, block_tokens=64):
    d_c, d_R = 512, 64
    D = d_c + d_R
    if paged:
        bt, num_blocks = _paged_layout(rng, seqlens, block_tokens)
        pool = _normal_bf16(rng, (num_blocks, block_tokens, D))
        if poison:
            _poison_paged(pool, bt, seqlens, block_tokens)
        seq_stride = 0
    else:
        bt, num_blocks = None, 0
        seq_stride = int(max(seqlens))
        pool = _normal_bf16(rng, (B, seq_stride, D))
        if poison:
            for b, L in enumerate(seqlens):
                pool[b, int(L):, :] = BF16_QNAN
    q = _normal_bf16(rng, (B, n_h, D))
    return bt, num_blocks, seq_stride, pool, q


def _step_inputs(rng, wl: Workload, d_model: int = 7168):
    """Inputs of absorb / append / out-projection around decode.

    Draw order: q_c, q_r, W^UK, W^UV, h, [W^DKV; W^KR].  The appended token of
    sequence b goes at position seqlen_b - 1 (it is the decode token itself).
    """
    B, n_h, d_h, d_c, d_R = wl.batch, wl.n_heads, wl.d_head, wl.d_latent, wl.d_rope
    wl.q_c = _normal_bf16(rng, (B, n_h, d_h))
    wl.q_r = _normal_bf16(rng, (B, n_h, d_R))
    wl.w_uk = _normal_bf16(rng, (n_h, d_h, d_c), 1.0 / math.sqrt(d_c))
    wl.w_uv = _normal_bf16(rng, (n_h, wl.d_v, d_c), 1.0 / math.sqrt(d_c))
    wl.d_model = d_model
    wl.h = _normal_bf16(rng, (B, d_model))
    wl.w_dkv_kr = _normal_bf16(rng, (d_c + d_R, d_model), 1.0 / math.sqrt(d_model))
    wl.app_seq = np.arange(B, dtype=np.int32)
    wl.app_pos = (wl.seqlens - 1).astype(np.int32)
    wl.q_pos = (wl.seqlens - 1).astype(np.int32)


def make_v3(seed: int = 1, poison: bool = True, batch: int = 16, seqlen: int = 4096) -> Workload:
    """DeepSeek-V3-shaped single layer, contiguous cache.

    Draw order: cache [B, L, 576], q [B, 128, 576], then the step inputs.
    """
    rng = np.random.default_rng(seed)
    seqlens = np.full(batch, seqlen, dtype=np.int32)
    bt, nb, ss, pool, q = _v3_common(rng, batch, 128, seqlens, False, poison)
    wl = Workload(name="v3", seed=seed, n_heads=128, d_head=128, d_v=128, d_latent=512, d_rope=64,
                  rope_base=10000.0, scale=1.0 / math.sqrt(192), batch=batch, seqlens=seqlens,
                  block_tokens=64, paged=False, block_table=bt, num_blocks=nb, seq_stride=ss,
                  pool=pool, q=q, poisoned=poison)
    _step_inputs(rng, wl)
    return wl


def make_paged(seed: int = 2, poison: bool = True, batch: int = 64, lo: int = 1024, hi: int = 8192) -> Workload:
    """Paged batch.  Draw order: seqlens, block permutation, pool, q, step inputs."""
    rng = np.random.default_rng(seed)
    seqlens = rng.integers(lo, hi, size=batch, endpoint=True).astype(np.int32)
    bt, nb, ss, pool, q = _v3_common(rng, batch, 128, seqlens, True, poison)
    wl = Workload(name="paged", seed=seed, n_heads=128, d_head=128, d_v=128, d_latent=512, d_rope=64,
                  rope_base=10000.0, scale=1.0 / math.sqrt(192), batch=batch, seqlens=seqlens,
                  block_tokens=64, paged=True, block_table=bt, num_blocks=nb, seq_stride=ss,
                  pool=pool, q=q, poisoned=poison)
    _step_inputs(rng, wl)
    return wl


def make_long(seed: int = 3, poison: bool = True, batch: int = 4, seqlen: int = 131072) -> Workload:
    """Long context.  Draw order: block permutation, pool, q, step inputs."""
    rng = np.random.default_rng(seed)
    seqlens = np.full(batch, seqlen, dtype=np.int32)
    bt, nb, ss, pool, q = _v3_common(rng, batch, 128, seqlens, True, poison)
    wl = Workload(name="long", seed=seed, n_heads=128, d_head=128, d_v=128, d_latent=512, d_rope=64,
                  rope_base=10000.0, scale=1.0 / math.sqrt(192), batch=batch, seqlens=seqlens,
                  block_tokens=64, paged=True, block_table=bt, num_blocks=nb, seq_stride=ss,
                  pool=pool, q=q, poisoned=poison)
    _step_inputs(rng, wl)
    return wl


def make_lowhead(seed: int = 4, poison: bool = True, batch: int = 256, lo: int = 512, hi: int = 4096) -> Workload:
    """16-head bandwidth case.  Draw order: context lengths, block permutation,
    pool, q, step inputs.  Each sequence appends one token at position L_b and
    attends over L_b + 1 tokens."""
    rng = np.random.default_rng(seed)
    ctx = rng.integers(lo, hi, size=batch, endpoint=True).astype(np.int32)
    seqlens = (ctx + 1).astype(np.int32)
    bt, nb, ss, pool, q = _v3_common(rng, batch, 16, seqlens, True, poison)
    wl = Workload(name="lowhead", seed=seed, n_heads=16, d_head=128, d_v=128, d_latent=512, d_rope=64,
                  rope_base=10000.0, scale=1.0 / math.sqrt(192), batch=batch, seqlens=seqlens,
                  block_tokens=64, paged=True, block_table=bt, num_blocks=nb, seq_stride=ss,
                  pool=pool, q=q, poisoned=poison)
    _step_inputs(rng, wl)
    if poison:
        # the slot the append fills starts out poisoned, so a missed write shows up
        for b, L in enumerate(ctx):
            pool[bt[b, int(L) // 64], int(L) % 64, :] = BF16_QNAN
    return wl


def make_random(seed: int, n_heads: int, d_latent: int, d_rope: int, seqlens, d_head: int = 32,
                d_v: Optional[int] = None, paged: bool = True, block_tokens: int = 64,
                poison: bool = True, d_model: int = 128, q_std: float = 1.0,
                rope_base: float = 10000.0) -> Workload:
    """Small random case for sweeps over ragged lengths and shapes.

    Draw order: block permutation (paged), pool, q, then the step inputs.
    """
    rng = np.random.default_rng(seed)
    seqlens = np.asarray(seqlens, dtype=np.int32)
    B = len(seqlens)
    D = d_latent + d_rope
    if paged:
        bt, nb = _paged_layout(rng, seqlens, block_tokens)
        pool = _normal_bf16(rng, (nb, block_tokens, D))
        if poison:
            _poison_paged(pool, bt, seqlens, block_tokens)
        ss = 0
    else:
        bt, nb = None, 0
        ss = max(1, int(seqlens.max()) + 3)
        pool = _normal_bf16(rng, (B, ss, D))
        if poison:
            for b, L in enumerate(seqlens):
                pool[b, int(L):, :] = BF16_QNAN
    q = _normal_bf16(rng, (B, n_heads, D), q_std)
    wl = Workload(name="random", seed=seed, n_heads=n_heads, d_head=d_head, d_v=d_v or d_head,
                  d_latent=d_latent, d_rope=d_rope, rope_base=rope_base,
                  scale=1.0 / math.sqrt(d_head + d_rope), batch=B, seqlens=seqlens,
                  block_tokens=block_tokens, paged=paged, block_table=bt, num_blocks=nb,
                  seq_stride=ss, pool=pool, q=q, poisoned=poison)
    _step_inputs(rng, wl, d_model=d_model)
    return wl


def make(name: str, poison: bool = True) -> Workload:
    """Build one of the five named benchmark workloads with its default seed."""
    seed = CONFIG_SEEDS[name]
    return {"tiny": make_tiny, "v3": make_v3, "paged": make_paged, "long": make_long,
            "lowhead": make_lowhead}[name](seed=seed, poison=poison)

"""fp64 reference for the MLA decode path (TEST INFRASTRUCTURE ONLY).

Sources (pages on Multi-head Latent Attention):
  [V2]  "DeepSeek-V2 MLA visual reading" (syt-nju.github.io): low-rank joint
        compression, absorption, decoupled RoPE, cache-size table.
  [V3c] "MLA latent attention and the KV cache" (ai.saiita.com.cn): DeepSeek-V3
        per-token cache arithmetic.
  [STR] "MLA模型结构详解：从公式到推理代码" (gentlecold.top): equations, the naive
        and absorbed inference branches, the worked decode example.
  [KVS] "给 KV Cache 瘦身：MQA·GQA·MLA" (bilibili-notes): 576 = 512 + 64, ~70 KB.

Everything here is fp64 on bf16 inputs widened exactly.  Nothing is blocked,
fused or reordered beyond what the equations state; softmax is the plain
two-pass form (max, then exp-sum), never online.

Readings the pages leave open (each also listed in the design notes):
  * RoPE pairs are interleaved (x[2i], x[2i+1]) rotated counter-clockwise by
    pos * base^(-2i/d_R); the pages only say "rotation R_t by position".
  * Positions are 0-based; the decode token at position L-1 is written to the
    cache first and attends to itself (the [STR] worked example writes slot
    start_pos, then attends to start_pos + 1 tokens).
  * No norm of the latent before caching: norm(...) appears only in the [STR]
    pseudocode, not in its equations, and no gain vector is given.
  * A cache row is [c^KV (d_c) | RoPE(k^R) (d_R)]; a latent query is
    [q~ (d_c) | RoPE(q^R) (d_R)], in the order [STR] splits kv_and_pe and q.
  * A sequence with no visible tokens yields z = 0 and lse = -inf.

Parity pins (tests/test_oracle_*.py): naive route == absorbed route,
brute-force loops on tiny cases, closed forms printed on the pages, softmax
special cases, RoPE as complex multiplication, bf16 rounding against torch.
"""
from __future__ import annotations

import math

import numpy as np

__all__ = [
    "bf16_to_f64", "round_bf16_bits", "rope", "project_q", "absorb_q", "append_rows",
    "append_cache", "gather_rows", "softmax_two_pass", "decode_latent", "decode_absorbed",
    "decode_naive", "decode_brute", "out_proj", "output_projection",
    "mla_cache_elems", "mha_cache_elems", "naive_mla_cache_elems", "KIB", "MIB", "GIB",
]

KIB, MIB, GIB = 1024, 1024 ** 2, 1024 ** 3


# ---------------------------------------------------------------- bf16 helpers
def bf16_to_f64(bits) -> np.ndarray:
    """Exact value of bf16 bit patterns as float64 (sign, 8-bit exponent, 7-bit fraction)."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.int64)
    sign = np.where(b & 0x8000, -1.0, 1.0)
    exp = (b >> 7) & 0xFF
    frac = (b & 0x7F).astype(np.float64)
    normal = sign * np.ldexp(1.0 + frac / 128.0, (exp - 127).astype(np.int64))
    sub = sign * np.ldexp(frac / 128.0, -126)
    out = np.where(exp == 0, sub, normal)
    out = np.where((exp == 0xFF) & (frac == 0), sign * np.inf, out)
    out = np.where((exp == 0xFF) & (frac != 0), np.nan, out)
    return out


def round_bf16_bits(x) -> np.ndarray:
    """Round float64 values to bf16 with round-to-nearest-even; uint16 bits.

    Works on the exact fp64 value (no intermediate float32 rounding): the
    value is scaled so one bf16 ulp becomes 1, rounded half-to-even, scaled back.
    """
    x = np.asarray(x, dtype=np.float64)
    out = np.empty(x.shape, dtype=np.uint16)
    flat, res = x.reshape(-1), out.reshape(-1)
    nan = np.isnan(flat)
    fin = np.isfinite(flat) & (flat != 0.0)
    _, e = np.frexp(np.where(fin, flat, 1.0))          # |x| in [2^(e-1), 2^e)
    ulp_exp = np.maximum(e - 8, -133)                   # 8 significant bits; subnormal floor
    q = np.ldexp(np.rint(np.ldexp(np.where(fin, flat, 0.0), -ulp_exp)), ulp_exp)
    q = np.where(fin, q, flat)                          # zeros and infinities pass through
    big = np.abs(q) >= 2.0 ** 128
    q = np.where(big, np.copysign(np.inf, q), q)
    with np.errstate(invalid="ignore", over="ignore"):
        f32 = np.where(nan, 0.0, q).astype(np.float32)
    res[:] = (f32.view(np.uint32) >> np.uint32(16)).astype(np.uint16)
    res[nan] = 0x7FC0
    return out


# ---------------------------------------------------------------- RoPE
def rope(x, pos, base: float = 10000.0) -> np.ndarray:
    """Decoupled RoPE on the last axis ([V2] section on decoupled RoPE; [STR]
    "RoPE 为什么要解耦": q^R = RoPE(W^QR c^Q), k^R = RoPE(W^KR h)).

    Pair i = (x[2i], x[2i+1]) is rotated by angle pos * base^(-2i/d_R).
    ``pos`` broadcasts against x.shape[:-1].
    """
    x = np.asarray(x, dtype=np.float64)
    d = x.shape[-1]
    assert d % 2 == 0
    i = np.arange(d // 2, dtype=np.float64)
    theta = base ** (-2.0 * i / d)
    ang = np.asarray(pos, dtype=np.float64)[..., None] * theta
    c, s = np.cos(ang), np.sin(ang)
    out = np.empty_like(x)
    out[..., 0::2] = x[..., 0::2] * c - x[..., 1::2] * s
    out[..., 1::2] = x[..., 0::2] * s + x[..., 1::2] * c
    return out


# ---------------------------------------------------------------- projections
def project_q(h, w_q, d_head: int):
    """Query projection of the tiny case: q_i = W^Q_i h, split [q^C (d_h) | q^R]
    in the order [STR] splits q into q_nope, q_pe.  h: [B, d]; w_q: [n_h, d_h+d_R, d]."""
    q = np.einsum("hkd,bd->bhk", bf16_to_f64(w_q), bf16_to_f64(h))
    return q[..., :d_head], q[..., d_head:]


def absorb_q(q_c, q_r, pos, w_uk, rope_base: float = 10000.0) -> np.ndarray:
    """Latent-space query ([STR] "为什么矩阵吸收很关键": q^C.(W^UK c) = (q^C W^UK).c;
    worked example step 4: q_nope absorbed to [.., 16, 512]; q_pe gets RoPE).

    q_c [B, n_h, d_h], q_r [B, n_h, d_R] (before RoPE), pos [B],
    w_uk [n_h, d_h, d_c] (k^C_i = W^UK_i c).  Returns [B, n_h, d_c + d_R] fp64:
    [W^UK_i^T q^C_i | RoPE(q^R_i, pos_b)].
    """
    qc = np.asarray(q_c, dtype=np.float64)
    qr = np.asarray(q_r, dtype=np.float64)
    W = np.asarray(w_uk, dtype=np.float64)
    q_lat = np.einsum("hkc,bhk->bhc", W, qc)
    q_rot = rope(qr, np.asarray(pos)[:, None], rope_base)
    return np.concatenate([q_lat, q_rot], axis=-1)


def append_rows(h, w_dkv_kr, pos, d_latent: int, rope_base: float = 10000.0) -> np.ndarray:
    """New cache rows before rounding ([STR] c_t^KV = W^DKV h_t; wkv_a(x) gives
    kv_latent and k_pe, then RoPE(k_pe)).  h [T, d], w [d_c + d_R, d] -> [T, d_c + d_R]."""
    rows = np.asarray(h, dtype=np.float64) @ np.asarray(w_dkv_kr, dtype=np.float64).T
    rows[:, d_latent:] = rope(rows[:, d_latent:], np.asarray(pos), rope_base)
    return rows


def _row_index(block_table, b: int, t: np.ndarray, block_tokens: int, seq_stride: int) -> np.ndarray:
    """Flat pool row of token t of sequence b (paged: block table; else contiguous)."""
    t = np.asarray(t, dtype=np.int64)
    if block_table is None:
        return b * seq_stride + t
    return np.asarray(block_table)[b, t // block_tokens].astype(np.int64) * block_tokens + t % block_tokens


def append_cache(pool_bits, h, w_dkv_kr, seq_idx, pos, d_latent: int, block_table=None,
                 block_tokens: int = 64, seq_stride: int = 0, rope_base: float = 10000.0) -> np.ndarray:
    """Cache write ([STR] worked example step 3: kv_cache[:, start_pos] = kv_latent,
    pe_cache[:, start_pos] = k_pe).  Returns a copy of the pool (bf16 bits) with
    row pos[t] of sequence seq_idx[t] replaced by the bf16-rounded new row."""
    rows = round_bf16_bits(append_rows(bf16_to_f64(h), bf16_to_f64(w_dkv_kr), pos, d_latent, rope_base))
    out = np.array(pool_bits, copy=True)
    flat = out.reshape(-1, out.shape[-1])
    for t in range(rows.shape[0]):
        r = _row_index(block_table, int(seq_idx[t]), np.array([pos[t]]), block_tokens, seq_stride)[0]
        flat[r] = rows[t]
    return out


def gather_rows(pool_bits, b: int, seqlen: int, block_table=None, block_tokens: int = 64,
                seq_stride: int = 0) -> np.ndarray:
    """The seqlen visible cache rows of sequence b as fp64 [seqlen, d_c + d_R]."""
    flat = np.asarray(pool_bits).reshape(-1, np.asarray(pool_bits).shape[-1])
    idx = _row_index(block_table, b, np.arange(seqlen), block_tokens, seq_stride)
    return bf16_to_f64(flat[idx])


# ---------------------------------------------------------------- attention
def softmax_two_pass(s: np.ndarray):
    """Softmax over the last axis: max pass, then exp-sum pass.  Returns (a, lse)."""
    m = s.max(axis=-1, keepdims=True)
    e = np.exp(s - m)
    l = e.sum(axis=-1, keepdims=True)
    return e / l, (m + np.log(l))[..., 0]


def decode_latent(q_lat, rows, scale: float, d_latent: int):
    """Absorbed decode for one sequence ([STR] worked example steps 4-5):
    score = (q~ . kv_cache + q_pe . pe_cache) * scale, softmax, z = A . kv_cache.

    q_lat [n_h, d_c + d_R] fp64, rows [L, d_c + d_R] fp64.
    Returns z [n_h, d_c], lse [n_h] (natural log of the softmax denominator,
    including the running max).  L == 0 gives z = 0, lse = -inf.
    """
    q_lat = np.asarray(q_lat, dtype=np.float64)
    n_h = q_lat.shape[0]
    if rows.shape[0] == 0:
        return np.zeros((n_h, d_latent)), np.full(n_h, -np.inf)
    c, k_r = rows[:, :d_latent], rows[:, d_latent:]
    score_c = q_lat[:, :d_latent] @ c.T            # einsum over the latent
    score_r = q_lat[:, d_latent:] @ k_r.T          # einsum over the RoPE key
    a, lse = softmax_two_pass((score_c + score_r) * scale)
    return a @ c, lse


def decode_absorbed(q_c, q_r_rot, w_uk, w_uv, rows, scale: float, d_latent: int):
    """Route B, absorbed branch ([STR] pseudocode, optimised branch):
    q~ = q^C W^UK, score = q~.c + q^R.k^R, z = A c, o = z W^UV.  One sequence.
    q_c [n_h, d_h], q_r_rot [n_h, d_R] (RoPE applied), w_uk [n_h, d_h, d_c],
    w_uv [n_h, d_v, d_c].  Returns o [n_h, d_v], z [n_h, d_c], lse [n_h]."""
    q_lat = np.einsum("hkc,hk->hc", w_uk, q_c)
    z, lse = decode_latent(np.concatenate([q_lat, q_r_rot], axis=-1), rows, scale, d_latent)
    return out_proj(z[None], w_uv)[0], z, lse


def decode_naive(q_c, q_r_rot, w_uk, w_uv, rows, scale: float, d_latent: int):
    """Route A, naive branch ([STR] pseudocode naive branch; equations
    k^C = W^UK c, v^C = W^UV c, q_i = [q^C_i; q^R_i], k_i = [k^C_i; k^R]):
    recover every head's full key and value, then standard softmax attention.
    Returns o [n_h, d_v], lse [n_h]."""
    n_h = q_c.shape[0]
    d_v = w_uv.shape[1]
    L = rows.shape[0]
    if L == 0:
        return np.zeros((n_h, d_v)), np.full(n_h, -np.inf)
    c, k_r = rows[:, :d_latent], rows[:, d_latent:]
    o = np.empty((n_h, d_v))
    lse = np.empty(n_h)
    for i in range(n_h):
        k_c = c @ w_uk[i].T                        # [L, d_h]
        v_c = c @ w_uv[i].T                        # [L, d_v]
        k = np.concatenate([k_c, k_r], axis=1)     # k_{j,i} = [k^C_{j,i}; k^R_j]
        q = np.concatenate([q_c[i], q_r_rot[i]])   # q_i = [q^C_i; q^R_i]
        a, lse[i] = softmax_two_pass((k @ q) * scale)
        o[i] = a @ v_c
    return o, lse


def decode_brute(q_lat, rows, scale: float, d_latent: int):
    """Pure-Python loops over heads, tokens and dims (tiny cases only)."""
    q_lat = [[float(v) for v in r] for r in np.asarray(q_lat)]
    rows = [[float(v) for v in r] for r in np.asarray(rows)]
    D = len(q_lat[0])
    zs, lses = [], []
    for qh in q_lat:
        if not rows:
            zs.append([0.0] * d_latent)
            lses.append(-math.inf)
            continue
        s = []
        for r in rows:
            acc = 0.0
            for k in range(D):
                acc += qh[k] * r[k]
            s.append(acc * scale)
        m = max(s)
        w = [math.exp(v - m) for v in s]
        tot = sum(w)
        z = [0.0] * d_latent
        for wj, r in zip(w, rows):
            for k in range(d_latent):
                z[k] += wj / tot * r[k]
        zs.append(z)
        lses.append(m + math.log(tot))
    return np.array(zs), np.array(lses)


def out_proj(z, w_uv) -> np.ndarray:
    """Value up-projection after the latent sum ([STR] sum_j A_j W^UV c_j =
    W^UV sum_j A_j c_j; worked example step 5: o = z . W_UV -> [.., 16, 128]).
    z [B, n_h, d_c], w_uv [n_h, d_v, d_c] -> o [B, n_h, d_v]."""
    return np.einsum("hvc,bhc->bhv", np.asarray(w_uv, dtype=np.float64), np.asarray(z, dtype=np.float64))


def output_projection(o, w_o) -> np.ndarray:
    """Flatten heads and apply W^O ([STR] worked example step 5: u [1, 1, 2048]).
    o [B, n_h, d_v], w_o [d, n_h * d_v] -> u [B, d]."""
    o = np.asarray(o, dtype=np.float64)
    return o.reshape(o.shape[0], -1) @ np.asarray(w_o, dtype=np.float64).T


# ---------------------------------------------------------------- closed forms
def mla_cache_elems(d_latent: int, d_rope: int, layers: int = 1) -> int:
    """Cached elements per token: (d_c + d_R) * l ([V2] cache table; [STR] d_c + d_h^R)."""
    return (d_latent + d_rope) * layers


def mha_cache_elems(n_heads: int, d_head: int, layers: int = 1) -> int:
    """Cached elements per token for MHA: 2 * n_h * d_h * l ([V2] cache table; [STR])."""
    return 2 * n_heads * d_head * layers


def naive_mla_cache_elems(n_heads: int, d_qk: int, d_v: int) -> int:
    """Per-layer elements when full K (d_qk) and V (d_v) are cached per head
    ([STR] worked example step 3: 16 * (192 + 128))."""
    return n_heads * (d_qk + d_v)

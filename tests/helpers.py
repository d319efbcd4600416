"""Shared test utilities: device upload of bf16 bit arrays and the parity metrics."""
from __future__ import annotations

import numpy as np
import torch

import oracle as orc

# GPU vs oracle tolerance for floating-point outputs (bf16 storage, fp32 accumulation):
# max|d| <= 1e-2 * max|ref|  and  sum|d| / sum|ref| <= 2e-3  (mean relative error, L1 form)
MAX_REL = 1e-2
MEAN_REL = 2e-3
# lse: both decode kernels round the softmax weights p_j = 2^(x_j - m) to bf16 for
# the value contraction and sum those same rounded weights into l, so that z is
# an exact convex combination of the weights the MMA used.  bf16 keeps 8
# significant bits: each weight carries a relative error of at most 2^-8, so
# l does too and |d lse| <= ln(1 + 2^-8) (~3.9e-3; ~1e-3 typical on a 2-token
# sequence, less on long ones where the errors average out).  The relative
# 1e-3 |lse| term is the allowance for fp32 score accumulation (576-term dot
# products, exp2 / log2) that held for every case at large |lse|.
LSE_ABS = float(np.log1p(2.0 ** -8))
LSE_REL = 1e-3


def bits_to_dev(bits: np.ndarray, device="cuda") -> torch.Tensor:
    """uint16 bf16 bit patterns -> torch.bfloat16 tensor on the device."""
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16))
    return t.to(device).view(torch.bfloat16)


def dev_to_bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def i32(a, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(np.asarray(a, dtype=np.int32))).to(device)


def err_stats(got: np.ndarray, ref: np.ndarray):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    d = np.abs(got - ref)
    max_rel = d.max() / max(np.abs(ref).max(), 1e-300)
    mean_rel = d.sum() / max(np.abs(ref).sum(), 1e-300)
    return float(max_rel), float(mean_rel)


def assert_close(got, ref, what: str, max_rel=MAX_REL, mean_rel=MEAN_REL):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    assert np.isfinite(got).all(), f"{what}: non-finite values"
    mx, mn = err_stats(got, ref)
    assert mx <= max_rel and mn <= mean_rel, f"{what}: max_rel={mx:.3e} mean_rel={mn:.3e}"
    return mx, mn


def assert_lse_close(got, ref, what="lse", tol=LSE_ABS):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    both_inf = np.isneginf(got) & np.isneginf(ref)
    with np.errstate(invalid="ignore"):
        d = np.where(both_inf, 0.0, np.abs(got - ref))
    assert np.all(d <= tol + LSE_REL * np.abs(np.where(both_inf, 0.0, ref))), \
        f"{what}: max |d| = {np.nanmax(d):.3e}"


def ulp_diff_bf16(a_bits: np.ndarray, b_bits: np.ndarray) -> np.ndarray:
    """Distance in bf16 ulps between two bf16 arrays (same-sign finite values)."""
    def key(b):
        b = b.astype(np.int32)
        return np.where(b & 0x8000, -(b & 0x7FFF), b)
    return np.abs(key(a_bits) - key(b_bits))


def oracle_decode(wl, q_lat_f64, pool_bits, seqlens, heads=None, batches=None):
    """Oracle z, lse for the chosen (batch, head) subset; q_lat_f64 [B, n_h, D]."""
    B = len(seqlens)
    batches = range(B) if batches is None else batches
    zs, ls = {}, {}
    for b in batches:
        rows = orc.gather_rows(pool_bits, b, int(seqlens[b]), wl.block_table, wl.block_tokens, wl.seq_stride)
        qh = q_lat_f64[b] if heads is None else q_lat_f64[b][heads]
        z, lse = orc.decode_latent(qh, rows, wl.scale, wl.d_latent)
        zs[b], ls[b] = z, lse
    return zs, ls


def bf16_ulp(x: np.ndarray) -> np.ndarray:
    """Spacing of bf16 values at |x| (8 significant bits, subnormal floor 2^-133)."""
    ax = np.abs(np.asarray(x, dtype=np.float64))
    _, e = np.frexp(np.where(ax > 0, ax, 1.0))
    return np.ldexp(1.0, np.maximum(e - 8, -133))


# fp32 accumulation allowance for a bf16 GEMM output, relative to sum_k |x_k w_k|:
# sqrt(K) * 2^-24 is the typical random-walk error at K = 7168 (~5e-6); 2^-14
# leaves a 10x margin and is still far below what a wrong index or term gives.
ACC_REL = 2.0 ** -14


def assert_bf16_gemm(got_bits, exact, abs_terms, what: str, acc_rel=ACC_REL, frac_1ulp=0.99):
    """bf16 output of an fp32-accumulated contraction vs its exact fp64 value:
    |got - exact| <= half a bf16 ulp + acc_rel * sum|terms|, elementwise, and at
    least `frac_1ulp` of the elements within 1 ulp of round-to-nearest(exact)."""
    got = orc.bf16_to_f64(got_bits)
    exact = np.asarray(exact, dtype=np.float64)
    bound = 0.5 * np.maximum(bf16_ulp(got), bf16_ulp(exact)) + acc_rel * np.asarray(abs_terms)
    err = np.abs(got - exact)
    bad = ~(err <= bound)
    assert not bad.any(), f"{what}: {bad.sum()} elements beyond the bound; worst excess " \
                          f"{np.max(err - bound):.3e}"
    near = ulp_diff_bf16(np.asarray(got_bits), orc.round_bf16_bits(exact)) <= 1
    assert near.mean() >= frac_1ulp, f"{what}: only {near.mean():.4f} within 1 ulp"

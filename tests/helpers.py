"""Shared test utilities: device upload of bf16 bit arrays and the parity metrics."""
from __future__ import annotations

import numpy as np
import torch

import oracle as orc

# GPU vs oracle tolerance for floating-point outputs (bf16 storage, fp32 accumulation):
#   max|d| <= 1e-2 * max|ref| on every output row (one (sequence, head) vector of the
#   last axis), and sum|d| / sum|ref| <= 2e-3 (mean relative error, L1 form) on every
#   sequence's output.  Batch-wide figures would let a long sequence's error hide
#   behind a short sequence's larger magnitude.  The mean bound is not applied per
#   row: the value contraction multiplies bf16-rounded softmax weights, and a row
#   whose weight sits on two tokens carries a relative error of 0.5 |e1 - e2| with
#   |e| up to 2^-8 (bf16 round-to-nearest), i.e. up to ~3.9e-3 on that row alone.
MAX_REL = 1e-2
MEAN_REL = 2e-3
# lse = log sum_j exp(s_j): the kernels sum the fp32 weights into it, so the only
# errors are fp32 score accumulation and exp2 / log2 rounding.
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
    """(max_rel, mean_rel) of the whole array, batch-wide."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    d = np.abs(got - ref)
    max_rel = d.max() / max(np.abs(ref).max(), 1e-300)
    mean_rel = d.sum() / max(np.abs(ref).sum(), 1e-300)
    return float(max_rel), float(mean_rel)


def row_stats(got: np.ndarray, ref: np.ndarray):
    """Per-row (max_rel, mean_rel) arrays; a row is one vector of the last axis."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    g2 = got.reshape(-1, got.shape[-1])
    r2 = ref.reshape(-1, ref.shape[-1])
    d = np.abs(g2 - r2)
    a = np.abs(r2)
    max_rel = d.max(axis=1) / np.maximum(a.max(axis=1), 1e-300)
    mean_rel = d.sum(axis=1) / np.maximum(a.sum(axis=1), 1e-300)
    return max_rel, mean_rel


def assert_close(got, ref, what: str, max_rel=MAX_REL, mean_rel=MEAN_REL):
    """max bound on every row (last axis); mean bound on every sequence (the leading
    axis of a [sequence, head, ...] array, or the whole array when it holds one
    sequence's [head, ...] output)."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    assert np.isfinite(got).all(), f"{what}: non-finite values"
    mx, _ = row_stats(got, ref)
    units = got.shape[0] if got.ndim >= 3 else 1
    d = np.abs(got - ref).reshape(units, -1)
    a = np.abs(ref).reshape(units, -1)
    mn = d.sum(axis=1) / np.maximum(a.sum(axis=1), 1e-300)
    bad_rows, bad_units = mx > max_rel, mn > mean_rel
    if bad_rows.any() or bad_units.any():
        r = int(np.argmax(mx))
        u = int(np.argmax(mn))
        raise AssertionError(
            f"{what}: {int(bad_rows.sum())} of {bad_rows.size} rows beyond the max bound "
            f"(worst row {tuple(int(v) for v in np.unravel_index(r, got.shape[:-1]))}: max_rel={mx[r]:.3e}); "
            f"{int(bad_units.sum())} of {units} sequences beyond the mean bound (worst sequence {u}: "
            f"mean_rel={mn[u]:.3e})")
    return float(mx.max()), float(mn.max())


def assert_lse_close(got, ref, what="lse", rel=LSE_REL):
    """|d lse| <= rel * max(1, |lse|) elementwise; -inf (empty sequence) must match."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    both_inf = np.isneginf(got) & np.isneginf(ref)
    with np.errstate(invalid="ignore"):
        d = np.where(both_inf, 0.0, np.abs(got - ref))
    bound = rel * np.maximum(1.0, np.abs(np.where(both_inf, 0.0, ref)))
    ok = d <= bound
    assert ok.all(), f"{what}: {int((~ok).sum())} values beyond 1e-3 max(1,|lse|); max |d| = {np.nanmax(d):.3e}"


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

"""GPU parity: the CUDA library (through its C ABI) against the fp64 oracle."""
import math

import numpy as np
import pytest
import torch

import mla_inputs as mi
import oracle as orc
from helpers import (assert_bf16_gemm, assert_close, assert_lse_close, bits_to_dev, dev_to_bits, i32,
                     oracle_decode, ulp_diff_bf16)


def append_abs_terms(h_bits, w_bits, d_latent):
    """sum_k |h_k w_k| per output element of the append projection; the RoPE
    pair (2i, 2i+1) mixes the two sums of its pair."""
    a = np.abs(orc.bf16_to_f64(h_bits)) @ np.abs(orc.bf16_to_f64(w_bits)).T
    r = a[:, d_latent:]
    pair = r[:, 0::2] + r[:, 1::2]
    a[:, d_latent::2] = pair
    a[:, d_latent + 1::2] = pair
    return a

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mla():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from __graft_entry__ import build
    build()
    import mla_latent_kv_76_b300 as m
    return m


def run_decode(mla, wl, q_bits=None, pool=None, num_workers=0, flags=0, z_fp32=True, seqlens=None,
               block_table=None):
    dims = mla.Dims.of(wl)
    q = bits_to_dev(wl.q if q_bits is None else q_bits)
    pool = bits_to_dev(wl.pool) if pool is None else pool
    bt = block_table if block_table is not None else (i32(wl.block_table) if wl.paged else None)
    sl = i32(wl.seqlens if seqlens is None else seqlens)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    z, lse = mla.mla_decode_attn(dims, q, pool, sl, wl.scale, block_table=bt, num_blocks=wl.num_blocks,
                                 seq_stride=wl.seq_stride, num_workers=num_workers, flags=flags,
                                 z_is_fp32=z_fp32, dev_status=status)
    torch.cuda.synchronize()
    return z.float().cpu().numpy(), lse.cpu().numpy(), mla.mla_read_status(status)


def check_decode(wl, z, lse, heads=None, batches=None):
    q64 = orc.bf16_to_f64(wl.q)
    zs, ls = oracle_decode(wl, q64, wl.pool, wl.seqlens, heads=heads, batches=batches)
    bs = sorted(zs)
    zg = np.stack([z[b] if heads is None else z[b][heads] for b in bs])
    lg = np.stack([lse[b] if heads is None else lse[b][heads] for b in bs])
    zr = np.stack([zs[b] for b in bs])
    lr = np.stack([ls[b] for b in bs])
    nonempty = np.array([wl.seqlens[b] > 0 for b in bs])
    if nonempty.any():
        assert_close(zg[nonempty], zr[nonempty], f"z[{wl.name}]")
    assert np.all(zg[~nonempty] == 0)
    assert_lse_close(lg, lr)


# ---------------------------------------------------------------- tiny case, whole chain
def test_tiny_chain(mla):
    wl = mi.make("tiny")
    dims = mla.Dims.of(wl)
    pool = bits_to_dev(wl.pool)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    mla.mla_append_cache(dims, bits_to_dev(wl.h), bits_to_dev(wl.w_dkv_kr), i32(wl.app_seq), i32(wl.app_pos),
                         pool, n_seqs=1, seq_stride=wl.seq_stride, dev_status=status)
    ref_pool = orc.append_cache(wl.pool, wl.h, wl.w_dkv_kr, wl.app_seq, wl.app_pos, wl.d_latent, None,
                                wl.block_tokens, wl.seq_stride, wl.rope_base)
    got_pool = dev_to_bits(pool)
    assert np.array_equal(got_pool[0, 129:], wl.pool[0, 129:])          # slack untouched (NaN)
    exact = orc.append_rows(orc.bf16_to_f64(wl.h), orc.bf16_to_f64(wl.w_dkv_kr), wl.app_pos, wl.d_latent,
                            wl.rope_base)
    assert_bf16_gemm(got_pool[0, :129], exact, append_abs_terms(wl.h, wl.w_dkv_kr, wl.d_latent), "append")
    # query: W^Q h of the decode token (oracle), rounded to bf16, absorbed on the GPU
    q_c, q_r = orc.project_q(wl.h[128:129], wl.w_q, wl.d_head)
    qc_b, qr_b = orc.round_bf16_bits(q_c), orc.round_bf16_bits(q_r)
    q = mla.mla_absorb_q(dims, bits_to_dev(qc_b), bits_to_dev(qr_b), i32(wl.q_pos), bits_to_dev(wl.w_uk))
    q_ref = orc.absorb_q(orc.bf16_to_f64(qc_b), orc.bf16_to_f64(qr_b), wl.q_pos, orc.bf16_to_f64(wl.w_uk),
                         wl.rope_base)
    assert_close(q.float().cpu().numpy(), q_ref, "q")
    status2 = torch.zeros(1, dtype=torch.int32, device="cuda")
    z, lse = mla.mla_decode_attn(dims, q, pool, i32(wl.seqlens), wl.scale, seq_stride=wl.seq_stride,
                                 dev_status=status2)
    o = mla.mla_out_proj(dims, z.to(torch.bfloat16), bits_to_dev(wl.w_uv))
    torch.cuda.synchronize()
    assert mla.mla_read_status(status) == 0 and mla.mla_read_status(status2) == 0
    rows = orc.gather_rows(ref_pool, 0, 129, None, 64, wl.seq_stride)
    q_rot = orc.rope(orc.bf16_to_f64(qr_b)[0], 128, wl.rope_base)
    o_ref, z_ref, lse_ref = orc.decode_absorbed(orc.bf16_to_f64(qc_b)[0], q_rot, orc.bf16_to_f64(wl.w_uk),
                                                orc.bf16_to_f64(wl.w_uv), rows, wl.scale, wl.d_latent)
    # the cache rows and query went through bf16 once more than the oracle's: compare
    # z against the oracle fed the GPU's own q and cache
    z_own, lse_own = orc.decode_latent(orc.bf16_to_f64(dev_to_bits(q))[0],
                                       orc.gather_rows(got_pool, 0, 129, None, 64, wl.seq_stride),
                                       wl.scale, wl.d_latent)
    assert_close(z.cpu().numpy()[0], z_own, "z (own inputs)")
    assert_lse_close(lse.cpu().numpy()[0], lse_own)
    assert_close(z.cpu().numpy()[0], z_ref, "z (chain)", mean_rel=5e-3)
    o_own = orc.out_proj(orc.bf16_to_f64(dev_to_bits(z.to(torch.bfloat16))), orc.bf16_to_f64(wl.w_uv))[0]
    assert_close(o.float().cpu().numpy()[0], o_own, "o (own z)")
    assert_close(o.float().cpu().numpy()[0], o_ref, "o (chain)", mean_rel=5e-3)


# ---------------------------------------------------------------- decode sweeps
CASES = [
    dict(n_heads=4, d_latent=64, d_rope=16, seqlens=[129], paged=False),
    dict(n_heads=16, d_latent=512, d_rope=64, seqlens=[1, 63, 64, 65, 127, 128, 129, 1000], paged=True),
    dict(n_heads=20, d_latent=128, d_rope=16, seqlens=[300, 5, 0, 77], paged=True),
    dict(n_heads=8, d_latent=256, d_rope=32, seqlens=[640, 1, 2000], paged=False),
    dict(n_heads=128, d_latent=512, d_rope=64, seqlens=[1, 65, 700, 2048], paged=True),
    dict(n_heads=128, d_latent=512, d_rope=64, seqlens=[4096, 4096], paged=False),
    dict(n_heads=16, d_latent=512, d_rope=64, seqlens=[3000, 5, 0, 129, 64, 4097], paged=False),
]


@pytest.mark.parametrize("case", range(len(CASES)))
@pytest.mark.parametrize("workers", [0, 1, 3, 7])
def test_decode_matches_oracle(mla, case, workers):
    c = CASES[case]
    wl = mi.make_random(1000 + case, c["n_heads"], c["d_latent"], c["d_rope"], c["seqlens"], paged=c["paged"])
    z, lse, st = run_decode(mla, wl, num_workers=workers)
    assert st == 0
    check_decode(wl, z, lse)


def test_decode_bf16_output(mla):
    wl = mi.make_random(77, 128, 512, 64, [333, 2048, 64], paged=True)
    z, lse, st = run_decode(mla, wl, z_fp32=False)
    assert st == 0
    q64 = orc.bf16_to_f64(wl.q)
    zs, _ = oracle_decode(wl, q64, wl.pool, wl.seqlens)
    # bf16 storage of z adds up to half an ulp per element on top of the fp32 result
    assert_close(z, np.stack([zs[b] for b in range(3)]), "z bf16", mean_rel=3e-3)


def test_paged_and_contiguous_are_bit_identical(mla):
    wl = mi.make_random(5, 128, 512, 64, [1, 64, 65, 1000, 3000], paged=True)
    B, D = wl.batch, wl.row_dim
    S = int(wl.seqlens.max())
    cont = np.full((B, S, D), mi.BF16_QNAN, dtype=np.uint16)
    flat = wl.pool.reshape(-1, D)
    for b, L in enumerate(wl.seqlens):
        t = np.arange(L)
        cont[b, :L] = flat[wl.block_table[b, t // 64] * 64 + t % 64]
    wc = mi.make_random(5, 128, 512, 64, wl.seqlens, paged=False)
    wc.pool, wc.q, wc.seq_stride = cont, wl.q, S
    for workers in (0, 3):
        zp, lp, s1 = run_decode(mla, wl, num_workers=workers)
        zc, lc, s2 = run_decode(mla, wc, num_workers=workers)
        assert s1 == 0 and s2 == 0
        assert np.array_equal(zp.view(np.uint32), zc.view(np.uint32))
        assert np.array_equal(lp.view(np.uint32), lc.view(np.uint32))


def test_repeat_runs_are_bit_identical(mla):
    wl = mi.make_random(6, 128, 512, 64, [777, 4096], paged=True)
    z1, l1, _ = run_decode(mla, wl)
    z2, l2, _ = run_decode(mla, wl)
    assert np.array_equal(z1.view(np.uint32), z2.view(np.uint32))
    assert np.array_equal(l1.view(np.uint32), l2.view(np.uint32))


def test_split_count_does_not_change_the_result(mla):
    """Every split-KV partition gives the oracle's answer.  (They differ from one
    another only through the bf16 rounding of the softmax weights, which depends
    on each split's running max.)"""
    wl = mi.make_random(7, 16, 512, 64, [5000, 17, 2222], paged=True)
    q64 = orc.bf16_to_f64(wl.q)
    zs, ls = oracle_decode(wl, q64, wl.pool, wl.seqlens)
    zr = np.stack([zs[b] for b in range(3)])
    lr = np.stack([ls[b] for b in range(3)])
    for w in (1, 2, 5, 13, 64, 200):
        z, lse, st = run_decode(mla, wl, num_workers=w)
        assert st == 0
        assert_close(z, zr, f"z workers={w}")
        assert_lse_close(lse, lr)


def test_zero_query_gives_the_mean_of_visible_rows(mla):
    """Uniform weights: any leak from slack (NaN), a wrong length or a wrong
    block changes the mean."""
    wl = mi.make_random(8, 16, 512, 64, [1, 63, 64, 65, 300], paged=True)
    wl.q = np.zeros_like(wl.q)
    z, lse, st = run_decode(mla, wl, num_workers=3)
    assert st == 0
    for b, L in enumerate(wl.seqlens):
        rows = orc.gather_rows(wl.pool, b, int(L), wl.block_table, 64, 0)
        want = rows[:, :wl.d_latent].mean(0)
        assert np.allclose(z[b], want[None, :], rtol=0, atol=1e-5 * max(1.0, np.abs(want).max()))
        assert np.allclose(lse[b], math.log(L), atol=1e-5)


def test_out_of_range_inputs_are_reported_not_read(mla):
    wl = mi.make_random(9, 16, 512, 64, [100, 200, 50], paged=True)
    # a sequence longer than its table's capacity counts as empty and is reported
    sl = wl.seqlens.copy()
    sl[1] = wl.max_blocks * 64 + 1
    z, lse, st = run_decode(mla, wl, seqlens=sl)
    assert st == 6 and np.all(z[1] == 0) and np.all(np.isneginf(lse[1]))
    q64 = orc.bf16_to_f64(wl.q)
    zs, _ = oracle_decode(wl, q64, wl.pool, wl.seqlens, batches=[0, 2])
    assert_close(np.stack([z[0], z[2]]), np.stack([zs[0], zs[2]]), "z other sequences")
    # a block id outside the pool is not dereferenced
    bt = wl.block_table.copy()
    bt[0, 0] = wl.num_blocks + 5
    z, lse, st = run_decode(mla, wl, block_table=i32(bt))
    assert st == 6 and np.isfinite(z).all()


# ---------------------------------------------------------------- append / absorb / out-projection
def test_append_identity_weights_is_bit_exact(mla):
    """W = I (576 x 576), h rows that encode (sequence, position), zero RoPE
    inputs: every written row must equal its h row bit for bit, at the slot the
    block table names, and no other slot may change."""
    D, d_c = 576, 512
    wl = mi.make_random(10, 16, d_c, 64, [70, 5, 130, 64], paged=True, d_model=D)
    seq = np.array([0, 0, 1, 2, 2, 2, 3, 3], dtype=np.int32)
    pos = np.array([0, 69, 4, 63, 64, 129, 0, 63], dtype=np.int32)
    h = np.zeros((len(seq), D))
    h[:, 0], h[:, 1] = seq + 1, pos + 1
    h[:, 2:d_c] = (np.arange(2, d_c) % 64) / 8.0
    hb = orc.round_bf16_bits(h)
    w = orc.round_bf16_bits(np.eye(D))
    dims = mla.Dims(16, 32, 32, d_c, 64, 64, 10000.0)
    pool = bits_to_dev(wl.pool)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    mla.mla_append_cache(dims, bits_to_dev(hb), bits_to_dev(w), i32(seq), i32(pos), pool, n_seqs=4,
                         block_table=i32(wl.block_table), num_blocks=wl.num_blocks, dev_status=status)
    torch.cuda.synchronize()
    assert mla.mla_read_status(status) == 0
    got = dev_to_bits(pool)
    want = orc.append_cache(wl.pool, hb, w, seq, pos, d_c, wl.block_table, 64, 0)
    got[got == 0x8000] = 0
    want[want == 0x8000] = 0
    assert np.array_equal(got, want)


def test_append_values_and_bounds(mla):
    wl = mi.make("lowhead")
    dims = mla.Dims.of(wl)
    pool = bits_to_dev(wl.pool)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    mla.mla_append_cache(dims, bits_to_dev(wl.h), bits_to_dev(wl.w_dkv_kr), i32(wl.app_seq), i32(wl.app_pos),
                         pool, n_seqs=wl.batch, block_table=i32(wl.block_table), num_blocks=wl.num_blocks,
                         dev_status=status)
    torch.cuda.synchronize()
    assert mla.mla_read_status(status) == 0
    got = dev_to_bits(pool)
    want = orc.append_cache(wl.pool, wl.h, wl.w_dkv_kr, wl.app_seq, wl.app_pos, wl.d_latent, wl.block_table,
                            64, 0, wl.rope_base)
    changed = np.any(want != wl.pool, axis=-1)
    assert changed.sum() == wl.batch
    assert np.array_equal(got[~changed], want[~changed])                  # nothing else touched
    flat_idx = wl.block_table[wl.app_seq, wl.app_pos // 64].astype(np.int64) * 64 + wl.app_pos % 64
    got_rows = got.reshape(-1, wl.row_dim)[flat_idx]
    exact = orc.append_rows(orc.bf16_to_f64(wl.h), orc.bf16_to_f64(wl.w_dkv_kr), wl.app_pos, wl.d_latent,
                            wl.rope_base)
    assert_bf16_gemm(got_rows, exact, append_abs_terms(wl.h, wl.w_dkv_kr, wl.d_latent), "append")
    # out-of-range position / sequence: skipped and reported
    bad_pos = wl.app_pos.copy()
    bad_pos[0] = wl.max_blocks * 64
    bad_seq = wl.app_seq.copy()
    bad_seq[1] = wl.batch
    before = dev_to_bits(pool)
    status.zero_()
    mla.mla_append_cache(dims, bits_to_dev(wl.h[:2]), bits_to_dev(wl.w_dkv_kr), i32(bad_seq[:2]),
                         i32(bad_pos[:2]), pool, n_seqs=wl.batch, block_table=i32(wl.block_table),
                         num_blocks=wl.num_blocks, dev_status=status)
    torch.cuda.synchronize()
    assert mla.mla_read_status(status) == 6
    assert np.array_equal(dev_to_bits(pool), before)


@pytest.mark.parametrize("n_tok,paged", [(1, True), (7, False), (16, True), (31, False), (32, True), (33, False),
                                         (100, True), (128, False), (129, True), (256, True), (300, False)])
def test_append_at_model_width(mla, n_tok, paged):
    """d_model = 7168 (the DeepSeek-V3 hidden size), the tensor-core kernel
    (cluster split of d_model): one tile for up to 32 tokens, tiles of 128
    tokens beyond (a partial last tile included).  Written rows against the
    fp64 oracle, every other row untouched."""
    rng = np.random.default_rng(100 + n_tok)
    lens = rng.integers(1, 700, size=n_tok)
    wl = mi.make_random(200 + n_tok, 4, 512, 64, lens, paged=paged, poison=False, d_model=7168)
    dims = mla.Dims.of(wl)
    pool = bits_to_dev(wl.pool)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    mla.mla_append_cache(dims, bits_to_dev(wl.h), bits_to_dev(wl.w_dkv_kr), i32(wl.app_seq), i32(wl.app_pos),
                         pool, n_seqs=wl.batch, block_table=i32(wl.block_table) if paged else None,
                         num_blocks=wl.num_blocks, seq_stride=wl.seq_stride, dev_status=status)
    torch.cuda.synchronize()
    assert mla.mla_read_status(status) == 0
    got = dev_to_bits(pool).reshape(-1, wl.row_dim)
    want = orc.append_cache(wl.pool, wl.h, wl.w_dkv_kr, wl.app_seq, wl.app_pos, wl.d_latent,
                            wl.block_table if paged else None, 64, wl.seq_stride, wl.rope_base).reshape(-1, wl.row_dim)
    if paged:
        flat = wl.block_table[wl.app_seq, wl.app_pos // 64].astype(np.int64) * 64 + wl.app_pos % 64
    else:
        flat = wl.app_seq.astype(np.int64) * wl.seq_stride + wl.app_pos
    others = np.ones(got.shape[0], dtype=bool)
    others[flat] = False
    assert np.array_equal(got[others], want[others])
    exact = orc.append_rows(orc.bf16_to_f64(wl.h), orc.bf16_to_f64(wl.w_dkv_kr), wl.app_pos, wl.d_latent,
                            wl.rope_base)
    assert_bf16_gemm(got[flat], exact, append_abs_terms(wl.h, wl.w_dkv_kr, wl.d_latent), "append")


@pytest.mark.parametrize("B", [1, 16, 40, 256])
def test_absorb_and_out_proj(mla, B):
    rng = np.random.default_rng(B)
    n_h, d_h, d_c, d_R, d_v = 16, 128, 512, 64, 128
    qc = mi.f32_to_bf16_bits(rng.standard_normal((B, n_h, d_h)).astype(np.float32))
    qr = mi.f32_to_bf16_bits(rng.standard_normal((B, n_h, d_R)).astype(np.float32))
    wuk = mi.f32_to_bf16_bits((rng.standard_normal((n_h, d_h, d_c)) / math.sqrt(d_c)).astype(np.float32))
    wuv = mi.f32_to_bf16_bits((rng.standard_normal((n_h, d_v, d_c)) / math.sqrt(d_c)).astype(np.float32))
    pos = rng.integers(0, 200000, size=B).astype(np.int32)
    z = mi.f32_to_bf16_bits(rng.standard_normal((B, n_h, d_c)).astype(np.float32))
    dims = mla.Dims(n_h, d_h, d_v, d_c, d_R, 64, 10000.0)
    q = mla.mla_absorb_q(dims, bits_to_dev(qc), bits_to_dev(qr), i32(pos), bits_to_dev(wuk))
    o = mla.mla_out_proj(dims, bits_to_dev(z), bits_to_dev(wuv))
    torch.cuda.synchronize()
    q_ref = orc.absorb_q(orc.bf16_to_f64(qc), orc.bf16_to_f64(qr), pos, orc.bf16_to_f64(wuk))
    o_ref = orc.out_proj(orc.bf16_to_f64(z), orc.bf16_to_f64(wuv))
    assert_close(q.float().cpu().numpy(), q_ref, "q")
    assert_close(o.float().cpu().numpy(), o_ref, "o")
    qc64, qr64 = orc.bf16_to_f64(qc), orc.bf16_to_f64(qr)
    abs_q = np.einsum("hkc,bhk->bhc", np.abs(orc.bf16_to_f64(wuk)), np.abs(qc64))
    pair = np.abs(qr64[..., 0::2]) + np.abs(qr64[..., 1::2])
    abs_r = np.repeat(pair, 2, axis=-1)
    assert_bf16_gemm(dev_to_bits(q), q_ref, np.concatenate([abs_q, abs_r], -1), "q")
    abs_o = np.einsum("hvc,bhc->bhv", np.abs(orc.bf16_to_f64(wuv)), np.abs(orc.bf16_to_f64(z)))
    assert_bf16_gemm(dev_to_bits(o), o_ref, abs_o, "o")


# ---------------------------------------------------------------- full-size workloads
@pytest.mark.parametrize("name", ["v3", "paged", "long"])
def test_full_size_decode(mla, name):
    wl = mi.make(name)
    z, lse, st = run_decode(mla, wl)
    assert st == 0
    heads = None if name != "long" else np.arange(0, 128, 9)
    check_decode(wl, z, lse, heads=heads)


def test_full_size_lowhead_chain(mla):
    """Append one token per sequence, then decode over L_b + 1 tokens (launch
    configuration of the 16-head bandwidth case)."""
    wl = mi.make("lowhead")
    dims = mla.Dims.of(wl)
    pool = bits_to_dev(wl.pool)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    mla.mla_append_cache(dims, bits_to_dev(wl.h), bits_to_dev(wl.w_dkv_kr), i32(wl.app_seq), i32(wl.app_pos),
                         pool, n_seqs=wl.batch, block_table=i32(wl.block_table), num_blocks=wl.num_blocks,
                         dev_status=status)
    z, lse, st = run_decode(mla, wl, pool=pool)
    assert st == 0 and mla.mla_read_status(status) == 0
    before = wl.pool
    wl.pool = dev_to_bits(pool)     # the oracle reads the cache the append produced ...
    flat_idx = wl.block_table[wl.app_seq, wl.app_pos // 64].astype(np.int64) * 64 + wl.app_pos % 64
    exact = orc.append_rows(orc.bf16_to_f64(wl.h), orc.bf16_to_f64(wl.w_dkv_kr), wl.app_pos, wl.d_latent,
                            wl.rope_base)
    assert_bf16_gemm(wl.pool.reshape(-1, wl.row_dim)[flat_idx], exact,
                     append_abs_terms(wl.h, wl.w_dkv_kr, wl.d_latent), "append")   # ... which is right
    keep = np.ones(wl.pool.shape[0] * 64, dtype=bool)
    keep[flat_idx] = False
    assert np.array_equal(wl.pool.reshape(-1, wl.row_dim)[keep], before.reshape(-1, wl.row_dim)[keep])
    check_decode(wl, z, lse)


def test_full_size_v3_step(mla):
    """The whole step at the DeepSeek-V3 shape, as the benchmark runs it:
    absorb -> append -> decode -> up-projection, compared with the oracle."""
    wl = mi.make("v3")
    dims = mla.Dims.of(wl)
    pool = bits_to_dev(wl.pool)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    q = mla.mla_absorb_q(dims, bits_to_dev(wl.q_c), bits_to_dev(wl.q_r), i32(wl.q_pos), bits_to_dev(wl.w_uk))
    mla.mla_append_cache(dims, bits_to_dev(wl.h), bits_to_dev(wl.w_dkv_kr), i32(wl.app_seq), i32(wl.app_pos),
                         pool, n_seqs=wl.batch, seq_stride=wl.seq_stride, dev_status=status)
    z, lse = mla.mla_decode_attn(dims, q, pool, i32(wl.seqlens), wl.scale, seq_stride=wl.seq_stride,
                                 z_is_fp32=False, dev_status=status)
    o = mla.mla_out_proj(dims, z, bits_to_dev(wl.w_uv))
    torch.cuda.synchronize()
    assert mla.mla_read_status(status) == 0
    ref_pool = orc.append_cache(wl.pool, wl.h, wl.w_dkv_kr, wl.app_seq, wl.app_pos, wl.d_latent, None, 64,
                                wl.seq_stride, wl.rope_base)
    q_ref = orc.absorb_q(orc.bf16_to_f64(wl.q_c), orc.bf16_to_f64(wl.q_r), wl.q_pos, orc.bf16_to_f64(wl.w_uk),
                         wl.rope_base)
    w_uv = orc.bf16_to_f64(wl.w_uv)
    og = o.float().cpu().numpy()
    o_ref = []
    for b in range(0, wl.batch, 5):
        rows = orc.gather_rows(ref_pool, b, int(wl.seqlens[b]), None, 64, wl.seq_stride)
        zr, _ = orc.decode_latent(q_ref[b], rows, wl.scale, wl.d_latent)
        o_ref.append(orc.out_proj(zr[None], w_uv)[0])
    assert_close(og[0::5], np.stack(o_ref), "o (full step)", mean_rel=6e-3)


# ---------------------------------------------------------------- tensor-core decode (128 heads, d_c 512, d_R 64)
TC_LENS = [0, 1, 63, 64, 65, 127, 128, 129, 191, 4097]


@pytest.mark.parametrize("workers", [0, 1, 2, 5, 40, 300])
def test_tc_decode_ragged_lengths(mla, workers):
    """Every tail length, an empty sequence, and more split-KV workers than
    tiles (idle CTA pairs); slack and unused blocks are NaN-poisoned."""
    wl = mi.make_random(2001, 128, 512, 64, TC_LENS, paged=True)
    z, lse, st = run_decode(mla, wl, num_workers=workers)
    assert st == 0
    check_decode(wl, z, lse)


def test_tc_decode_contiguous_ragged(mla):
    wl = mi.make_random(2002, 128, 512, 64, [4096, 1, 333, 0, 2049], paged=False)
    for workers in (0, 3):
        z, lse, st = run_decode(mla, wl, num_workers=workers)
        assert st == 0
        check_decode(wl, z, lse)


def test_tc_and_generic_paths_agree_with_the_oracle(mla):
    wl = mi.make_random(2003, 128, 512, 64, [700, 2048, 65], paged=True)
    zt, lt, s1 = run_decode(mla, wl)
    zg, lg, s2 = run_decode(mla, wl, flags=1)   # MLA_DECODE_FORCE_GENERIC
    assert s1 == 0 and s2 == 0
    check_decode(wl, zt, lt)
    check_decode(wl, zg, lg)


def test_tc_zero_query_gives_the_mean_of_visible_rows(mla):
    wl = mi.make_random(2004, 128, 512, 64, [1, 63, 64, 65, 300], paged=True)
    wl.q = np.zeros_like(wl.q)
    z, lse, st = run_decode(mla, wl, num_workers=3)
    assert st == 0
    for b, L in enumerate(wl.seqlens):
        rows = orc.gather_rows(wl.pool, b, int(L), wl.block_table, 64, 0)
        want = rows[:, :wl.d_latent].mean(0)
        assert np.allclose(z[b], want[None, :], rtol=0, atol=1e-5 * max(1.0, np.abs(want).max()))
        assert np.allclose(lse[b], math.log(L), atol=1e-5)


def test_tc_growing_scores_trigger_rescaling(mla):
    """Cache rows whose magnitude grows along the sequence make the running
    maximum climb tile after tile, so the output is rescaled many times."""
    wl = mi.make_random(2005, 128, 512, 64, [3000, 1500], paged=False)
    pool = orc.bf16_to_f64(wl.pool)
    grow = (1.0 + np.arange(pool.shape[1]) / 256.0)[None, :, None]
    wl.pool = orc.round_bf16_bits(np.where(np.isnan(pool), 0.0, pool) * grow)
    for workers in (0, 1):
        z, lse, st = run_decode(mla, wl, num_workers=workers)
        assert st == 0
        check_decode(wl, z, lse)


def test_tc_out_of_range_inputs_are_reported_not_read(mla):
    wl = mi.make_random(2006, 128, 512, 64, [100, 200, 50], paged=True)
    sl = wl.seqlens.copy()
    sl[1] = wl.max_blocks * 64 + 1
    z, lse, st = run_decode(mla, wl, seqlens=sl)
    assert st == 6 and np.all(z[1] == 0) and np.all(np.isneginf(lse[1]))
    q64 = orc.bf16_to_f64(wl.q)
    zs, _ = oracle_decode(wl, q64, wl.pool, wl.seqlens, batches=[0, 2])
    assert_close(np.stack([z[0], z[2]]), np.stack([zs[0], zs[2]]), "z other sequences")
    bt = wl.block_table.copy()
    bt[0, 0] = wl.num_blocks + 5
    z, lse, st = run_decode(mla, wl, block_table=i32(bt))
    assert st == 6 and np.isfinite(z).all()


# ---------------------------------------------------------------- batch limits
def _check_sampled(wl, z, lse, batches):
    for b in batches:
        L = int(wl.seqlens[b])
        if L == 0:
            assert np.all(z[b] == 0) and np.all(np.isneginf(lse[b]))
            continue
        rows = orc.gather_rows(wl.pool, b, L, wl.block_table, wl.block_tokens, wl.seq_stride)
        z_ref, lse_ref = orc.decode_latent(orc.bf16_to_f64(wl.q[b]), rows, wl.scale, wl.d_latent)
        assert_close(z[b], z_ref, f"z[{b}]")
        assert_lse_close(lse[b], lse_ref)


def test_tc_decode_at_its_batch_limit(mla):
    """1024 sequences, the most the tensor-core decode takes (each CTA holds the
    tile and plan prefixes of the whole batch in shared memory); ragged
    1..129 tokens, contiguous cache; sampled sequences against the oracle."""
    rng = np.random.default_rng(2100)
    wl = mi.make_random(2100, 128, 512, 64, rng.integers(1, 130, size=1024), paged=False)
    z, lse, st = run_decode(mla, wl)
    assert st == 0 and np.isfinite(z).all()
    _check_sampled(wl, z, lse, list(range(0, 1024, 41)) + [1023])


def test_generic_decode_at_the_batch_limit(mla):
    """4096 sequences (the largest batch mla_decode_attn accepts) on the
    shape-generic path, with empty sequences among them, paged cache."""
    rng = np.random.default_rng(2101)
    wl = mi.make_random(2101, 16, 64, 16, rng.integers(0, 130, size=4096), paged=True)
    assert (wl.seqlens == 0).any()
    z, lse, st = run_decode(mla, wl)
    assert st == 0
    empty = np.flatnonzero(wl.seqlens == 0)[:8]
    _check_sampled(wl, z, lse, sorted(set(list(range(0, 4096, 97)) + [4095] + list(empty))))


# ---------------------------------------------------------------- 16-head tensor-core path
def test_lowhead_tc_and_generic_paths_agree_with_the_oracle(mla):
    """16 heads at d_c = 512, d_R = 64 take the one-CTA-per-SM tensor-core
    kernel; the shape-generic kernel (forced) must give the same answers."""
    wl = mi.make_random(2201, 16, 512, 64, [1, 700, 2048, 65, 0, 4096, 63], paged=True)
    zt, lt, s1 = run_decode(mla, wl)
    zg, lg, s2 = run_decode(mla, wl, flags=1)   # MLA_DECODE_FORCE_GENERIC
    assert s1 == 0 and s2 == 0
    check_decode(wl, zt, lt)
    check_decode(wl, zg, lg)


def test_lowhead_tc_growing_scores_trigger_rescaling(mla):
    """Rows growing along the sequence move the running maximum block after
    block on the 16-head kernel too (its O^T columns are rescaled per head)."""
    wl = mi.make_random(2202, 16, 512, 64, [3000, 1500, 64], paged=False)
    pool = orc.bf16_to_f64(wl.pool)
    grow = (1.0 + np.arange(pool.shape[1]) / 256.0)[None, :, None]
    wl.pool = orc.round_bf16_bits(np.where(np.isnan(pool), 0.0, pool) * grow)
    for workers in (0, 1, 5):
        z, lse, st = run_decode(mla, wl, num_workers=workers)
        assert st == 0
        check_decode(wl, z, lse)


def test_lowhead_tc_zero_query_gives_the_mean_of_visible_rows(mla):
    wl = mi.make_random(2203, 16, 512, 64, [1, 63, 64, 65, 300], paged=True)
    wl.q = np.zeros_like(wl.q)
    z, lse, st = run_decode(mla, wl, num_workers=3)
    assert st == 0
    for b, L in enumerate(wl.seqlens):
        rows = orc.gather_rows(wl.pool, b, int(L), wl.block_table, 64, 0)
        want = rows[:, :wl.d_latent].mean(0)
        assert np.allclose(z[b], want[None, :], rtol=0, atol=1e-5 * max(1.0, np.abs(want).max()))
        assert np.allclose(lse[b], math.log(L), atol=1e-5)

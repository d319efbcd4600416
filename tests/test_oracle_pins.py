"""Pins of the CPU oracle to things other than itself (no GPU needed).

Each test ties an oracle function to a fact the pages print, a closed form,
an identity the pages state (naive route == absorbed route), a library
routine for a special case, or brute force on tiny inputs.
"""
import math

import numpy as np
import pytest
import scipy.special
import torch

import mla_inputs as mi
import oracle as orc
from conftest import read_golden


# ------------------------------------------------------------------ bf16
def test_bf16_widening_all_patterns_match_torch():
    bits = np.arange(1 << 16, dtype=np.uint16)
    ours = orc.bf16_to_f64(bits)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    same = (ours == ref) | (np.isnan(ours) & np.isnan(ref))
    assert same.all()


def test_bf16_rounding_matches_torch_on_float32_values():
    rng = np.random.default_rng(123)
    x = np.concatenate([
        rng.standard_normal(200000).astype(np.float32),
        (rng.standard_normal(20000) * 1e-38).astype(np.float32),   # subnormal range
        (rng.standard_normal(20000) * 1e38).clip(-3.3e38, 3.3e38).astype(np.float32),  # near overflow
        np.array([0.0, -0.0, np.inf, -np.inf, 1.0, -1.0], dtype=np.float32),
    ])
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    ours = orc.round_bf16_bits(x.astype(np.float64))
    assert np.array_equal(ours, ref)
    assert np.array_equal(mi.f32_to_bf16_bits(x), ref)      # the input generator too


def test_bf16_rounding_ties_and_no_double_rounding():
    one = 1.0
    # tie between 1 and 1 + 2^-7 goes to the even significand (1.0)
    assert orc.round_bf16_bits(np.array([one + 2.0 ** -8]))[0] == 0x3F80
    # tie between 1 + 2^-7 (odd) and 1 + 2^-6 goes to 1 + 2^-6
    assert orc.round_bf16_bits(np.array([one + 3 * 2.0 ** -8]))[0] == 0x3F82
    # just above the tie must round up; rounding through float32 first would not
    assert orc.round_bf16_bits(np.array([one + 2.0 ** -8 + 2.0 ** -40]))[0] == 0x3F81
    assert orc.round_bf16_bits(np.array([np.nan]))[0] == 0x7FC0


# ------------------------------------------------------------------ RoPE
def test_rope_position_zero_is_identity():
    x = np.random.default_rng(1).standard_normal((5, 64))
    assert np.array_equal(orc.rope(x, np.zeros(5), 10000.0), x)


def test_rope_is_complex_rotation_and_keeps_norm():
    rng = np.random.default_rng(2)
    x = rng.standard_normal((7, 64))
    pos = rng.integers(0, 200000, size=7)
    out = orc.rope(x, pos, 10000.0)
    theta = 10000.0 ** (-np.arange(32) / 32.0)
    z = (x[:, 0::2] + 1j * x[:, 1::2]) * np.exp(1j * pos[:, None] * theta)
    assert np.allclose(out[:, 0::2], z.real, atol=1e-12, rtol=0)
    assert np.allclose(out[:, 1::2], z.imag, atol=1e-12, rtol=0)
    assert np.allclose(np.linalg.norm(out, axis=1), np.linalg.norm(x, axis=1), rtol=1e-13)


def test_rope_two_dims_closed_form_and_frequency_schedule():
    # d_R = 2: theta_0 = 1, so (1, 0) at position p lands on (cos p, sin p)
    for p in (0, 1, 5, 1000):
        out = orc.rope(np.array([[1.0, 0.0]]), np.array([p]), 10000.0)[0]
        assert abs(out[0] - math.cos(p)) < 1e-15 and abs(out[1] - math.sin(p)) < 1e-15
    # d_R = 4, base 10000: the second pair turns at 10000^(-1/2) = 0.01 rad per position
    out = orc.rope(np.array([[0.0, 0.0, 1.0, 0.0]]), np.array([100]), 10000.0)[0]
    assert np.allclose(out, [0, 0, math.cos(1.0), math.sin(1.0)], atol=1e-14)


def test_rope_scores_depend_only_on_relative_position():
    rng = np.random.default_rng(3)
    q, k = rng.standard_normal(64), rng.standard_normal(64)
    for m, n, t in [(5, 3, 100), (1000, 10, 77777), (0, 9, 131071)]:
        a = orc.rope(q, m) @ orc.rope(k, n)
        b = orc.rope(q, m + t) @ orc.rope(k, n + t)
        assert abs(a - b) < 1e-11


# ------------------------------------------------------------------ closed forms
def test_closed_forms_match_printed_figures():
    g = read_golden("closed_forms.txt")
    L, H, dh, dc, dr = (int(g[k]) for k in ("v3_layers", "v3_heads", "v3_head_dim", "v3_latent", "v3_rope"))
    assert orc.mla_cache_elems(dc, dr) == int(g["v3_elems_per_token_layer"])
    mla_b = orc.mla_cache_elems(dc, dr, L) * 2
    mha_b = orc.mha_cache_elems(H, dh, L) * 2
    assert mla_b == 70272 and mha_b == 3997696
    assert int(mla_b / orc.KIB) == int(g["v3_mla_bytes_per_token_kib"])            # 68.6 KiB, printed "about 68"
    assert round(mla_b / 1000) == int(g["v3_mla_bytes_per_token_kb_approx"])       # 70.3 kB
    assert round(mha_b / orc.MIB, 1) == float(g["v3_mha_bytes_per_token_mib"])     # 3.81 MiB
    assert round(100 * mla_b / mha_b, 1) == float(g["v3_mla_over_mha_percent"])    # 1.758 %
    assert round(mha_b * 32768 / orc.GIB) == int(g["v3_32k_mha_gib"])             # 122.0 GiB
    assert round(mla_b * 32768 / orc.GIB, 1) == float(g["v3_32k_mla_gib"])         # 2.14 GiB
    # worked example of the 16-head demo config
    naive = orc.naive_mla_cache_elems(int(g["demo_heads"]), int(g["demo_qk_head_dim"]),
                                      int(g["demo_v_head_dim"]))
    assert naive == int(g["demo_naive_elems"])
    assert 100 * 576 / naive == float(g["demo_ratio_percent"])
    assert 100 - 100 * 576 / naive == float(g["demo_reduction_percent"])
    # d_c = 4 d_h, d_R = d_h / 2  ->  9/2 d_h per layer
    for d_h in (64, 128, 256):
        assert 2 * orc.mla_cache_elems(4 * d_h, d_h // 2) == int(g["v2_mla_over_dh_numer"]) * d_h
    # the 7B MHA example (32 layers, 32 heads, d 128, 2 bytes)
    b7 = orc.mha_cache_elems(32, 128, 32) * 2
    assert b7 / orc.KIB == int(g["mha7b_bytes_per_token_kib"])
    assert round(b7 * 4096 / 1e9, 1) == float(g["mha7b_4096_gb"])


# ------------------------------------------------------------------ softmax / decode
def test_two_pass_softmax_matches_scipy():
    rng = np.random.default_rng(4)
    s = rng.standard_normal((6, 300)) * 7
    a, lse = orc.softmax_two_pass(s)
    assert np.allclose(a, scipy.special.softmax(s, axis=-1), rtol=1e-13, atol=0)
    assert np.allclose(lse, scipy.special.logsumexp(s, axis=-1), rtol=1e-14, atol=0)


def test_single_token_returns_its_latent():
    rng = np.random.default_rng(5)
    q = rng.standard_normal((3, 80))
    row = rng.standard_normal((1, 80))
    z, lse = orc.decode_latent(q, row, 0.3, 64)
    assert np.array_equal(z, np.repeat(row[:, :64], 3, axis=0))
    assert np.allclose(lse, 0.3 * (q @ row[0]), rtol=1e-15)


def test_zero_query_gives_uniform_mean():
    rng = np.random.default_rng(6)
    for L in (1, 2, 63, 64, 65, 129):
        rows = rng.standard_normal((L, 80))
        z, lse = orc.decode_latent(np.zeros((4, 80)), rows, 0.5, 64)
        assert np.allclose(z, rows[:, :64].mean(0), rtol=1e-13, atol=1e-15)
        assert np.allclose(lse, math.log(L), rtol=1e-15)


def test_duplicated_rows_split_weight_evenly():
    rng = np.random.default_rng(7)
    q = rng.standard_normal((2, 80))
    r1, r2 = rng.standard_normal(80), rng.standard_normal(80)
    z, lse = orc.decode_latent(q, np.stack([r1, r1, r2]), 0.25, 64)
    s1, s2 = 0.25 * (q @ r1), 0.25 * (q @ r2)
    w1, w2 = 2 * np.exp(s1), np.exp(s2)
    want = (w1[:, None] * r1[:64] + w2[:, None] * r2[:64]) / (w1 + w2)[:, None]
    assert np.allclose(z, want, rtol=1e-12, atol=1e-14)
    assert np.allclose(lse, np.log(w1 + w2), rtol=1e-13)


def test_empty_sequence():
    z, lse = orc.decode_latent(np.ones((2, 80)), np.zeros((0, 80)), 1.0, 64)
    assert np.array_equal(z, np.zeros((2, 64))) and np.all(np.isneginf(lse))


@pytest.mark.parametrize("L", [1, 63, 64, 65, 127, 128, 129])
def test_brute_force_loops_agree(L):
    rng = np.random.default_rng(100 + L)
    q = rng.standard_normal((4, 80))
    rows = rng.standard_normal((L, 80))
    z, lse = orc.decode_latent(q, rows, 1 / math.sqrt(48), 64)
    zb, lb = orc.decode_brute(q, rows, 1 / math.sqrt(48), 64)
    assert np.allclose(z, zb, rtol=1e-12, atol=1e-13)
    assert np.allclose(lse, lb, rtol=1e-13, atol=1e-13)


@pytest.mark.parametrize("L", [1, 2, 64, 129, 500])
def test_naive_route_equals_absorbed_route(L):
    """The two inference branches compute the same attention (associativity:
    q^C.(W^UK c) = (q^C W^UK).c and sum_j a_j W^UV c_j = W^UV sum_j a_j c_j)."""
    rng = np.random.default_rng(200 + L)
    n_h, d_h, d_v, d_c, d_R = 3, 24, 20, 40, 8        # d_h != d_c != d_v catches transposes
    q_c = rng.standard_normal((n_h, d_h))
    q_r = orc.rope(rng.standard_normal((n_h, d_R)), L - 1)
    w_uk = rng.standard_normal((n_h, d_h, d_c)) / math.sqrt(d_c)
    w_uv = rng.standard_normal((n_h, d_v, d_c)) / math.sqrt(d_c)
    rows = rng.standard_normal((L, d_c + d_R))
    scale = 1 / math.sqrt(d_h + d_R)
    o_a, lse_a = orc.decode_naive(q_c, q_r, w_uk, w_uv, rows, scale, d_c)
    o_b, _, lse_b = orc.decode_absorbed(q_c, q_r, w_uk, w_uv, rows, scale, d_c)
    assert np.max(np.abs(o_a - o_b)) <= 1e-10 * max(1.0, np.max(np.abs(o_a)))
    assert np.max(np.abs(lse_a - lse_b)) <= 1e-10


def test_tiny_case_full_chain_routes_agree():
    wl = mi.make("tiny")
    D = wl.row_dim
    pool = orc.append_cache(wl.pool, wl.h, wl.w_dkv_kr, wl.app_seq, wl.app_pos, wl.d_latent,
                            None, wl.block_tokens, wl.seq_stride, wl.rope_base)
    assert pool.shape == (1, 192, D)
    assert np.all(pool[0, 129:] == mi.BF16_QNAN)                # slack untouched
    rows = orc.gather_rows(pool, 0, 129, None, 64, wl.seq_stride)
    assert np.isfinite(rows).all()
    q_c, q_r = orc.project_q(wl.h[128:129], wl.w_q, wl.d_head)
    q_r_rot = orc.rope(q_r, 128, wl.rope_base)
    w_uk, w_uv = orc.bf16_to_f64(wl.w_uk), orc.bf16_to_f64(wl.w_uv)
    o_a, lse_a = orc.decode_naive(q_c[0], q_r_rot[0], w_uk, w_uv, rows, wl.scale, wl.d_latent)
    o_b, z_b, lse_b = orc.decode_absorbed(q_c[0], q_r_rot[0], w_uk, w_uv, rows, wl.scale, wl.d_latent)
    assert np.max(np.abs(o_a - o_b)) <= 1e-10 * max(1.0, np.max(np.abs(o_a)))
    assert np.max(np.abs(lse_a - lse_b)) <= 1e-10
    q_lat = orc.absorb_q(q_c, q_r, np.array([128]), w_uk, wl.rope_base)
    z_l, lse_l = orc.decode_latent(q_lat[0], rows, wl.scale, wl.d_latent)
    assert np.allclose(z_l, z_b, rtol=1e-12, atol=1e-14) and np.allclose(lse_l, lse_b, rtol=1e-13)


# ------------------------------------------------------------------ append
def test_append_identity_weights_copies_rows_bit_exactly():
    """W = I and zero RoPE inputs: every new row is its h row, bit for bit, at
    (block_table[seq][pos // 64], pos % 64); every other slot is untouched."""
    rng = np.random.default_rng(8)
    D, d_c = 80, 64
    seqlens = np.array([70, 5, 130])
    bt, nb = mi._paged_layout(rng, seqlens, 64)
    pool = np.full((nb, 64, D), mi.BF16_QNAN, dtype=np.uint16)
    seq = np.array([0, 0, 1, 2, 2, 2])
    pos = np.array([0, 69, 4, 63, 64, 129])
    h = np.zeros((len(seq), D))
    h[:, 2:d_c] = np.arange(2, d_c) / 8.0           # small dyadic values: exact in bf16
    h[:, 0], h[:, 1] = seq + 1, pos + 1             # the row encodes where it belongs
    hb = orc.round_bf16_bits(h)
    assert np.array_equal(orc.bf16_to_f64(hb), h)
    out = orc.append_cache(pool, hb, orc.round_bf16_bits(np.eye(D)), seq, pos, d_c, bt, 64, 0)
    want = pool.copy()
    for t in range(len(seq)):
        want[bt[seq[t], pos[t] // 64], pos[t] % 64] = hb[t]
    # the rotated zero RoPE part may come out as -0.0; signed zeros compare equal
    out[out == 0x8000] = 0
    assert np.array_equal(out, want)


def test_append_rope_part_is_rotated_projection():
    rng = np.random.default_rng(9)
    d, d_c, d_R = 48, 16, 8
    h = rng.standard_normal((3, d))
    w = rng.standard_normal((d_c + d_R, d))
    pos = np.array([0, 7, 4000])
    rows = orc.append_rows(h, w, pos, d_c, 10000.0)
    raw = h @ w.T
    assert np.allclose(rows[:, :d_c], raw[:, :d_c], rtol=1e-14)
    kr = raw[:, d_c:]
    theta = 10000.0 ** (-np.arange(d_R // 2) / (d_R // 2))
    zc = (kr[:, 0::2] + 1j * kr[:, 1::2]) * np.exp(1j * pos[:, None] * theta)
    assert np.allclose(rows[:, d_c::2], zc.real, atol=1e-12) and np.allclose(rows[:, d_c + 1::2], zc.imag, atol=1e-12)


# ------------------------------------------------------------------ worked example
def test_worked_example_shapes():
    g = {k: tuple(int(x) for x in v.split(",")) for k, v in read_golden("worked_example_shapes.txt").items()}
    rng = np.random.default_rng(10)
    dim, n_h, nope, rope_d, d_c, v_d, start = 2048, 16, 128, 64, 512, 128, 1024
    bf = lambda a: orc.bf16_to_f64(orc.round_bf16_bits(a))
    x = bf(rng.standard_normal((1, 1, dim)))
    w_q = orc.round_bf16_bits(rng.standard_normal((n_h, nope + rope_d, dim)) / math.sqrt(dim))
    w_a = orc.round_bf16_bits(rng.standard_normal((d_c + rope_d, dim)) / math.sqrt(dim))
    w_uk = bf(rng.standard_normal((n_h, nope, d_c)) / math.sqrt(d_c))
    w_uv = bf(rng.standard_normal((n_h, v_d, d_c)) / math.sqrt(d_c))
    w_o = bf(rng.standard_normal((dim, n_h * v_d)) / math.sqrt(n_h * v_d))
    assert x.shape == g["x"]
    q_nope, q_pe = orc.project_q(orc.round_bf16_bits(x[0]), w_q, nope)
    q = np.concatenate([q_nope, q_pe], -1)[None]
    assert q.shape == g["q"] and q_nope[None].shape == g["q_nope"] and q_pe[None].shape == g["q_pe"]
    kv_and_pe = (orc.bf16_to_f64(w_a) @ x[0, 0])[None, None]
    assert kv_and_pe.shape == g["kv_and_pe"]
    assert kv_and_pe[..., :d_c].shape == g["kv_latent"] and kv_and_pe[..., d_c:].shape == g["k_pe"]
    cache = np.full((1, 2048, d_c + rope_d), mi.BF16_QNAN, dtype=np.uint16)
    cache[0, :start] = orc.round_bf16_bits(rng.standard_normal((start, d_c + rope_d)))
    cache = orc.append_cache(cache, orc.round_bf16_bits(x[0]), w_a, [0], [start], d_c, None, 64, 2048)
    rows = orc.gather_rows(cache, 0, start + 1, None, 64, 2048)
    assert rows[None, :, :d_c].shape == g["kv_cache_visible"] and rows[None, :, d_c:].shape == g["pe_cache_visible"]
    q_lat = orc.absorb_q(q_nope, q_pe, np.array([start]), w_uk)
    assert q_lat[None, :, :, :d_c].shape == g["q_nope_absorb"]
    scale = 1 / math.sqrt(nope + rope_d)
    score = (q_lat[0, :, :d_c] @ rows[:, :d_c].T + q_lat[0, :, d_c:] @ rows[:, d_c:].T) * scale
    assert score[None, None].shape == g["score"]
    a, _ = orc.softmax_two_pass(score)
    assert a[None, None].shape == g["attn"]
    z, _ = orc.decode_latent(q_lat[0], rows, scale, d_c)
    assert z[None, None].shape == g["z"]
    o = orc.out_proj(z[None], w_uv)
    assert o[None].shape == g["o"]
    u = orc.output_projection(o, w_o)
    assert u[None].shape == g["u"]
    assert np.isfinite(u).all()


# ------------------------------------------------------------------ sensitivity
def test_pins_catch_planted_mistakes(monkeypatch):
    """Plant plausible mistakes in the oracle and check a pin above fails."""
    rng = np.random.default_rng(11)
    n_h, d_h, d_v, d_c, d_R, L = 2, 12, 10, 16, 8, 9
    q_c = rng.standard_normal((n_h, d_h))
    q_r = rng.standard_normal((n_h, d_R))
    w_uk = rng.standard_normal((n_h, d_h, d_c))
    w_uv = rng.standard_normal((n_h, d_v, d_c))
    rows = rng.standard_normal((L, d_c + d_R))

    def routes_agree():
        o_a, _ = orc.decode_naive(q_c, q_r, w_uk, w_uv, rows, 0.2, d_c)
        o_b, _, _ = orc.decode_absorbed(q_c, q_r, w_uk, w_uv, rows, 0.2, d_c)
        return np.max(np.abs(o_a - o_b)) <= 1e-10 * max(1.0, np.max(np.abs(o_a)))

    assert routes_agree()
    good = orc.mla.decode_latent

    def dropped_rope_term(q_lat, rows_, scale, d_latent):
        q2 = np.array(q_lat, copy=True)
        q2[:, d_latent:] = 0.0
        return good(q2, rows_, scale, d_latent)
    monkeypatch.setattr(orc.mla, "decode_latent", dropped_rope_term)
    assert not routes_agree()
    monkeypatch.setattr(orc.mla, "decode_latent", good)

    def wrong_sign_rope(x, pos, base=10000.0):
        return orc.mla.__dict__["_rope_ok"](x, -np.asarray(pos), base)
    orc.mla.__dict__["_rope_ok"] = orc.mla.rope
    monkeypatch.setattr(orc.mla, "rope", wrong_sign_rope)
    out = orc.mla.rope(np.array([[1.0, 0.0]]), np.array([1]))[0]
    assert abs(out[1] - math.sin(1.0)) > 0.1          # the two-dim closed form catches it
    del orc.mla.__dict__["_rope_ok"]

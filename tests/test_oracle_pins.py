"""Pins of the CPU oracle to things other than itself.

Each test checks one oracle function against a closed form, a textbook value,
brute force on a tiny input, an exact identity of the method, or a special
case; together they are chosen so that a dropped term, a wrong sign or index,
or a transposed operand in the oracle fails at least one of them.
"""
import json
import math
import os

import numpy as np
import pytest

import synth
from oracle import wan_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
rng = np.random.default_rng(1234)


# ---------------------------------------------------------------- activations

def test_gelu_textbook_values():
    # GELU(x) = x * Phi(x); Phi(1) = 0.8413447460685429 (standard normal table).
    # The tanh approximation gives 0.8411919906082768 at 1 and would fail.
    g = O.gelu(np.array([1.0, -1.0, 0.0, 2.0]))
    assert g[0] == pytest.approx(0.8413447460685429, abs=1e-15)
    assert g[1] == pytest.approx(-0.15865525393145707, abs=1e-15)
    assert g[2] == 0.0
    assert g[3] == pytest.approx(2 * 0.9772498680518208, abs=1e-14)


def test_silu_textbook_values():
    s = O.silu(np.array([0.0, 1.0, -1.0]))
    assert s[0] == 0.0
    assert s[1] == pytest.approx(1.0 / (1.0 + math.e ** -1), abs=1e-15)
    assert s[2] == pytest.approx(-1.0 / (1.0 + math.e), abs=1e-15)


# ---------------------------------------------------------------- LayerNorm / modulation

def test_layer_norm_moments_and_affine_invariance():
    x = rng.normal(size=(7, 64)) * 3 + 1.5
    y = O.layer_norm(x, 1e-6)
    assert np.allclose(y.mean(-1), 0.0, atol=1e-14)
    var = x.var(-1)
    assert np.allclose(y.var(-1), var / (var + 1e-6), atol=1e-13)
    # invariant to x -> a x + c per row (a > 0), up to the eps term
    y2 = O.layer_norm(4.0 * x - 7.0, 1e-12)
    assert np.allclose(y2, O.layer_norm(x, 1e-12), atol=1e-12)


def test_layer_norm_constant_row_is_zero():
    assert np.all(O.layer_norm(np.full((2, 8), 3.25), 1e-6) == 0.0)


def test_modulate_zero_is_identity():
    y = rng.normal(size=(5, 16))
    assert np.array_equal(O.modulate(y, 0.0, 0.0), y)
    assert np.allclose(O.modulate(y, 1.0, -1.0), 1.0)


# ---------------------------------------------------------------- time embedding

def test_sinusoid_closed_forms():
    # tau = 0: all cosines 1, all sines 0
    s0 = O.sinusoid(np.array([0.0]))[0]
    assert np.array_equal(s0[:128], np.ones(128)) and np.array_equal(s0[128:], np.zeros(128))
    # w_0 = 1: tau = pi/2 gives cos = 0 and sin = 1 in the first pair
    s = O.sinusoid(np.array([math.pi / 2 / 1000]))[0]
    assert abs(s[0]) < 1e-15 and s[128] == pytest.approx(1.0, abs=1e-15)
    # w_64 = 10000^(-1/2) = 1/100: tau = 100 pi gives cos(pi) = -1, sin(pi) = 0
    s = O.sinusoid(np.array([100 * math.pi / 1000]))[0]
    assert s[64] == pytest.approx(-1.0, abs=1e-12) and abs(s[128 + 64]) < 1e-12
    assert np.allclose(s[:128] ** 2 + s[128:] ** 2, 1.0, atol=1e-15)


def test_time_embedding_zero_weights():
    D = 8
    w = {"t1_w": np.zeros((D, 256)), "t1_b": np.full(D, 0.5), "t2_w": np.zeros((D, D)),
         "t2_b": np.full(D, 1.0), "m_w": np.zeros((6 * D, D)), "m_b": np.arange(6 * D) * 0.1,
         "hm_w": np.ones((2 * D, D)), "hm_b": np.zeros(2 * D)}
    e, e0, hm = O.time_embedding(np.array([0.3, 0.9]), w, D)
    assert np.array_equal(e, np.ones((2, D)))              # e = b2
    assert np.allclose(e0[1, 2], np.arange(2 * D, 3 * D) * 0.1)   # gate1 slot = third D-chunk of bm
    silu1 = 1.0 / (1.0 + math.exp(-1.0))
    assert np.allclose(hm, D * silu1)                       # ones-matrix times SiLU(1)


# ---------------------------------------------------------------- RoPE

def test_rope_axis_split():
    assert O.rope_axis_dims(128) == (44, 42, 42)
    assert O.rope_axis_dims(64) == (24, 20, 20)


def test_rope_preserves_pair_norms_and_zero_position_is_identity():
    grid = (3, 4, 5)
    x = rng.normal(size=(60, 2, 64))
    pos = O.token_positions(grid)
    y = O.rope3d(x, pos)
    assert np.allclose(x[..., 0::2] ** 2 + x[..., 1::2] ** 2, y[..., 0::2] ** 2 + y[..., 1::2] ** 2, atol=1e-13)
    assert np.array_equal(y[0], x[0])          # token 0 sits at (0,0,0)


def test_rope_dot_product_depends_only_on_relative_offset():
    d = 64
    q = rng.normal(size=(1, 1, d))
    k = rng.normal(size=(1, 1, d))
    pa, pb = np.array([[2, 1, 3]]), np.array([[0, 4, 1]])
    ref = np.sum(O.rope3d(q, pa) * O.rope3d(k, pb))
    for shift in ([1, 0, 0], [0, 2, 0], [0, 0, 5], [3, 1, 2]):
        s = np.array([shift])
        assert np.sum(O.rope3d(q, pa + s) * O.rope3d(k, pb + s)) == pytest.approx(ref, abs=1e-12)
    # a different relative offset gives a different score
    assert abs(np.sum(O.rope3d(q, pa) * O.rope3d(k, pb + np.array([[1, 0, 0]]))) - ref) > 1e-6


def test_rope_axis_layout_frame_height_width():
    # Only the first d_f dims rotate with the frame index, the next d_h with the
    # height index, the last d_w with the width index.
    d = 128
    df, dh, dw = O.rope_axis_dims(d)
    x = rng.normal(size=(1, 1, d))
    yf = O.rope3d(x, np.array([[1, 0, 0]]))
    yh = O.rope3d(x, np.array([[0, 1, 0]]))
    yw = O.rope3d(x, np.array([[0, 0, 1]]))
    ch = lambda y: np.flatnonzero(np.abs(y - x)[0, 0] > 0)
    assert ch(yf).min() == 0 and ch(yf).max() < df
    assert ch(yh).min() >= df and ch(yh).max() < df + dh
    assert ch(yw).min() >= df + dh and ch(yw).max() < d


def test_rope_reduces_to_textbook_1d_rope():
    # With the token grid (L, 1, 1) only the frame axis moves.  On the frame part
    # this must equal RoFormer's rotary embedding: pair j of position p is the
    # complex number (x_2j + i x_2j+1) multiplied by exp(i p theta^(-2j/d_f)).
    d, L, theta = 64, 7, 10000.0
    df = O.rope_axis_dims(d)[0]
    x = rng.normal(size=(L, 1, d))
    y = O.rope3d(x, O.token_positions((L, 1, 1)), theta)
    for p in range(L):
        for j in range(df // 2):
            z = complex(x[p, 0, 2 * j], x[p, 0, 2 * j + 1]) * np.exp(1j * p * theta ** (-2 * j / df))
            assert y[p, 0, 2 * j] == pytest.approx(z.real, abs=1e-12)
            assert y[p, 0, 2 * j + 1] == pytest.approx(z.imag, abs=1e-12)
    assert np.array_equal(y[..., df:], x[..., df:])


def test_token_positions_order():
    pos = O.token_positions((2, 3, 4))
    assert pos[0].tolist() == [0, 0, 0]
    assert pos[1].tolist() == [0, 0, 1]       # width fastest
    assert pos[4].tolist() == [0, 1, 0]
    assert pos[12].tolist() == [1, 0, 0]
    assert pos[23].tolist() == [1, 2, 3]


# ---------------------------------------------------------------- attention

def _brute_attention(q, k, v):
    Lq, H, d = q.shape
    Lk = k.shape[0]
    out = np.zeros((Lq, H, v.shape[-1]))
    for h in range(H):
        for i in range(Lq):
            logits = [sum(q[i, h, c] * k[j, h, c] for c in range(d)) / math.sqrt(d) for j in range(Lk)]
            m = max(logits)
            ws = [math.exp(a - m) for a in logits]
            z = sum(ws)
            for c in range(v.shape[-1]):
                out[i, h, c] = sum(ws[j] * v[j, h, c] for j in range(Lk)) / z
    return out


def test_attention_brute_force():
    q = rng.normal(size=(5, 2, 4)) * 2
    k = rng.normal(size=(7, 2, 4)) * 2
    v = rng.normal(size=(7, 2, 4))
    assert np.allclose(O.attention(q, k, v), _brute_attention(q, k, v), atol=1e-13)
    # row chunking must not change anything
    assert np.allclose(O.attention(q, k, v, chunk=2), O.attention(q, k, v), atol=1e-15)


def test_attention_special_cases():
    q = rng.normal(size=(6, 3, 8))
    v1 = rng.normal(size=(1, 3, 8))
    assert np.allclose(O.attention(q, rng.normal(size=(1, 3, 8)), v1), np.broadcast_to(v1, (6, 3, 8)), atol=1e-15)
    kc = np.broadcast_to(rng.normal(size=(1, 3, 8)), (9, 3, 8))
    v = rng.normal(size=(9, 3, 8))
    assert np.allclose(O.attention(q, kc, v), np.broadcast_to(v.mean(0), (6, 3, 8)), atol=1e-14)
    # large logits select the best-matching key
    k = np.eye(8)[:, None, :].repeat(3, axis=1) * 1e3
    qq = np.eye(8)[[2, 5], None, :].repeat(3, axis=1)
    v = rng.normal(size=(8, 3, 8))
    o = O.attention(qq, k, v)
    assert np.allclose(o[0], v[2], atol=1e-12) and np.allclose(o[1], v[5], atol=1e-12)
    # outputs are convex combinations of the values
    o = O.attention(q, rng.normal(size=(9, 3, 8)), v[:1].repeat(9, 0) + rng.normal(size=(9, 3, 8)))
    assert o.shape == (6, 3, 8)


def test_attention_convexity():
    q, k, v = rng.normal(size=(4, 1, 8)) * 3, rng.normal(size=(10, 1, 8)) * 3, rng.normal(size=(10, 1, 8))
    o = O.attention(q, k, v)
    assert np.all(o <= v.max(0) + 1e-12) and np.all(o >= v.min(0) - 1e-12)


# ---------------------------------------------------------------- patchify / unpatchify

def test_patchify_index_formula_brute_force():
    B, C, F, H, W = 2, 3, 2, 4, 6
    lat = rng.normal(size=(B, C, F, H, W))
    p = O.patchify_tokens(lat)
    Hp, Wp = H // 2, W // 2
    for b in range(B):
        for c in range(C):
            for f in range(F):
                for y in range(H):
                    for x in range(W):
                        i, di, j, dj = y // 2, y % 2, x // 2, x % 2
                        assert p[b, (f * Hp + i) * Wp + j, c * 4 + di * 2 + dj] == lat[b, c, f, y, x]


def test_patchify_identity_weight_and_unpatchify_roundtrip():
    B, C, F, H, W = 1, 4, 3, 6, 4
    lat = rng.normal(size=(B, C, F, H, W))
    x = O.patchify(lat, np.eye(C * 4), np.zeros(C * 4))
    assert np.array_equal(x, O.patchify_tokens(lat))
    assert np.array_equal(O.unpatchify(x, C, F, H, W), lat)


def test_patchify_i2v_zero_columns():
    # I2V: extra input channels with zero-initialised projection columns leave the
    # 16-channel result unchanged.
    D = 8
    lat16 = rng.normal(size=(1, 16, 2, 4, 4))
    extra = rng.normal(size=(1, 20, 2, 4, 4))
    w16 = rng.normal(size=(D, 64))
    b = rng.normal(size=D)
    w36 = np.concatenate([w16, np.zeros((D, 80))], axis=1)
    a = O.patchify(lat16, w16, b)
    c = O.patchify(np.concatenate([lat16, extra], axis=1), w36, b)
    assert np.allclose(a, c, atol=1e-14)


# ---------------------------------------------------------------- guidance and Euler

def test_cfg_special_cases():
    vc, vu = rng.normal(size=(3, 5)), rng.normal(size=(3, 5))
    assert np.allclose(O.cfg_combine(vc, vu, 1.0), vc, rtol=0, atol=1e-15)
    assert np.array_equal(O.cfg_combine(vc, vu, 0.0), vu)
    a, b = O.cfg_combine(vc, vu, 2.0), O.cfg_combine(vc, vu, 5.0)
    assert np.allclose(O.cfg_combine(vc, vu, 3.5), (a + b) / 2, atol=1e-14)   # affine in s


def test_euler_exact_velocity_lands_on_data():
    # x_t = t x0 + (1 - t) x1 (t = 1 noise, t = 0 data); dx/dt = x0 - x1.
    x0, x1 = rng.normal(size=100), rng.normal(size=100)
    v = x0 - x1
    assert np.allclose(O.euler_step(x0, v, -1.0), x1, atol=1e-15)
    x = x0.copy()
    ts = O.timesteps(20)
    assert ts[0] == 1.0 and ts[-1] == 0.0 and len(ts) == 21
    for k in range(20):
        x = O.euler_step(x, v, ts[k + 1] - ts[k])
    assert np.allclose(x, x1, atol=1e-14)


def test_euler_zero_velocity_and_cfg_euler():
    x = rng.normal(size=10)
    assert np.array_equal(O.euler_step(x, np.zeros(10), -0.05), x)
    vc, vu = rng.normal(size=10), rng.normal(size=10)
    assert np.allclose(O.cfg_euler_step(x, vc, vu, 1.0, -0.05), x - 0.05 * vc, atol=1e-15)


# ---------------------------------------------------------------- block / forward

def _tiny(seed=0, **kw):
    s = synth.TINY.replace(**kw)
    w = synth.make_weights(s, seed)
    inp = synth.make_inputs(s, seed)
    return s, w, inp


def _ctx(s, w, inp):
    return O.text_projection(inp["text"], w)


def test_adaln_zero_reduces_block_to_residual_path():
    s, w, inp = _tiny()
    hp = O.Hyper.of(s)
    blk = dict(w["blocks"][0])
    x = rng.normal(size=(s.tokens, s.dim))
    ctx = _ctx(s, w, inp)[0]
    zero = np.zeros((6, s.dim))
    out = O.dit_block(x, zero, blk, ctx, None, hp)
    expect = x + O.cross_attention(x, blk, ctx, None, hp)
    assert np.allclose(out, expect, atol=1e-14)
    blk["co_w"] = np.zeros_like(blk["co_w"])
    blk["co_b"] = np.zeros_like(blk["co_b"])
    assert np.array_equal(O.dit_block(x, zero, blk, ctx, None, hp), x)


def test_block_row_sampling_matches_full_block():
    s, w, inp = _tiny()
    hp = O.Hyper.of(s)
    blk = w["blocks"][0]
    x = rng.normal(size=(s.tokens, s.dim))
    ctx = _ctx(s, w, inp)[0]
    mods = rng.normal(size=(6, s.dim)) * 0.1
    full = O.dit_block(x, mods, blk, ctx, None, hp)
    rows = np.array([0, 5, 17, s.tokens - 1])
    assert np.allclose(O.dit_block(x, mods, blk, ctx, None, hp, rows=rows), full[rows], atol=1e-13)


def test_decoupled_cross_attention_sums_two_softmaxes():
    s, w, inp = _tiny(img_len=5, i2v=False)
    hp = O.Hyper.of(s)
    blk = dict(w["blocks"][0])
    blk["ckvi_w"], blk["ckvi_b"] = blk["ckv_w"], blk["ckv_b"]
    x = rng.normal(size=(10, s.dim))
    ctx = _ctx(s, w, inp)[0]
    one = O.cross_attention(x, blk, ctx, None, hp) - blk["co_b"]
    two = O.cross_attention(x, blk, ctx, ctx, hp) - blk["co_b"]
    assert np.allclose(two, 2 * one, atol=1e-13)


def test_forward_batch_permutation_equivariance():
    s, w, inp = _tiny()
    ctx = _ctx(s, w, inp)
    lat = np.concatenate([inp["latent"], 0.5 * inp["latent"]], axis=0)
    t = np.array([0.3, 0.8])
    v = O.dit_forward(lat, t, ctx, None, w, s)
    vp = O.dit_forward(lat[::-1], t[::-1], ctx[::-1], None, w, s)
    assert np.allclose(v[::-1], vp, atol=1e-13)
    assert v.shape == (2, s.c_out, s.frames, s.height, s.width)


def test_forward_row_sampling_matches_full_forward():
    s, w, inp = _tiny()
    ctx = _ctx(s, w, inp)
    lat = np.concatenate([inp["latent"]] * 2, axis=0)
    t = np.array([0.4, 0.4])
    v = O.dit_forward(lat, t, ctx, None, w, s)
    rows = np.array([1, 9, 47])
    hv, _ = O.dit_forward(lat, t, ctx, None, w, s, rows=rows)
    tok = O.patchify_tokens(v)          # head outputs arranged as tokens
    assert np.allclose(hv, tok[:, rows], atol=1e-13)


def test_guided_step_with_scale_one_is_conditional_euler():
    s, w, inp = _tiny(guide_scale=1.0)
    ctx = _ctx(s, w, inp)
    t = float(inp["t"][0])
    xn = O.guided_step(inp["latent"], t, -0.05, ctx, None, w, s)
    v = O.dit_forward(inp["latent"], np.array([t]), ctx[:1], None, w, s)
    assert np.allclose(xn, inp["latent"] - 0.05 * v, atol=1e-14)


# ---------------------------------------------------------------- geometry fixture

def test_latent_geometry_fixture():
    with open(os.path.join(GOLDEN, "latent_geometry.json")) as f:
        g = json.load(f)
    for case in g["cases"]:
        T1, H, W = case["video"]
        lat = [1 + (T1 - 1) // g["compression"][0], H // g["compression"][1], W // g["compression"][2]]
        assert lat == case["latent"]
        tokens = lat[0] * (lat[1] // 2) * (lat[2] // 2)
        assert tokens == case["tokens"]
        cfg = synth.WORKLOADS[case["workload"]]
        assert [cfg.frames, cfg.height, cfg.width] == lat and cfg.tokens == tokens
    c, s_ = g["i2v_channels"]["c"], g["i2v_channels"]["s"]
    assert 2 * c + s_ == synth.BLOCK_14B_I2V.c_in


def test_gelu_tanh_variant_textbook_values_and_closeness_to_erf_form():
    # tanh form = x * sigmoid(odd function of x): exact at 0, GELU(x) - GELU(-x) = x, tends
    # to x and 0 in the tails, and stays within 1e-3 of the erf form everywhere.
    assert O.gelu_tanh(0.0) == 0.0
    x = np.linspace(-6, 6, 1201)
    assert np.allclose(O.gelu_tanh(x) - O.gelu_tanh(-x), x, atol=1e-14)
    assert abs(O.gelu_tanh(30.0) - 30.0) < 1e-12 and abs(O.gelu_tanh(-30.0)) < 1e-12
    assert np.max(np.abs(O.gelu_tanh(x) - O.gelu(x))) < 1e-3
    # sqrt(2/pi) * (1 + 0.044715) at x = 1: 0.5 (1 + tanh(0.8333...))
    assert abs(O.gelu_tanh(1.0) - 0.5 * (1.0 + np.tanh(np.sqrt(2 / np.pi) * 1.044715))) < 1e-15


def test_rms_norm_variant_unit_rms_scale_invariance_and_weight():
    rng = np.random.default_rng(3)
    x = rng.normal(size=(7, 64)) * 3.0
    ones = np.ones(64)
    y = O.rms_norm(x, ones, 0.0)
    assert np.allclose(np.sqrt((y ** 2).mean(axis=-1)), 1.0, atol=1e-13)
    assert np.allclose(O.rms_norm(5.0 * x, ones, 0.0), y, atol=1e-13)       # invariant to a positive scale
    assert np.allclose(O.rms_norm(-x, ones, 0.0), -y, atol=1e-13)           # odd
    w = rng.normal(size=64)
    assert np.allclose(O.rms_norm(x, w, 0.0), y * w, atol=1e-13)           # weight is elementwise
    # eps: a zero row stays zero; a tiny row is damped, not blown up
    assert np.all(O.rms_norm(np.zeros((1, 64)), ones, 1e-6) == 0.0)


def test_qk_norm_variant_makes_block_invariant_to_q_k_projection_scale():
    # With RMSNorm on q and k, scaling the q and k projection weights and biases by any
    # positive factor leaves the block unchanged (the norm removes the scale; only the
    # eps = 1e-6 term, ~1e-5 of mean(q^2) here, is not scaled).
    s = synth.TINY.replace(qk_norm=True, gelu_tanh=True)
    w = synth.make_weights(s, 0)
    inp = synth.make_inputs(s, 0)
    hp = O.Hyper.of(s)
    x = O.patchify(inp["latent"], w["patch_w"], w["patch_b"])[0]
    ctx = O.text_projection(inp["text"][:1], w)[0]
    mods = np.zeros((6, s.dim)) + 0.1
    blk = w["blocks"][0]
    base = O.dit_block(x, mods, blk, ctx, None, hp)
    blk2 = dict(blk)
    D = s.dim
    blk2["qkv_w"] = blk["qkv_w"].copy(); blk2["qkv_b"] = blk["qkv_b"].copy()
    blk2["qkv_w"][:2 * D] *= 7.5
    blk2["qkv_b"][:2 * D] *= 7.5
    assert np.allclose(O.dit_block(x, mods, blk2, ctx, None, hp), base, rtol=1e-4, atol=1e-6)
    # ... while without the norm the same scaling changes the result
    hp_plain = O.Hyper.of(s.replace(qk_norm=False))
    assert not np.allclose(O.dit_block(x, mods, blk2, ctx, None, hp_plain),
                           O.dit_block(x, mods, blk, ctx, None, hp_plain), rtol=1e-3, atol=1e-3)


# ---------------------------------------------------------------- 8-bit variant

def _grid_values(shape, r):
    """Random finite E4M3 values (codes 0x00..0x7E with random sign) scaled by 2^r."""
    codes = rng.integers(0, 0x7F, size=shape)
    sign = np.where(rng.random(shape) < 0.5, -1.0, 1.0)
    return O.e4m3_decode(codes) * sign * np.ldexp(1.0, r)


def test_e4m3_decode_format_values():
    # OCP 8-bit floating point, E4M3: bias 7, max normal 1.75 * 2^8 = 448, min normal 2^-6,
    # min subnormal 2^-9, S.1111.111 is NaN, no infinities.
    v = O.e4m3_decode(np.arange(256))
    assert v[0x7E] == 448.0 and v[0xFE] == -448.0
    assert v[0x08] == 2.0 ** -6 and v[0x07] == 7 * 2.0 ** -9 and v[0x01] == 2.0 ** -9
    assert v[0x38] == 1.0 and v[0x39] == 1.125 and v[0x40] == 2.0 and v[0x30] == 0.5
    assert np.isnan(v[0x7F]) and np.isnan(v[0xFF]) and np.isnan(v).sum() == 2
    pos = v[1:0x7F]
    assert len(pos) == 126 and np.all(np.diff(pos) > 0)
    # the library's E4M3 ("fn": finite + NaN) type decodes the same bytes the same way
    import torch
    tv = torch.from_numpy(np.arange(256, dtype=np.uint8)).view(torch.float8_e4m3fn).double().numpy()
    fin = ~np.isnan(v)
    assert np.array_equal(tv[fin], v[fin]) and np.all(np.isnan(tv[~fin]))


def test_e4m3_round_ties_to_even_saturation_and_library_agreement():
    import torch
    x = (rng.standard_normal(200000) * np.exp(rng.uniform(-12, 6, 200000))).astype(np.float32)
    x = x[np.abs(x) < 448]
    lib = torch.from_numpy(x).to(torch.float8_e4m3fn).double().numpy()
    assert np.array_equal(O.e4m3_round(x), lib)
    # midpoints between neighbours round to the even mantissa
    v = O.e4m3_decode(np.arange(0, 0x7E))
    mids = 0.5 * (v[:-1] + v[1:])
    r = O.e4m3_round(mids)
    even = np.where(np.arange(0, 0x7D) % 2 == 0, v[:-1], v[1:])
    assert np.array_equal(r, even)
    # saturation at +-448 (the kernels' satfinite conversion), identity on the grid
    assert np.array_equal(O.e4m3_round([449.0, 464.0, 1e9, -1e9]), [448.0, 448.0, 448.0, -448.0])
    fin = np.concatenate([v, -v])
    assert np.array_equal(O.e4m3_round(fin), fin)
    codes = np.arange(256)
    ok = ~np.isnan(O.e4m3_decode(codes))
    assert np.array_equal(O.e4m3_encode(O.e4m3_decode(codes[ok])), codes[ok].astype(np.uint8))


def test_quant_rows_max_maps_to_448_and_error_bound():
    x = rng.standard_normal((64, 300)) * np.exp(rng.uniform(-8, 8, (64, 1)))
    x[3] = 0.0
    codes, s = O.quant_rows(x)
    x32 = x.astype(np.float32).astype(np.float64)
    i = np.abs(x32).argmax(axis=1)
    rows = np.arange(64) != 3
    assert np.all(np.abs(O.e4m3_decode(codes[np.arange(64), i]))[rows] == 448.0)
    assert np.all(codes[3] == 0) and s[3] == 0.0
    d = O.dequant(codes, s[:, None])
    err = np.abs(d - x32)
    normal = np.abs(x32) >= (2.0 ** -6) * s[:, None] * 1.0001
    # relative 2^-4 (half an ulp of 3 mantissa bits) in the normal range, 2^-10 s below,
    # plus the fp32 rounding of the scaled value
    assert np.all(err[normal] <= (2.0 ** -4 + 1e-6) * np.abs(x32[normal]))
    assert np.all(err[~normal] <= (2.0 ** -10 + 1e-6) * np.broadcast_to(s[:, None], err.shape)[~normal])


def test_linear_fp8_exact_on_representable_inputs_and_brute_force():
    # Each row of A (and of W) holds E4M3 grid values times 2^r with one entry equal to
    # 448 * 2^r: its scale is 2^r exactly and quantisation is the identity, so the FP8
    # GEMM must equal the exact product (checked by plain loops on a small case).
    M, N, K = 5, 4, 9
    ra, rw = rng.integers(-6, 6, M), rng.integers(-6, 6, N)
    A = np.stack([_grid_values(K, r) for r in ra]); A[np.arange(M), rng.integers(0, K, M)] = 448.0 * np.ldexp(1.0, ra)
    W = np.stack([_grid_values(K, r) for r in rw]); W[np.arange(N), rng.integers(0, K, N)] = -448.0 * np.ldexp(1.0, rw)
    a8, sa = O.quant_rows(A)
    w8, sw = O.quant_rows(W)
    assert np.array_equal(sa, np.ldexp(1.0, ra)) and np.array_equal(sw, np.ldexp(1.0, rw))
    b = rng.standard_normal(N)
    y = O.linear_fp8(a8, sa, w8, sw, b)
    for m in range(M):
        for n in range(N):
            acc = b[n]
            for k in range(K):
                acc += A[m, k] * W[n, k]
            assert y[m, n] == pytest.approx(acc, rel=1e-13, abs=1e-12)


def test_linear_fp8_scales_are_per_row_and_per_channel():
    # Rows and channels of very different magnitudes keep the E4M3 relative accuracy;
    # one scale per tensor would flush the small ones to zero.
    A = rng.standard_normal((8, 256)) * np.array([1e-4, 1, 1e3, 1, 1e-2, 1, 30, 1])[:, None]
    W = rng.standard_normal((6, 256)) * np.array([1e-3, 1, 1e2, 1, 1, 5e-2])[:, None]
    a8, sa = O.quant_rows(A)
    w8, sw = O.quant_rows(W)
    y = O.linear_fp8(a8, sa, w8, sw)
    ref = A @ W.T
    # each product carries at most (1 + 2^-4)^2 - 1 relative error
    bound = (2 * 2.0 ** -4 + 2.0 ** -8) * (np.abs(A) @ np.abs(W).T)
    assert np.all(np.abs(y - ref) <= bound)
    # error relative to sum |a w|: ~2^-4 / sqrt(K) for independent roundings, on every row
    # (a per-tensor activation scale measures 0.13-0.23 on the 1e-4 row)
    rel = np.abs(y - ref) / (np.abs(A) @ np.abs(W).T)
    assert rel.max() < 0.04 and np.median(rel) < 0.006


def _attn_operands(L, H, d, block=128):
    """q, k, v on scaled E4M3 grids whose group maxima are 448 * 2^r exactly."""
    q = np.empty((L, H, d)); k = np.empty((L, H, d)); v = np.empty((L, H, d))
    for l in range(L):
        for h in range(H):
            r = int(rng.integers(-7, -3))
            q[l, h] = _grid_values(d, r); q[l, h, rng.integers(0, d)] = 448.0 * 2.0 ** r
    for h in range(H):
        for j0 in range(0, L, block):
            r = int(rng.integers(-7, -3))
            n = min(block, L - j0)
            k[j0:j0 + n, h] = _grid_values((n, d), r)
            k[j0 + rng.integers(0, n), h, rng.integers(0, d)] = -448.0 * 2.0 ** r
        for c in range(d):
            r = int(rng.integers(-5, 3))
            v[:, h, c] = _grid_values(L, r); v[rng.integers(0, L), h, c] = 448.0 * 2.0 ** r
    return q, k, v


def test_attention_8bit_exact_on_representable_inputs():
    # Quantisation is the identity on these operands, so the 8-bit attention equals the
    # exact attention; a scale applied along the wrong axis (per key instead of per key
    # block, per token instead of per channel for v) or a dropped one breaks the equality.
    L, H, d = 300, 2, 16
    q, k, v = _attn_operands(L, H, d)
    q8, sq = O.quant_attn_q(q)
    k8, sk = O.quant_attn_k(k)
    v8, sv = O.quant_attn_v(v)
    assert sq.shape == (L, H) and sk.shape == (H, 3) and sv.shape == (H, d)
    assert np.array_equal(O.dequant(q8, sq[..., None]), q)
    o8 = O.attention_8bit(q8, sq, k8, sk, v8, sv)
    assert np.allclose(o8, O.attention(q, k, v), rtol=1e-12, atol=1e-14 * np.abs(v).max())
    # key masking: only the first kv_len keys; with one key every row returns v[0]
    o1 = O.attention_8bit(q8, sq, k8, sk, v8, sv, kv_len=1)
    assert np.allclose(o1, np.broadcast_to(v[0], o1.shape), rtol=1e-14, atol=0)
    o_m = O.attention_8bit(q8, sq, k8, sk, v8, sv, kv_len=200)
    assert np.allclose(o_m, O.attention(q, k[:200], v[:200]), rtol=1e-12, atol=1e-14 * np.abs(v).max())


def test_attention_quantisers_group_by_token_head_key_block_and_channel():
    # Brute force over the groups: each scale is the group's |max| / 448 and every value of
    # the group keeps E4M3 relative accuracy, whatever the other groups' magnitudes.
    L, H, d, blk = 300, 2, 8, 128
    mag = np.exp(rng.uniform(-10, 10, (L, H, d)))
    x = rng.standard_normal((L, H, d)) * mag
    x32 = x.astype(np.float32).astype(np.float64)
    q8, sq = O.quant_attn_q(x)
    k8, sk = O.quant_attn_k(x, blk)
    v8, sv = O.quant_attn_v(x)

    def check(codes, scale_of):
        err = np.abs(O.e4m3_decode(codes) * scale_of - x32)
        normal = np.abs(x32) >= 2.0 ** -6 * scale_of * 1.0001
        assert np.all(err[normal] <= (2.0 ** -4 + 1e-6) * np.abs(x32[normal]))
        assert np.all(err[~normal] <= (2.0 ** -10 + 1e-6) * scale_of[~normal])

    sq_b, sk_b, sv_b = np.empty((L, H, d)), np.empty((L, H, d)), np.empty((L, H, d))
    for h in range(H):
        for l in range(L):
            assert sq[l, h] == np.float32(np.abs(x32[l, h]).max() / np.float32(448))
            sq_b[l, h] = sq[l, h]
        for j in range(3):
            g = x32[j * blk:(j + 1) * blk, h]
            assert sk[h, j] == np.float32(np.abs(g).max() / np.float32(448))
            sk_b[j * blk:(j + 1) * blk, h] = sk[h, j]
        for c in range(d):
            assert sv[h, c] == np.float32(np.abs(x32[:, h, c]).max() / np.float32(448))
            sv_b[:, h, c] = sv[h, c]
    check(q8, sq_b)
    check(k8, sk_b)
    check(v8, sv_b)


def test_attention_8bit_channel_scales_keep_relative_accuracy():
    # Value channels of very different magnitudes: every output channel keeps E4M3
    # relative accuracy (one scale per tensor would zero the small channels).
    L, H, d = 384, 1, 32
    q = rng.standard_normal((L, H, d))
    k = rng.standard_normal((L, H, d)) * np.repeat([0.3, 1.0, 2.0], 128)[:, None, None]
    v = rng.standard_normal((L, H, d)) * np.exp(rng.uniform(-9, 9, d))[None, None, :]
    o8 = O.self_attention_8bit(q, k, v)
    ref = O.attention(q, k, v)
    rel = np.abs(o8 - ref) / np.abs(O.attention(q, k, np.abs(v)))
    assert rel.max() < 0.25 and np.median(rel) < 0.05


def test_fp8_block_variant_close_to_exact_and_zero_gates_reduce_to_exact():
    s = synth.TINY
    w = synth.make_weights(s, 0)
    inp = synth.make_inputs(s, 0)
    x = O.patchify(inp["latent"], w["patch_w"], w["patch_b"])[0]
    ctx = O.text_projection(inp["text"][:1], w)[0]
    blk = w["blocks"][0]
    mods = np.zeros((6, s.dim)) + 0.1
    exact = O.dit_block(x, mods, blk, ctx, None, O.Hyper.of(s))
    for bits in (1, 2, 3):
        y = O.dit_block(x, mods, blk, ctx, None, O.Hyper.of(s.replace(fp8=bits)))
        d = (y - x) - (exact - x)
        rel = np.sqrt((d ** 2).mean() / ((exact - x) ** 2).mean())
        assert 1e-4 < rel < 0.08, (bits, rel)
    # gates 0: self-attention and FFN contribute nothing, only cross-attention (not 8-bit)
    mods0 = mods.copy(); mods0[2] = 0.0; mods0[5] = 0.0
    y0 = O.dit_block(x, mods0, blk, ctx, None, O.Hyper.of(s.replace(fp8=3)))
    assert np.allclose(y0, O.dit_block(x, mods0, blk, ctx, None, O.Hyper.of(s)), rtol=0, atol=1e-12)


# ---------------------------------------------------------------- cross-attention and head

def _cross_weights(D, rng_, **over):
    blk = {"cq_w": rng_.normal(size=(D, D)) * 0.3, "cq_b": rng_.normal(size=D) * 0.1,
           "ckv_w": rng_.normal(size=(2 * D, D)) * 0.3, "ckv_b": rng_.normal(size=2 * D) * 0.1,
           "co_w": rng_.normal(size=(D, D)) * 0.3, "co_b": rng_.normal(size=D) * 0.1}
    blk.update(over)
    return blk


def test_cross_attention_single_text_token_is_its_value_projection():
    # One key: every softmax row is exactly 1, so each output row is the output projection
    # of that token's value half (rows D..2D of the key/value projection), whatever x is.
    # A swap of the key and value halves, a dropped bias or a missing output projection
    # changes the result.
    D, H = 12, 3
    r = np.random.default_rng(7)
    blk = _cross_weights(D, r)
    hp = O.Hyper(D, H, (1, 1, 1))
    ctx = r.normal(size=(1, D))
    x = r.normal(size=(5, D)) * 2.0
    v = np.array([sum(blk["ckv_w"][D + n, c] * ctx[0, c] for c in range(D)) + blk["ckv_b"][D + n]
                  for n in range(D)])
    expect = np.array([sum(blk["co_w"][n, c] * v[c] for c in range(D)) + blk["co_b"][n] for n in range(D)])
    out = O.cross_attention(x, blk, ctx, None, hp)
    assert np.allclose(out, np.broadcast_to(expect, out.shape), atol=1e-12)


def test_cross_attention_two_keys_logistic_closed_form():
    # Two text tokens, a query fixed by the bias (cq_w = 0), identity value and output
    # projections: per head, the output is sigmoid(z) v0 + sigmoid(-z) v1 with
    # z = q_h . (k0_h - k1_h) / sqrt(d).  Pins which half of ckv_w makes keys, the
    # 1/sqrt(d) scale, and that heads do not mix.
    D, H = 8, 2
    d = D // H
    r = np.random.default_rng(11)
    q = np.array([0.5, -1.0, 0.25, 2.0, -0.75, 0.5, 1.5, -0.25])
    Wk = r.normal(size=(D, D))
    blk = {"cq_w": np.zeros((D, D)), "cq_b": q,
           "ckv_w": np.concatenate([Wk, np.eye(D)]), "ckv_b": np.zeros(2 * D),
           "co_w": np.eye(D), "co_b": np.zeros(D)}
    ctx = r.normal(size=(2, D))
    k = ctx @ Wk.T
    expect = np.empty(D)
    for h in range(H):
        sl = slice(h * d, (h + 1) * d)
        z = float(q[sl] @ (k[0, sl] - k[1, sl])) / math.sqrt(d)
        p0 = 1.0 / (1.0 + math.exp(-z))
        expect[sl] = p0 * ctx[0, sl] + (1.0 - p0) * ctx[1, sl]
    out = O.cross_attention(r.normal(size=(3, D)), blk, ctx, None, O.Hyper(D, H, (1, 1, 1)))
    assert np.allclose(out, np.broadcast_to(expect, out.shape), atol=1e-13)


def test_cross_attention_query_layer_norm():
    # The query passes through a LayerNorm: a positive scale and a constant shift of each
    # row of x leave the output unchanged (up to eps), while a change of x's shape does not.
    D, H = 16, 4
    r = np.random.default_rng(13)
    blk = _cross_weights(D, r)
    hp = O.Hyper(D, H, (1, 1, 1))
    ctx = r.normal(size=(6, D))
    x = r.normal(size=(4, D))
    a = np.array([3.0, 0.5, 7.0, 1.5])[:, None]
    c = np.array([10.0, -4.0, 0.25, 100.0])[:, None]
    out = O.cross_attention(x, blk, ctx, None, hp)
    assert np.allclose(O.cross_attention(a * x + c, blk, ctx, None, hp), out, atol=1e-6)
    assert not np.allclose(O.cross_attention(x ** 3, blk, ctx, None, hp), out, atol=1e-3)


def test_cross_attention_decoupled_one_token_each_is_sum_of_values():
    # One text and one image token: two separate softmaxes (each exactly 1), so the output
    # is the output projection of v_text + v_image; one joint softmax over the
    # concatenated context would average them instead.
    D, H = 8, 2
    r = np.random.default_rng(17)
    blk = _cross_weights(D, r)
    blk["ckvi_w"], blk["ckvi_b"] = r.normal(size=(2 * D, D)), r.normal(size=2 * D)
    ct, ci = r.normal(size=(1, D)), r.normal(size=(1, D))
    vt = blk["ckv_w"][D:] @ ct[0] + blk["ckv_b"][D:]
    vi = blk["ckvi_w"][D:] @ ci[0] + blk["ckvi_b"][D:]
    expect = blk["co_w"] @ (vt + vi) + blk["co_b"]
    out = O.cross_attention(r.normal(size=(3, D)), blk, ct, ci, O.Hyper(D, H, (1, 1, 1)))
    assert np.allclose(out, np.broadcast_to(expect, out.shape), atol=1e-12)


def test_head_layer_norm_modulation_and_projection_closed_form():
    # Rows [a+b, a-b, a+b, a-b] have mean a and variance b^2, so LN gives
    # [1, -1, 1, -1] * b / sqrt(b^2 + eps).  With (shift, scale) = hm and a 4-cycle
    # permutation as the projection, each output is LN * (1 + scale) + shift at the
    # permuted index plus the bias: a swapped shift/scale, a transposed weight or a
    # missing LN changes it.
    eps = 1e-6
    x = np.array([[3.0 + 2.0, 3.0 - 2.0, 3.0 + 2.0, 3.0 - 2.0],
                  [-1.0 + 0.5, -1.0 - 0.5, -1.0 + 0.5, -1.0 - 0.5]])
    bs = np.array([2.0, 0.5])
    shift = np.array([0.1, -0.2, 0.3, 0.05])
    scale = np.array([1.0, 0.0, -0.5, 2.0])
    perm = [1, 2, 3, 0]  # output n reads modulated feature perm[n]
    w = {"head_w": np.eye(4)[perm], "head_b": np.array([0.01, 0.02, 0.03, 0.04])}
    out = O.head(x, np.stack([shift, scale]), w, eps)
    sign = np.array([1.0, -1.0, 1.0, -1.0])
    for r_ in range(2):
        ln = sign * bs[r_] / math.sqrt(bs[r_] ** 2 + eps)
        mod = ln * (1.0 + scale) + shift
        assert np.allclose(out[r_], [mod[perm[n]] + w["head_b"][n] for n in range(4)], atol=1e-14)
    # zero modulation and identity projection: the head is the plain LayerNorm
    w0 = {"head_w": np.eye(4), "head_b": np.zeros(4)}
    out0 = O.head(x, np.zeros((2, 4)), w0, eps)
    assert np.allclose(out0[0], sign * 2.0 / math.sqrt(4.0 + eps), atol=1e-15)

"""CPU fp64 oracle of the Wan DiT denoising step.

TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check in
``__graft_entry__.smoke()`` and the CPU-baseline / reference arm of
``bench.py`` may import or run this module.  The CUDA path never does, and the
two share no code: this file imports numpy and scipy only.

Every function is the plain definition of one step, in float64, written from
these sources (cited by title and section):

* [Method] hyper.ai summary of "Wan: Open and Advanced Large-Scale Video
  Generative Models" (arXiv 2503.20314), section "方法" (Method): the VAE
  compression, the DiT (patchify with a (1,2,2) 3D conv into (B, L, D),
  transformer blocks with text cross-attention, an MLP of Linear + SiLU on the
  time embedding predicting six modulation parameters, a depatchify module),
  and flow matching (velocity of the linear path between data x1 and noise x0,
  MSE loss).
* [Code] zizhi168.cn "阿里Wan 2.1视频生成模型深度剖析", section "核心代码实现亮点"
  (core code highlights): the classifier-free guidance combination, the I2V
  mask/latent concatenation, CLIP context concatenated ahead of the text
  context, DiT-style modulation with self- and cross-attention per block, and
  ``rope_apply(q, grid_sizes, freqs)`` on q and k before flash attention.
* [I2V] x-humanoid.csdn.net reading notes on the Wan report, section 1.1
  "模型设计": noise latent, condition latent and mask concatenated on channels,
  an extra zero-initialised input projection, CLIP features through a 3-layer
  MLP injected by decoupled cross-attention.
* [Sampler] kwkr.cn hands-on article, sections 3.2 and 4.4: Euler integration of
  the learned velocity field, about 20 steps, ``latent = latent + v*dt``.

Where these pages are silent the plainest reading is taken; each reading is
named where it is used (READING: ...).

Parity pins: every function here is checked by tests/test_oracle_pins.py
against closed forms, brute force, invariants and special cases.  The full
composition (``dit_forward`` over 30 blocks, ``sample``, and the 8-bit block)
has no printed worked example: beyond the pins of its parts and the zero-gate
identity it is "parity unpinned".
"""
from __future__ import annotations

import numpy as np
from scipy.special import erf

f64 = np.float64


# ---------------------------------------------------------------- primitives

def silu(x):
    """SiLU(x) = x * sigmoid(x): the activation of the time-embedding MLP [Method]."""
    x = np.asarray(x, f64)
    return x / (1.0 + np.exp(-x))


def gelu(x):
    """GELU in its exact erf form, x * Phi(x).  READING: the pages do not name the
    FFN activation's variant; the erf form is the definition."""
    x = np.asarray(x, f64)
    return 0.5 * x * (1.0 + erf(x / np.sqrt(2.0)))


def gelu_tanh(x):
    """The tanh approximation of GELU, 0.5 x (1 + tanh(sqrt(2/pi) (x + 0.044715 x^3))).
    Variant (not on the pages): selected by the gelu_tanh flag for fidelity with released
    checkpoints that use it."""
    x = np.asarray(x, f64)
    return 0.5 * x * (1.0 + np.tanh(np.sqrt(2.0 / np.pi) * (x + 0.044715 * x ** 3)))


def rms_norm(x, w, eps):
    """RMSNorm over the last axis with a learned weight: x / sqrt(mean(x^2) + eps) * w.
    Variant (not on the pages): selected by the qk_norm flag, applied to the full width
    of q and of k before RoPE."""
    x = np.asarray(x, f64)
    return x / np.sqrt((x * x).mean(axis=-1, keepdims=True) + eps) * np.asarray(w, f64)


def linear(x, w, b=None):
    """nn.Linear: x [..., in] times w [out, in] transposed, plus bias [out]."""
    y = np.asarray(x, f64) @ np.asarray(w, f64).T
    if b is not None:
        y = y + np.asarray(b, f64)
    return y


def layer_norm(x, eps):
    """LayerNorm over the last axis with biased variance and no affine.
    READING: eps = 1e-6; the modulated norms carry no affine parameters."""
    x = np.asarray(x, f64)
    mu = x.mean(axis=-1, keepdims=True)
    var = ((x - mu) ** 2).mean(axis=-1, keepdims=True)
    return (x - mu) / np.sqrt(var + eps)


def modulate(y, shift, scale):
    """DiT-style modulation y * (1 + scale) + shift [Code, attention paragraph]."""
    return y * (1.0 + scale) + shift


# ---------------------------------------------------------------- patchify

def patchify_tokens(lat):
    """Cut the latent [B, C, F, H, W] into (1,2,2) patches.

    Returns [B, L, C*4] with token order (f, i, j), j fastest, and feature order
    (c, di, dj):  p[b, (f*Hp + i)*Wp + j, c*4 + di*2 + dj] = lat[b, c, f, 2i+di, 2j+dj].
    """
    lat = np.asarray(lat, f64)
    B, C, F, H, W = lat.shape
    Hp, Wp = H // 2, W // 2
    p = lat.reshape(B, C, F, Hp, 2, Wp, 2).transpose(0, 2, 3, 5, 1, 4, 6)
    return p.reshape(B, F * Hp * Wp, C * 4)


def patchify(lat, w, b):
    """The DiT's patchify module: a 3D conv with kernel = stride = (1,2,2) turning the
    latent into the sequence (B, L, D) [Method, DiT paragraph].  w is the conv weight
    flattened to [D, C*4] (index c*4 + di*2 + dj)."""
    return linear(patchify_tokens(lat), w, b)


def unpatchify(tok, C, F, H, W):
    """The depatchify module [Method]: the inverse scatter of ``patchify_tokens``.
    tok [B, L, C*4] -> [B, C, F, H, W]."""
    tok = np.asarray(tok, f64)
    B = tok.shape[0]
    Hp, Wp = H // 2, W // 2
    t = tok.reshape(B, F, Hp, Wp, C, 2, 2).transpose(0, 4, 1, 2, 5, 3, 6)
    return t.reshape(B, C, F, H, W)


# ---------------------------------------------------------------- time embedding

def sinusoid(t, dim=256):
    """Frequency embedding of the timestep.  READING (pages silent): tau = 1000*t,
    s = [cos(tau*w_k), sin(tau*w_k)] for k < dim/2 with w_k = 10000^(-k/(dim/2))."""
    half = dim // 2
    k = np.arange(half, dtype=f64)
    omega = 10000.0 ** (-k / half)
    tau = 1000.0 * np.atleast_1d(np.asarray(t, f64))
    ang = tau[:, None] * omega[None, :]
    return np.concatenate([np.cos(ang), np.sin(ang)], axis=-1)


def time_embedding(t, w, dim, freq_dim=256):
    """The MLP of Linear and SiLU layers on the time embedding that predicts six
    modulation parameters, shared by all blocks [Method, DiT paragraph; shared
    AdaLN ablation in the experiments list].

    Returns e [B, D], e0 [B, 6, D] (shift1, scale1, gate1, shift2, scale2, gate2)
    and the head modulation hm [B, 2, D] (shift, scale).
    READING: e = W2 SiLU(W1 s + b1) + b2; e0 = Wm SiLU(e) + bm;
    hm = Whm SiLU(e) + bhm.
    """
    s = sinusoid(t, freq_dim)
    e = linear(silu(linear(s, w["t1_w"], w["t1_b"])), w["t2_w"], w["t2_b"])
    e0 = linear(silu(e), w["m_w"], w["m_b"]).reshape(-1, 6, dim)
    hm = linear(silu(e), w["hm_w"], w["hm_b"]).reshape(-1, 2, dim)
    return e, e0, hm


# ---------------------------------------------------------------- 3D RoPE

def rope_axis_dims(d):
    """READING of ``rope_apply(q, grid_sizes, freqs)`` [Code]: the head dim splits
    into [frame | height | width] parts of sizes (d - 4*floor(d/6), 2*floor(d/6),
    2*floor(d/6)); d = 128 gives (44, 42, 42), d = 64 gives (24, 20, 20)."""
    dh = 2 * (d // 6)
    return d - 2 * dh, dh, dh


def token_positions(grid, tokens=None):
    """Integer (f, i, j) grid position of each token index l = (f*Hg + i)*Wg + j."""
    Fg, Hg, Wg = grid
    l = np.arange(Fg * Hg * Wg) if tokens is None else np.asarray(tokens)
    return np.stack([l // (Hg * Wg), (l // Wg) % Hg, l % Wg], axis=-1)


def rope_angles(pos, d, theta):
    """Angles [n, d/2]: pair j of axis a rotates by pos_a * theta^(-2j/d_a)."""
    dims = rope_axis_dims(d)
    pos = np.asarray(pos, f64)
    parts = []
    for a in range(3):
        n = dims[a] // 2
        omega = theta ** (-2.0 * np.arange(n, dtype=f64) / dims[a])
        parts.append(pos[:, a:a + 1] * omega[None, :])
    return np.concatenate(parts, axis=1)


def rope3d(x, pos, theta=10000.0):
    """Rotate adjacent pairs (2m, 2m+1) of x [n, H, d] by the 3D-RoPE angle of each
    token's (f, i, j) position: (x0 cos - x1 sin, x0 sin + x1 cos)."""
    x = np.asarray(x, f64)
    ang = rope_angles(pos, x.shape[-1], theta)[:, None, :]
    c, s = np.cos(ang), np.sin(ang)
    x0, x1 = x[..., 0::2], x[..., 1::2]
    out = np.empty_like(x)
    out[..., 0::2] = x0 * c - x1 * s
    out[..., 1::2] = x0 * s + x1 * c
    return out


# ---------------------------------------------------------------- attention

def attention(q, k, v, chunk=2048):
    """softmax(q k^T / sqrt(d)) v per head, full and bidirectional (no mask).
    q [Lq, H, d], k and v [Lk, H, d] -> [Lq, H, d].  Query rows are independent, so
    they are evaluated ``chunk`` rows at a time; the max subtraction is the exact
    shift invariance of softmax."""
    q, k, v = (np.asarray(a, f64) for a in (q, k, v))
    Lq, H, d = q.shape
    out = np.empty((Lq, H, v.shape[-1]), f64)
    for h in range(H):
        kh, vh = k[:, h, :], v[:, h, :]
        for r0 in range(0, Lq, chunk):
            s = q[r0:r0 + chunk, h, :] @ kh.T / np.sqrt(d)
            s = s - s.max(axis=1, keepdims=True)
            p = np.exp(s)
            p = p / p.sum(axis=1, keepdims=True)
            out[r0:r0 + chunk, h, :] = p @ vh
    return out


# ---------------------------------------------------------------- 8-bit variant
# [Method] hyper.ai summary, section 方法 (Method), the inference paragraph: FP8 GEMMs and
# an 8-bit FlashAttention speed up the DiT.  The pages fix neither the 8-bit format nor
# the scaling; READING (the plainest one that the hardware runs natively): OCP FP8 E4M3
# codes, round to nearest even with saturation at +-448, each tensor scaled by its
# absolute maximum over a group so that the maximum maps to 448:
#   GEMM activations per row (token), GEMM weights per output channel;
#   attention q per (token, head), k per (head, 128-key block), v per (head, channel).
# The quantisation decisions are taken in fp32, like the kernels: inv = fl32(448 / amax),
# code = e4m3(fl32(x * inv)), dequantisation scale s = fl32(amax / 448) (0 when amax = 0).

E4M3_MAX = 448.0


def e4m3_decode(code):
    """Value of an E4M3 code (1 sign, 4 exponent bits with bias 7, 3 mantissa bits; no
    infinities; exponent 15 with mantissa 7 is NaN; exponent 0 holds the subnormals
    M * 2^-9)."""
    c = np.asarray(code, np.int64) & 0xFF
    sgn = np.where(c & 0x80, -1.0, 1.0)
    E, M = (c >> 3) & 0xF, c & 7
    val = np.where(E == 0, M * 2.0 ** -9, (1.0 + M / 8.0) * 2.0 ** (E.astype(f64) - 7.0))
    val = np.where((E == 15) & (M == 7), np.nan, val)
    return sgn * val


def e4m3_round(x):
    """Nearest E4M3 value to x (ties to even), magnitudes above 448 saturated to 448.
    The grid spacing in the binade [2^e, 2^(e+1)) is 2^(e-3) for e >= -6 and 2^-9 below."""
    x = np.asarray(x, f64)
    a = np.abs(x)
    _, ex = np.frexp(np.where(a > 0, a, 1.0))          # a = m 2^ex, m in [0.5, 1)
    e = np.maximum(ex.astype(f64) - 1.0, -6.0)         # floor(log2 a), floored at -6
    ulp = 2.0 ** (e - 3.0)
    r = np.minimum(np.rint(a / ulp) * ulp, E4M3_MAX)   # a / ulp is exact: rint = ties-to-even
    return np.where(a > 0, np.sign(x) * r, 0.0 * x)


def e4m3_encode(x):
    """E4M3 code of e4m3_round(x) (the byte the kernels store)."""
    r = e4m3_round(x)
    a = np.abs(r)
    _, ex = np.frexp(np.where(a > 0, a, 1.0))
    e = ex.astype(np.int64) - 1
    normal = a >= 2.0 ** -6
    mant_n = np.rint((a / np.ldexp(1.0, e) - 1.0) * 8.0).astype(np.int64)
    code_n = ((e + 7) << 3) | mant_n
    code_s = np.rint(a / 2.0 ** -9).astype(np.int64)
    code = np.where(normal, code_n, code_s)
    return (code | np.where(np.signbit(r), 0x80, 0)).astype(np.uint8)


def _f32(x):
    return np.asarray(x, np.float32)


def quant_scale(amax):
    """(inv, s) for a group absolute maximum: inv = fl32(448 / amax) multiplies the values
    before rounding, s = fl32(amax / 448) dequantises.  An all-zero group gets inv = s = 0."""
    amax = _f32(amax)
    safe = np.where(amax > 0, amax, np.float32(1))
    inv = np.where(amax > 0, np.float32(E4M3_MAX) / safe, np.float32(0)).astype(np.float32)
    s = (amax / np.float32(E4M3_MAX)).astype(np.float32)
    return inv, s


def quantize_groups(x, axes):
    """Codes and dequantisation scales of x with one scale per group; ``axes`` are the
    axes each group spans (reduced by the absolute maximum).  x is taken as fp32."""
    x32 = _f32(x)
    amax = np.abs(x32).max(axis=axes, keepdims=True)
    inv, s = quant_scale(amax)
    codes = e4m3_encode((x32 * inv).astype(np.float32))
    return codes, s


def quant_rows(x):
    """Per-row E4M3 quantisation of a [rows, K] matrix: codes [rows, K], scales [rows]."""
    c, s = quantize_groups(x, axes=(-1,))
    return c, s[..., 0]


def dequant(codes, s):
    return e4m3_decode(codes) * np.asarray(s, f64)


def linear_fp8(a_codes, sa, w_codes, sw, b=None):
    """FP8 GEMM: (A8 sa) (W8 sw)^T + b, every product exact, accumulation in fp64.
    a_codes [M, K] with row scales sa [M]; w_codes [N, K] with per-output-channel scales
    sw [N]."""
    y = (e4m3_decode(a_codes) @ e4m3_decode(w_codes).T) * np.asarray(sa, f64)[:, None] * np.asarray(sw, f64)[None, :]
    if b is not None:
        y = y + np.asarray(b, f64)
    return y


def quant_attn_q(q):
    """q [L, H, d] -> codes [L, H, d], scales [L, H] (one per token and head)."""
    c, s = quantize_groups(q, axes=(-1,))
    return c, s[..., 0]


def quant_attn_k(k, block=128):
    """k [L, H, d] -> codes [L, H, d], scales [H, ceil(L/block)] (one per head and block
    of ``block`` consecutive keys; a ragged last block spans the keys it has)."""
    k32 = _f32(k)
    L, H, d = k32.shape
    nb = (L + block - 1) // block
    codes = np.empty(k32.shape, np.uint8)
    scales = np.empty((H, nb), np.float32)
    for j in range(nb):
        c, s = quantize_groups(k32[j * block:(j + 1) * block], axes=(0, 2))
        codes[j * block:(j + 1) * block] = c
        scales[:, j] = s[0, :, 0]
    return codes, scales


def quant_attn_v(v):
    """v [L, H, d] -> codes [L, H, d], scales [H, d] (one per head and channel, over all
    keys)."""
    c, s = quantize_groups(v, axes=(0,))
    return c, s[0]


def attention_8bit(q8, sq, k8, sk, v8, sv, block=128, kv_len=None):
    """Attention on the dequantised 8-bit operands, softmax and products in fp64:
    softmax(Q K^T / sqrt(d)) V with Q = dec(q8) sq, K = dec(k8) sk (per key block),
    V = dec(v8) sv; only the first kv_len keys take part.  The kernel's own rounding of
    the probabilities to E4M3 is not modelled here: its effect is bounded by
    2^-4 * attention(q, k, |V|) per element (relative error of E4M3 rounding in the
    normal range), which the parity tests use."""
    Q = dequant(q8, np.asarray(sq)[..., None])
    blk_of_key = np.arange(k8.shape[0]) // block
    K = e4m3_decode(k8) * np.asarray(sk, f64).T[blk_of_key][:, :, None]
    V = e4m3_decode(v8) * np.asarray(sv, f64)[None]
    if kv_len is not None:
        K, V = K[:kv_len], V[:kv_len]
    return attention(Q, K, V)


def self_attention_8bit(q, k, v, kv_len=None):
    """The 8-bit self-attention of the variant: quantise q, k, v as above, then
    attention_8bit.  Returns (o, (Q, K, V) dequantised) for bound computations."""
    q8, sq = quant_attn_q(q)
    k8, sk = quant_attn_k(k)
    v8, sv = quant_attn_v(v)
    return attention_8bit(q8, sq, k8, sk, v8, sv, kv_len=kv_len)


def heads(x, H):
    x = np.asarray(x, f64)
    return x.reshape(x.shape[0], H, x.shape[1] // H)


# ---------------------------------------------------------------- block

class Hyper:
    """The scalars a block needs."""

    def __init__(self, dim, heads, grid, theta=10000.0, eps=1e-6, qk_norm=False, gelu_tanh=False, fp8=0):
        self.dim, self.heads, self.grid, self.theta, self.eps = dim, heads, grid, theta, eps
        self.qk_norm, self.gelu_tanh = qk_norm, gelu_tanh
        self.fp8 = fp8  # bit 0: 8-bit self-attention; bit 1: FP8 QKV and FFN-up GEMMs

    @classmethod
    def of(cls, shape):
        return cls(shape.dim, shape.heads, shape.grid, shape.theta, shape.eps,
                   getattr(shape, "qk_norm", False), getattr(shape, "gelu_tanh", False),
                   getattr(shape, "fp8", 0))


def cross_attention(xr, blk, ctx_txt, ctx_img, hp):
    """Cross-attention to the text context [Method; Code], plus for I2V the CLIP image
    context injected by decoupled cross-attention [I2V 1.1; Code, img_emb paragraph].
    READING: no modulation and no gate on this sub-layer; its norm is a plain LN;
    decoupled = the text and image attentions use one shared query and output
    projection and separate key/value projections, and their outputs are summed."""
    D, H = hp.dim, hp.heads
    qc = heads(linear(layer_norm(xr, hp.eps), blk["cq_w"], blk["cq_b"]), H)
    kv = linear(ctx_txt, blk["ckv_w"], blk["ckv_b"])
    o = attention(qc, heads(kv[:, :D], H), heads(kv[:, D:], H))
    if ctx_img is not None:
        kvi = linear(ctx_img, blk["ckvi_w"], blk["ckvi_b"])
        o = o + attention(qc, heads(kvi[:, :D], H), heads(kvi[:, D:], H))
    return linear(o.reshape(o.shape[0], D), blk["co_w"], blk["co_b"])


def dit_block(x, mods, blk, ctx_txt, ctx_img, hp, rows=None, trace=None):
    """One transformer block on one sample x [L, D].

    mods [6, D] = (shift1, scale1, gate1, shift2, scale2, gate2), the shared
    time-embedding output plus this block's learned bias [Method].  Order
    self-attention -> cross-attention -> FFN [Code: "每个网络块包含一组自注意力层和一组
    交叉注意力层"]; READING: the FFN is Linear D->F, GELU, Linear F->D.

    ``rows``: when given, only these output rows are produced.  Self-attention
    still sees every key and value; all later steps act row by row, so the result
    equals the full block's rows.  ``trace``: optional dict that receives the
    intermediate values at those rows.
    """
    D, H = hp.dim, hp.heads
    x = np.asarray(x, f64)
    mods = np.asarray(mods, f64)
    sh1, sc1, g1, sh2, sc2, g2 = mods
    L = x.shape[0]
    rows = np.arange(L) if rows is None else np.asarray(rows)
    pos = token_positions(hp.grid)
    wq, wk, wv = blk["qkv_w"][:D], blk["qkv_w"][D:2 * D], blk["qkv_w"][2 * D:]
    bq, bk, bv = blk["qkv_b"][:D], blk["qkv_b"][D:2 * D], blk["qkv_b"][2 * D:]

    # self-attention with 3D RoPE on q and k [Code, flash_attention call]
    y = modulate(layer_norm(x, hp.eps), sh1, sc1)
    if hp.fp8 & 2:  # variant: FP8 GEMM, activations per token, weights per output channel
        y8, sy = quant_rows(y)
        wq8, swq = quant_rows(wq)
        wk8, swk = quant_rows(wk)
        wv8, swv = quant_rows(wv)
        kl, ql = linear_fp8(y8, sy, wk8, swk, bk), linear_fp8(y8[rows], sy[rows], wq8, swq, bq)
        vl = linear_fp8(y8, sy, wv8, swv, bv)
    else:
        kl, ql, vl = linear(y, wk, bk), linear(y[rows], wq, bq), linear(y, wv, bv)
    if hp.qk_norm:  # variant: RMSNorm of the full-width q and k before RoPE
        kl, ql = rms_norm(kl, blk["norm_k_w"], hp.eps), rms_norm(ql, blk["norm_q_w"], hp.eps)
    k = rope3d(heads(kl, H), pos, hp.theta)
    v = heads(vl, H)
    q = rope3d(heads(ql, H), pos[rows], hp.theta)
    if hp.fp8 & 1:  # variant: 8-bit self-attention
        o = self_attention_8bit(q, k, v).reshape(len(rows), D)
    else:
        o = attention(q, k, v).reshape(len(rows), D)
    xr = x[rows] + g1 * linear(o, blk["o_w"], blk["o_b"])
    if trace is not None:
        trace.update(y1=y[rows], q=q.reshape(len(rows), D), k=k[rows].reshape(len(rows), D),
                     v=v[rows].reshape(len(rows), D), attn=o, x_sa=xr)

    xr = xr + cross_attention(xr, blk, ctx_txt, ctx_img, hp)

    y2 = modulate(layer_norm(xr, hp.eps), sh2, sc2)
    if hp.fp8 & 2:
        y28, sy2 = quant_rows(y2)
        w18, sw1 = quant_rows(blk["f1_w"])
        u = linear_fp8(y28, sy2, w18, sw1, blk["f1_b"])
    else:
        u = linear(y2, blk["f1_w"], blk["f1_b"])
    h = (gelu_tanh if hp.gelu_tanh else gelu)(u)
    if trace is not None:
        trace.update(x_ca=xr, y2=y2)
    xr = xr + g2 * linear(h, blk["f2_w"], blk["f2_b"])
    return xr


def head(x, hm, w, eps):
    """Output head before depatchify.  READING: LN, modulation by (shift, scale)
    from the time embedding, then Linear D -> C_out*4."""
    y = modulate(layer_norm(x, eps), hm[0], hm[1])
    return linear(y, w["head_w"], w["head_b"])


def text_projection(text, w):
    """Text-context projection from the umT5 width to D.  READING: Linear, GELU, Linear."""
    return linear(gelu(linear(text, w["txt1_w"], w["txt1_b"])), w["txt2_w"], w["txt2_b"])


def dit_forward(latent, t, ctx_txt, ctx_img, w, shape, rows=None, on_block=None, trace=None):
    """The DiT's velocity prediction v [B, C_out, F, H, W] for latent [B, C_in, F, H, W],
    timesteps t [B] and contexts ctx_txt [B, Lt, D] (ctx_img [B, Li, D] or None).

    ``rows`` (single-block models only): compute the head output at these tokens
    and return it as [B, len(rows), C_out*4] together with the block output rows.
    ``on_block(b, i, x)`` is called after every block (checkpoints).
    """
    hp = Hyper.of(shape)
    latent = np.asarray(latent, f64)
    B = latent.shape[0]
    x = patchify(latent, w["patch_w"], w["patch_b"])
    _, e0, hm = time_embedding(np.broadcast_to(np.asarray(t, f64), (B,)), w, shape.dim, shape.freq_dim)
    if rows is not None:
        assert len(w["blocks"]) == 1, "row sampling needs a single block"
        outs, xs = [], []
        for b in range(B):
            blk = w["blocks"][0]
            ci = None if ctx_img is None else ctx_img[b]
            tr = None if trace is None else {}
            xr = dit_block(x[b], e0[b] + blk["mod"], blk, ctx_txt[b], ci, hp, rows=rows, trace=tr)
            if trace is not None:
                tr["x0"] = x[b][rows]
                trace.setdefault("per_batch", []).append(tr)
            xs.append(xr)
            outs.append(head(xr, hm[b], w, shape.eps))
        return np.stack(outs), np.stack(xs)
    v = []
    for b in range(B):
        xb = x[b]
        for i, blk in enumerate(w["blocks"]):
            ci = None if ctx_img is None else ctx_img[b]
            xb = dit_block(xb, e0[b] + blk["mod"], blk, ctx_txt[b], ci, hp)
            if on_block is not None:
                on_block(b, i, xb)
        v.append(unpatchify(head(xb, hm[b], w, shape.eps)[None], shape.c_out, shape.frames,
                            shape.height, shape.width)[0])
    return np.stack(v)


# ---------------------------------------------------------------- guidance + Euler

def cfg_combine(v_cond, v_uncond, guide_scale):
    """noise_pred = uncond + guide_scale * (cond - uncond) [Code, CFG snippet]."""
    v_cond, v_uncond = np.asarray(v_cond, f64), np.asarray(v_uncond, f64)
    return v_uncond + guide_scale * (v_cond - v_uncond)


def euler_step(x, v, dt):
    """One explicit Euler step of the flow ODE, x <- x + v*dt [Sampler 4.4].
    t runs from 1 (noise) to 0 (data); dt = t_next - t is negative."""
    return np.asarray(x, f64) + dt * np.asarray(v, f64)


def cfg_euler_step(x, v_cond, v_uncond, guide_scale, dt):
    return euler_step(x, cfg_combine(v_cond, v_uncond, guide_scale), dt)


def guided_step(x, t, dt, ctx, ctx_img, w, shape):
    """One guided denoising step: the DiT on [cond; uncond] with the same latent and
    timestep, then CFG and the Euler update of the predicted channels."""
    x = np.asarray(x, f64)
    lat = np.concatenate([x, x], axis=0)
    v = dit_forward(lat, np.array([t, t], f64), ctx, ctx_img, w, shape)
    return cfg_euler_step(x[:, :shape.c_out], v[0:1], v[1:2], shape.guide_scale, dt)


def timesteps(n):
    """Uniform schedule t_k = 1 - k/n, k = 0..n [Sampler 3.2: Euler, ~20 steps].
    READING: no timestep shift."""
    return 1.0 - np.arange(n + 1, dtype=f64) / n


def sample(x, ctx, ctx_img, w, shape, steps):
    """End-to-end Euler sampling from noise x at t = 1 to t = 0 [Sampler 4.4]."""
    ts = timesteps(steps)
    for k in range(steps):
        x = guided_step(x, ts[k], ts[k + 1] - ts[k], ctx, ctx_img, w, shape)
    return x

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
composition (``dit_forward`` over 30 blocks, ``sample``) has no printed worked
example: beyond the pins of its parts and the zero-gate identity it is
"parity unpinned".
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


def heads(x, H):
    x = np.asarray(x, f64)
    return x.reshape(x.shape[0], H, x.shape[1] // H)


# ---------------------------------------------------------------- block

class Hyper:
    """The scalars a block needs."""

    def __init__(self, dim, heads, grid, theta=10000.0, eps=1e-6, qk_norm=False, gelu_tanh=False):
        self.dim, self.heads, self.grid, self.theta, self.eps = dim, heads, grid, theta, eps
        self.qk_norm, self.gelu_tanh = qk_norm, gelu_tanh

    @classmethod
    def of(cls, shape):
        return cls(shape.dim, shape.heads, shape.grid, shape.theta, shape.eps,
                   getattr(shape, "qk_norm", False), getattr(shape, "gelu_tanh", False))


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
    kl, ql = linear(y, wk, bk), linear(y[rows], wq, bq)
    if hp.qk_norm:  # variant: RMSNorm of the full-width q and k before RoPE
        kl, ql = rms_norm(kl, blk["norm_k_w"], hp.eps), rms_norm(ql, blk["norm_q_w"], hp.eps)
    k = rope3d(heads(kl, H), pos, hp.theta)
    v = heads(linear(y, wv, bv), H)
    q = rope3d(heads(ql, H), pos[rows], hp.theta)
    o = attention(q, k, v).reshape(len(rows), D)
    xr = x[rows] + g1 * linear(o, blk["o_w"], blk["o_b"])
    if trace is not None:
        trace.update(y1=y[rows], q=q.reshape(len(rows), D), k=k[rows].reshape(len(rows), D),
                     v=v[rows].reshape(len(rows), D), attn=o, x_sa=xr)

    xr = xr + cross_attention(xr, blk, ctx_txt, ctx_img, hp)

    y2 = modulate(layer_norm(xr, hp.eps), sh2, sc2)
    h = (gelu_tanh if hp.gelu_tanh else gelu)(linear(y2, blk["f1_w"], blk["f1_b"]))
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

"""Seeded synthetic inputs for the Wan DiT denoising step.

This module draws numbers and names them; it holds none of the method's
arithmetic.  Both the CPU oracle (via the tests) and the CUDA path (via the
binding, the tests and the benchmark) take their inputs from here, so the two
sides see bit-identical values.

Generator: numpy's counter-based Philox4x64 bit generator, one independent
stream per tensor, keyed by SeedSequence([seed, crc32(name)]).  Normal draws are
numpy's float32 ziggurat sampler.  Both are platform independent, so a value
drawn here equals the value drawn on any other host with the same numpy.

Storage rounding: tensors the GPU keeps in bf16 (weights, biases, contexts in
the bf16 configurations) are rounded to the nearest bf16 value (ties to even)
and returned as float32 arrays holding exactly representable bf16 values, so the
oracle (fp64) and the kernels (bf16) start from the same numbers.

Shapes follow the Wan 2.1 technical report as summarised on the hyper.ai page
("方法", DiT paragraph: patchify kernel (1,2,2), sequence (B, L, D); VAE 4x8x8
compression) and the I2V design on the x-humanoid.csdn.net notes (section 1.1:
noise, condition latent and mask concatenated on channels; 257 CLIP tokens).
"""
from __future__ import annotations

import dataclasses
import zlib

import numpy as np

WEIGHT_STD = 0.02


@dataclasses.dataclass(frozen=True)
class DiTShape:
    """One workload: the DiT widths plus the latent/context geometry."""

    name: str
    dtype: str          # "bf16" or "f32": storage type of weights/activations
    batch: int          # DiT batch (2 = cond + uncond of one guided step)
    c_in: int           # latent channels fed to patchify
    c_out: int          # latent channels predicted
    frames: int         # latent F
    height: int         # latent H (even)
    width: int          # latent W (even)
    dim: int            # D
    heads: int          # H
    head_dim: int       # d
    ffn: int            # F (FFN hidden width)
    blocks: int         # number of transformer blocks
    text_len: int       # Lt
    text_dim: int       # raw text-embedding width fed to the text projection (0: context given at width D)
    img_len: int = 0    # Li (I2V image tokens, already at width D)
    freq_dim: int = 256
    theta: float = 10000.0
    eps: float = 1e-6
    guide_scale: float = 5.0
    dt: float = -0.05
    steps: int = 1      # sampling steps (20 for the end-to-end sampler)
    uncond_zero: bool = False   # uncond text embedding = zeros (tiny config)
    i2v: bool = False
    qk_norm: bool = False       # variant: RMSNorm (learned weight) on q and k before RoPE
    gelu_tanh: bool = False     # variant: tanh-form GELU in the FFN
    fp8: int = 0                # variant bits: 1 = 8-bit self-attention, 2 = FP8 QKV / FFN-up GEMMs

    @property
    def grid(self):
        return (self.frames, self.height // 2, self.width // 2)

    @property
    def tokens(self):
        f, h, w = self.grid
        return f * h * w

    def replace(self, **kw) -> "DiTShape":
        return dataclasses.replace(self, **kw)


# The workloads, by name:
#   tiny-f32                   one block, fp32, 16x3x8x8 latent -> 48 tokens, D=128, 2 heads of 64
#   wan1.3b-block              one 1.3B-shaped block, bf16, 480p latent 16x21x60x104 -> 32760 tokens
#   wan1.3b-30blk-guided-step  the 30-block 1.3B-shaped DiT, one guided step (cond + uncond)
#   wan14b-i2v-block           one 14B-shaped I2V block, 720p latent 36x21x90x160 -> 75600 tokens
#   wan1.3b-20step-sampler     the 30-block DiT, 20 guided Euler steps
WORKLOADS = {s.name: s for s in (
    DiTShape("tiny-f32", "f32", 2, 16, 16, 3, 8, 8, 128, 2, 64, 512, 1, 16, 128, uncond_zero=True),
    DiTShape("wan1.3b-block", "bf16", 1, 16, 16, 21, 60, 104, 1536, 12, 128, 8960, 1, 512, 4096),
    DiTShape("wan1.3b-30blk-guided-step", "bf16", 2, 16, 16, 21, 60, 104, 1536, 12, 128, 8960, 30, 512, 4096),
    DiTShape("wan14b-i2v-block", "bf16", 1, 36, 16, 21, 90, 160, 5120, 40, 128, 13824, 1, 512, 0,
             img_len=257, i2v=True),
    DiTShape("wan1.3b-20step-sampler", "bf16", 2, 16, 16, 21, 60, 104, 1536, 12, 128, 8960, 30, 512, 4096,
             steps=20),
)}
TINY = WORKLOADS["tiny-f32"]
BLOCK_1P3B = WORKLOADS["wan1.3b-block"]
STEP_1P3B = WORKLOADS["wan1.3b-30blk-guided-step"]
BLOCK_14B_I2V = WORKLOADS["wan14b-i2v-block"]
SAMPLER_1P3B = WORKLOADS["wan1.3b-20step-sampler"]


def _gen(seed: int, name: str) -> np.random.Generator:
    return np.random.Generator(np.random.Philox(np.random.SeedSequence([int(seed), zlib.crc32(name.encode())])))


def normal(seed: int, name: str, shape, std: float = 1.0) -> np.ndarray:
    a = _gen(seed, name).standard_normal(size=shape, dtype=np.float32)
    if std != 1.0:
        a *= np.float32(std)
    return a


def uniform(seed: int, name: str, shape, lo: float = 0.0, hi: float = 1.0) -> np.ndarray:
    a = _gen(seed, name).random(size=shape, dtype=np.float32)
    return (lo + (hi - lo) * a).astype(np.float32)


def round_bf16(a: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bf16 (ties to even); finite inputs only."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    r = (u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) & np.uint32(0xFFFF0000)
    return r.view(np.float32)


def store(shape: DiTShape, a: np.ndarray) -> np.ndarray:
    return round_bf16(a) if shape.dtype == "bf16" else np.ascontiguousarray(a, dtype=np.float32)


def block_weight_shapes(s: DiTShape):
    D, F = s.dim, s.ffn
    shapes = {
        "mod": (6, D),
        "qkv_w": (3 * D, D), "qkv_b": (3 * D,),
        "o_w": (D, D), "o_b": (D,),
        "cq_w": (D, D), "cq_b": (D,),
        "ckv_w": (2 * D, D), "ckv_b": (2 * D,),
        "co_w": (D, D), "co_b": (D,),
        "f1_w": (F, D), "f1_b": (F,),
        "f2_w": (D, F), "f2_b": (D,),
    }
    if s.img_len:
        shapes["ckvi_w"] = (2 * D, D)
        shapes["ckvi_b"] = (2 * D,)
    return shapes


def global_weight_shapes(s: DiTShape):
    D = s.dim
    shapes = {
        "patch_w": (D, s.c_in * 4), "patch_b": (D,),
        "t1_w": (D, s.freq_dim), "t1_b": (D,),
        "t2_w": (D, D), "t2_b": (D,),
        "m_w": (6 * D, D), "m_b": (6 * D,),
        "hm_w": (2 * D, D), "hm_b": (2 * D,),
        "head_w": (s.c_out * 4, D), "head_b": (s.c_out * 4,),
    }
    if s.text_dim:
        shapes.update({"txt1_w": (D, s.text_dim), "txt1_b": (D,), "txt2_w": (D, D), "txt2_b": (D,)})
    return shapes


def make_weights(s: DiTShape, seed: int = 0) -> dict:
    """Random-init weights ~N(0, 0.02), rounded to the storage type.

    For I2V the patchify columns of the 20 extra channels (condition latent and
    mask) start at zero, as the I2V design initialises its extra input projection.
    """
    w = {}
    for name, shp in global_weight_shapes(s).items():
        w[name] = store(s, normal(seed, name, shp, WEIGHT_STD))
    if s.i2v:
        w["patch_w"][:, 16 * 4:] = 0.0
    w["blocks"] = []
    for i in range(s.blocks):
        blk = {}
        for name, shp in block_weight_shapes(s).items():
            blk[name] = store(s, normal(seed, f"block{i}.{name}", shp, WEIGHT_STD))
        if s.qk_norm:  # RMSNorm weights around 1 (spread so that a mistake in them shows)
            for name in ("norm_q_w", "norm_k_w"):
                blk[name] = store(s, 1.0 + normal(seed, f"block{i}.{name}", (s.dim,), 0.1))
        w["blocks"].append(blk)
    return w


def make_inputs(s: DiTShape, seed: int = 0) -> dict:
    """Latent, timestep and contexts of one workload.

    latent   [1, c_in, F, H, W] float32 (shared by the cond and uncond branches)
    t        [1] float32 ~U(0,1) (the sampler overrides it with its schedule)
    text     [batch, Lt, text_dim] storage-rounded (raw text embedding, cond first)
             or, when text_dim == 0, ctx_txt [batch, Lt, D] already at width D
    ctx_img  [batch, Li, D] for I2V
    """
    F, H, W = s.frames, s.height, s.width
    inp = {}
    if s.i2v:
        noise = normal(seed, "latent.noise", (1, 16, F, H, W))
        cond = normal(seed, "latent.cond", (1, 16, F, H, W))
        mask = np.zeros((1, s.c_in - 32, F, H, W), np.float32)
        mask[:, :, 0] = 1.0
        inp["latent"] = np.concatenate([noise, cond, mask], axis=1)
    else:
        inp["latent"] = normal(seed, "latent", (1, s.c_in, F, H, W))
    inp["t"] = uniform(seed, "t", (1,))
    width = s.text_dim if s.text_dim else s.dim
    key = "text" if s.text_dim else "ctx_txt"
    parts = [store(s, normal(seed, "text.cond", (1, s.text_len, width)))]
    if s.batch > 1:
        if s.uncond_zero:
            parts.append(np.zeros((1, s.text_len, width), np.float32))
        else:
            parts.append(store(s, normal(seed, "text.uncond", (1, s.text_len, width))))
    inp[key] = np.concatenate(parts, axis=0)
    if s.img_len:
        inp["ctx_img"] = store(s, normal(seed, "ctx.img", (s.batch, s.img_len, s.dim)))
    return inp


def sample_rows(n_rows: int, count: int, seed: int = 0) -> np.ndarray:
    """Sorted distinct row indices to check at full size (always includes the last row)."""
    g = _gen(seed, f"rows.{n_rows}")
    count = min(count, n_rows)
    idx = g.choice(n_rows, size=count, replace=False)
    idx[-1] = n_rows - 1 if (n_rows - 1) not in idx else idx[-1]
    return np.unique(idx)

"""Thin Python binding of libwan (include/wan.h).

Argument marshalling only: every function forwards device pointers, sizes and the
current torch CUDA stream to the C entry point of the same name and raises WanError
on a non-zero status.  All arithmetic of the step runs in libwan's CUDA kernels; there
is no CPU or PyTorch fallback, and importing this module fails loudly when
libwan.so has not been built.  PyTorch is used for device memory and streams only.
"""
from __future__ import annotations

import ctypes as C
import os

import numpy as np
import torch

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libwan.so")

WAN_OK, WAN_ERR_INVALID_ARG, WAN_ERR_UNSUPPORTED, WAN_ERR_CUDA, WAN_ERR_TIMEOUT, WAN_ERR_WORKSPACE = 0, -1, -2, -3, -4, -5
WAN_BF16, WAN_F32, WAN_F16 = 0, 1, 2
WAN_EPI_STORE, WAN_EPI_GELU, WAN_EPI_RESIDUAL, WAN_EPI_GELU_TANH = 0, 1, 2, 3


class WanError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {lib.wan_status_string(status).decode()} ({status})")


def _load():
    if not os.path.exists(_LIB_PATH):
        raise ImportError(f"libwan.so is not built ({_LIB_PATH}); run "
                          "`python -m video_diffusion_transformer_04_b300._build`")
    return C.CDLL(_LIB_PATH)


lib = _load()

P, I, LL, F, SZ = C.c_void_p, C.c_int, C.c_longlong, C.c_float, C.c_size_t


class wan_dit_config(C.Structure):
    _fields_ = [("dtype", I), ("batch", I), ("c_in", I), ("c_out", I), ("frames", I), ("height", I), ("width", I),
                ("dim", I), ("heads", I), ("head_dim", I), ("ffn", I), ("blocks", I), ("text_len", I),
                ("img_len", I), ("freq_dim", I), ("theta", F), ("eps", F), ("qk_norm", I), ("gelu_tanh", I),
                ("fp8", I)]


_BLOCK_FIELDS = ["mod", "qkv_w", "qkv_b", "o_w", "o_b", "cq_w", "cq_b", "ckv_w", "ckv_b", "ckvi_w", "ckvi_b",
                 "co_w", "co_b", "f1_w", "f1_b", "f2_w", "f2_b", "norm_q_w", "norm_k_w",
                 "qkv_w8", "qkv_ws", "f1_w8", "f1_ws"]
_GLOBAL_FIELDS = ["patch_w", "patch_b", "t1_w", "t1_b", "t2_w", "t2_b", "m_w", "m_b", "hm_w", "hm_b", "head_w",
                  "head_b"]


class wan_block_weights(C.Structure):
    _fields_ = [(n, P) for n in _BLOCK_FIELDS]


class wan_dit_weights(C.Structure):
    _fields_ = [(n, P) for n in _GLOBAL_FIELDS] + [("blocks", C.POINTER(wan_block_weights))]


_SIGS = {
    "wan_status_string": (C.c_char_p, [I]),
    "wan_sync_status": (I, [P]),
    "wan_launch_count": (LL, []),
    "wan_watchdog_selftest": (I, [I, P]),
    "wan_patchify_workspace_size": (SZ, [I, I, I, I, I, I]),
    "wan_patchify": (I, [P, P, P, P, I, I, I, I, I, I, I, P, SZ, P]),
    "wan_adaln_modulate": (I, [P, P, P, P, I, I, I, F, I, P]),
    "wan_attn_workspace_size": (SZ, [I, I, I, I, I]),
    "wan_attn_rope3d": (I, [P, P, P, P, P, I, I, I, I, I, I, I, F, I, I, I, P, SZ, P]),
    "wan_qkv_rope_workspace_size": (SZ, [I]),
    "wan_qkv_rope": (I, [P, P, P, P, I, I, I, I, I, I, I, F, I, P, SZ, P]),
    "wan_qkv_rope_e4m3": (I, [P, P, P, P, P, P, I, I, I, I, I, I, I, F, P, SZ, P]),
    "wan_cross_attn_workspace_size": (SZ, [I, I, I, I, I, I]),
    "wan_cross_attn": (I, [P, P, P, P, P, P, P, I, I, I, I, I, I, I, I, P, SZ, P]),
    "wan_ffn": (I, [P, P, P, P, P, P, P, P, I, I, I, I, I, P]),
    "wan_linear": (I, [P, P, P, P, I, I, I, I, P, I, I, I, P]),
    "wan_text_embed_workspace_size": (SZ, [I, I, I, I]),
    "wan_text_embed": (I, [P, P, P, P, P, P, I, I, I, I, I, P, SZ, P]),
    "wan_text_embed_noalloc": (I, [P, P, P, P, P, P, I, I, I, I, I, P]),
    "wan_text_embed_noalloc_max_bytes": (SZ, []),
    "wan_cfg_euler_step": (I, [P, P, P, LL, F, F, I, P]),
    "wan_dit_workspace_size": (SZ, [C.POINTER(wan_dit_config)]),
    "wan_sample_workspace_size": (SZ, [C.POINTER(wan_dit_config)]),
    "wan_time_embed_workspace_size": (SZ, [C.POINTER(wan_dit_config)]),
    "wan_time_embed": (I, [C.POINTER(wan_dit_config), C.POINTER(wan_dit_weights), P, I, P, P, P, SZ, P]),
    "wan_dit_forward": (I, [C.POINTER(wan_dit_config), C.POINTER(wan_dit_weights), P, I, P, P, P, P, P, P, SZ,
                            P]),
    "wan_dit_guided_step": (I, [C.POINTER(wan_dit_config), C.POINTER(wan_dit_weights), P, P, F, P, P, P, P, P,
                                SZ, P]),
    "wan_sample": (I, [C.POINTER(wan_dit_config), C.POINTER(wan_dit_weights), P, I, F, P, P, P, P, P, P, SZ, P]),
    "wan_quant_rows_e4m3": (I, [P, I, LL, I, I, P, LL, P, P]),
    "wan_quant_attn_workspace_size": (SZ, [I, I, I]),
    "wan_quant_attn_e4m3": (I, [P, P, P, I, I, I, I, I, I, P, P, P, P, P, P, P, SZ, P]),
    "wan_attn_e4m3": (I, [P, P, P, P, P, P, P, P, I, I, I, I, P]),
    "wan_linear_e4m3": (I, [P, P, P, P, P, P, I, I, I, I, P, I, P]),
    "wan_profile_begin": (I, [I]),
    "wan_profile_end": (I, [C.POINTER(C.c_char_p), C.POINTER(C.c_double), C.POINTER(C.c_int), I]),
}
for _name, (_res, _args) in _SIGS.items():
    _fn = getattr(lib, _name)
    _fn.restype = _res
    _fn.argtypes = _args

EXPORTED = tuple(_SIGS)


def _p(x):
    """Device pointer of a CUDA tensor (None -> NULL; int passes through)."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if not x.is_cuda:
        raise ValueError("libwan takes device tensors")
    if not x.is_contiguous():
        raise ValueError("libwan takes contiguous tensors")
    return x.data_ptr()


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _nbytes(t):
    return 0 if t is None else t.numel() * t.element_size()


def _check(st, where):
    if st != WAN_OK:
        raise WanError(st, where)


def dtype_code(t: torch.dtype) -> int:
    if t == torch.float32:
        return WAN_F32
    if t == torch.float16:
        return WAN_F16
    if t == torch.bfloat16:
        return WAN_BF16
    raise ValueError(f"libwan has no storage type for {t}")


# ---------------------------------------------------------------- per-op entry points

def wan_sync_status(stream=None):
    _check(lib.wan_sync_status(_stream(stream)), "wan_sync_status")


def wan_launch_count() -> int:
    return lib.wan_launch_count()


def wan_watchdog_selftest(limit_ms=50, stream=None):
    _check(lib.wan_watchdog_selftest(limit_ms, _stream(stream)), "wan_watchdog_selftest")


def wan_patchify(latent, w, b, x, ws, stream=None):
    B, Cc, Fr, H, W = latent.shape
    D = w.shape[0]
    _check(lib.wan_patchify(_p(latent), _p(w), _p(b), _p(x), B, Cc, Fr, H, W, D, dtype_code(w.dtype), _p(ws),
                            ws.numel() * ws.element_size(), _stream(stream)), "wan_patchify")


def wan_patchify_workspace_size(B, Cc, Fr, H, W, dtype):
    return lib.wan_patchify_workspace_size(B, Cc, Fr, H, W, dtype)


def wan_adaln_modulate(x, shift, scale, y, eps=1e-6, stream=None):
    B, L, D = x.shape
    _check(lib.wan_adaln_modulate(_p(x), _p(shift), _p(scale), _p(y), B, L, D, eps, dtype_code(y.dtype),
                                  _stream(stream)), "wan_adaln_modulate")


def wan_attn_workspace_size(B, L, H, d, dtype):
    return lib.wan_attn_workspace_size(B, L, H, d, dtype)


def wan_attn_rope3d(q, k, v, o, grid, theta=10000.0, apply_rope=True, ws=None, kv_lens=None, stream=None):
    B, L, H, d = q.shape
    _check(lib.wan_attn_rope3d(_p(q), _p(k), _p(v), _p(o), _p(kv_lens), B, L, H, d, grid[0], grid[1], grid[2], theta,
                               1 if apply_rope else 0, dtype_code(v.dtype), dtype_code(q.dtype), _p(ws),
                               _nbytes(ws), _stream(stream)), "wan_attn_rope3d")


def wan_qkv_rope(y, w, b, qkv, heads, grid, theta=10000.0, ws=None, stream=None):
    """y [B, L, D] -> qkv [B, L, 3D] (q, k rotated; fp16 q|k next to bf16 v for bf16 y)."""
    B, L, D = y.shape
    d = D // heads
    if ws is None:
        ws = torch.empty(lib.wan_qkv_rope_workspace_size(d), dtype=torch.uint8, device=y.device)
    _check(lib.wan_qkv_rope(_p(y), _p(w), _p(b), _p(qkv), B, L, heads, d, grid[0], grid[1], grid[2], theta,
                            dtype_code(y.dtype), _p(ws), _nbytes(ws), _stream(stream)), "wan_qkv_rope")


def wan_qkv_rope_e4m3(y8, sy, w8, sw, b, qkv, heads, grid, theta=10000.0, ws=None, stream=None):
    """E4M3 rows y8 [B, L, D] (scales sy [B*L]) -> qkv [B, L, 3D] as wan_qkv_rope writes it."""
    B, L, D = y8.shape
    d = D // heads
    if ws is None:
        ws = torch.empty(lib.wan_qkv_rope_workspace_size(d), dtype=torch.uint8, device=y8.device)
    _check(lib.wan_qkv_rope_e4m3(_p(y8), _p(sy), _p(w8), _p(sw), _p(b), _p(qkv), B, L, heads, d, grid[0], grid[1],
                                 grid[2], theta, _p(ws), _nbytes(ws), _stream(stream)), "wan_qkv_rope_e4m3")


def wan_cross_attn_workspace_size(B, Lt, Li, H, d, dtype):
    return lib.wan_cross_attn_workspace_size(B, Lt, Li, H, d, dtype)


def wan_cross_attn(q, kt, vt, ki, vi, o, ws=None, kt_lens=None, stream=None):
    B, L, H, d = q.shape
    Lt = kt.shape[1]
    Li = ki.shape[1] if ki is not None else 0
    _check(lib.wan_cross_attn(_p(q), _p(kt), _p(vt), _p(kt_lens), _p(ki), _p(vi), _p(o), B, L, Lt, Li, H, d,
                              dtype_code(vt.dtype),
                              dtype_code(q.dtype), _p(ws), _nbytes(ws), _stream(stream)),
           "wan_cross_attn")


def wan_ffn(y, w1, b1, w2, b2, gate, x_inout, h_ws, stream=None):
    B, L, D = y.shape
    Fh = w1.shape[0]
    _check(lib.wan_ffn(_p(y), _p(w1), _p(b1), _p(w2), _p(b2), _p(gate), _p(x_inout), _p(h_ws), B, L, D, Fh,
                       dtype_code(y.dtype), _stream(stream)), "wan_ffn")


def wan_linear(x, w, b, out, epilogue=WAN_EPI_STORE, gate=None, rows_per_gate=0, stream=None):
    M, K = x.shape
    N = w.shape[0]
    _check(lib.wan_linear(_p(x), _p(w), _p(b), _p(out), M, N, K, epilogue, _p(gate), rows_per_gate,
                          dtype_code(x.dtype), dtype_code(out.dtype), _stream(stream)), "wan_linear")


def wan_quant_rows_e4m3(x, x8, s, stream=None):
    """x [M, K] (bf16 / fp16 / fp32) -> E4M3 codes x8 [M, K] (uint8) and row scales s [M]."""
    M, K = x.shape
    _check(lib.wan_quant_rows_e4m3(_p(x), dtype_code(x.dtype), x.stride(0), M, K, _p(x8), x8.stride(0), _p(s),
                                   _stream(stream)), "wan_quant_rows_e4m3")


def wan_quant_attn_workspace_size(B, H, d):
    return lib.wan_quant_attn_workspace_size(B, H, d)


def wan_quant_attn_e4m3(q, k, v, q8, sq, k8, sk, v8t, sv, ws, stream=None):
    """q, k, v [B, L, H, d] -> q8 [B, L, H, d], sq [B, L, H], k8, sk [B, H, nkb], v8t [B, H, d, Lp], sv [B, H, d]."""
    B, L, H, d = q.shape
    _check(lib.wan_quant_attn_e4m3(_p(q), _p(k), _p(v), dtype_code(q.dtype), dtype_code(v.dtype), B, L, H, d, _p(q8),
                                   _p(sq), _p(k8), _p(sk), _p(v8t), _p(sv), _p(ws), _nbytes(ws), _stream(stream)),
           "wan_quant_attn_e4m3")


def wan_attn_e4m3(q8, sq, k8, sk, v8t, sv, o, kv_lens=None, stream=None):
    B, L, H, d = q8.shape
    _check(lib.wan_attn_e4m3(_p(q8), _p(sq), _p(k8), _p(sk), _p(v8t), _p(sv), _p(o), _p(kv_lens), B, L, H, d,
                             _stream(stream)), "wan_attn_e4m3")


def wan_linear_e4m3(x8, sx, w8, sw, b, out, epilogue=WAN_EPI_STORE, gate=None, rows_per_gate=0, stream=None):
    M, K = x8.shape
    N = w8.shape[0]
    _check(lib.wan_linear_e4m3(_p(x8), _p(sx), _p(w8), _p(sw), _p(b), _p(out), M, N, K, epilogue, _p(gate),
                               rows_per_gate, _stream(stream)), "wan_linear_e4m3")


def wan_text_embed_workspace_size(B, Lt, D, dtype):
    return lib.wan_text_embed_workspace_size(B, Lt, D, dtype)


def wan_text_embed(text, w1, b1, w2, b2, ctx, ws, stream=None):
    B, Lt, Ct = text.shape
    D = w1.shape[0]
    _check(lib.wan_text_embed(_p(text), _p(w1), _p(b1), _p(w2), _p(b2), _p(ctx), B, Lt, Ct, D,
                              dtype_code(text.dtype), _p(ws), ws.numel() * ws.element_size(), _stream(stream)),
           "wan_text_embed")


def wan_text_embed_noalloc(text, w1, b1, w2, b2, ctx, stream=None):
    """wan_text_embed with libwan's static scratch: no allocation by libwan or here."""
    B, Lt, Ct = text.shape
    D = w1.shape[0]
    _check(lib.wan_text_embed_noalloc(_p(text), _p(w1), _p(b1), _p(w2), _p(b2), _p(ctx), B, Lt, Ct, D,
                                      dtype_code(text.dtype), _stream(stream)), "wan_text_embed_noalloc")


def wan_text_embed_noalloc_max_bytes() -> int:
    return lib.wan_text_embed_noalloc_max_bytes()


def wan_cfg_euler_step(x, v_cond, v_uncond, guide_scale, dt, stream=None):
    _check(lib.wan_cfg_euler_step(_p(x), _p(v_cond), _p(v_uncond), x.numel(), guide_scale, dt,
                                  dtype_code(v_cond.dtype), _stream(stream)), "wan_cfg_euler_step")


def wan_dit_workspace_size(cfg: wan_dit_config) -> int:
    return lib.wan_dit_workspace_size(C.byref(cfg))


def wan_sample_workspace_size(cfg: wan_dit_config) -> int:
    return lib.wan_sample_workspace_size(C.byref(cfg))


def wan_time_embed(cfg, weights, t, e0, hm, t_stride=1, stream=None):
    ws = torch.empty(lib.wan_time_embed_workspace_size(C.byref(cfg)) + 1024, dtype=torch.uint8, device=t.device)
    ws = ws[(-ws.data_ptr()) % 1024:]
    _check(lib.wan_time_embed(C.byref(cfg), C.byref(weights), _p(t), t_stride, _p(e0), _p(hm), _p(ws),
                              ws.numel(), _stream(stream)), "wan_time_embed")


def wan_dit_forward(cfg, weights, latent, t, ctx_txt, ctx_img, v_out, ws, latent_broadcast=False, txt_lens=None,
                    stream=None):
    _check(lib.wan_dit_forward(C.byref(cfg), C.byref(weights), _p(latent), 1 if latent_broadcast else 0, _p(t),
                               _p(ctx_txt), _p(txt_lens), _p(ctx_img), _p(v_out), _p(ws), _nbytes(ws),
                               _stream(stream)), "wan_dit_forward")


def wan_dit_guided_step(cfg, weights, x, t_pair, guide_scale, ctx_txt, ctx_img, v_ws, ws, txt_lens=None, stream=None):
    _check(lib.wan_dit_guided_step(C.byref(cfg), C.byref(weights), _p(x), _p(t_pair), guide_scale, _p(ctx_txt),
                                   _p(txt_lens), _p(ctx_img), _p(v_ws), _p(ws), _nbytes(ws), _stream(stream)),
           "wan_dit_guided_step")


def wan_sample(cfg, weights, x, steps, guide_scale, ctx_txt, ctx_img, t_sched, v_ws, ws, txt_lens=None, stream=None):
    _check(lib.wan_sample(C.byref(cfg), C.byref(weights), _p(x), steps, guide_scale, _p(ctx_txt), _p(txt_lens),
                          _p(ctx_img), _p(t_sched), _p(v_ws), _p(ws), _nbytes(ws), _stream(stream)),
           "wan_sample")


def wan_profile_begin(capacity=65536):
    _check(lib.wan_profile_begin(capacity), "wan_profile_begin")


def wan_profile_end(max_kinds=64):
    names = (C.c_char_p * max_kinds)()
    ms = (C.c_double * max_kinds)()
    counts = (C.c_int * max_kinds)()
    n = lib.wan_profile_end(names, ms, counts, max_kinds)
    if n < 0:
        raise WanError(n, "wan_profile_end")
    return {names[i].decode(): (ms[i], counts[i]) for i in range(n)}


# ---------------------------------------------------------------- model container

class DiT:
    """Device-resident weights of one DiT plus the config and pointer tables libwan takes.

    ``weights`` is a dict of float32 numpy arrays (already rounded to the storage type),
    e.g. from ``synth.make_weights``; it is uploaded once in the config's dtype.
    """

    def __init__(self, shape, weights: dict, device="cuda"):
        self.shape = shape
        self.tdtype = torch.float32 if shape.dtype == "f32" else torch.bfloat16
        self.cfg = wan_dit_config(
            dtype=WAN_F32 if shape.dtype == "f32" else WAN_BF16, batch=shape.batch, c_in=shape.c_in,
            c_out=shape.c_out, frames=shape.frames, height=shape.height, width=shape.width, dim=shape.dim,
            heads=shape.heads, head_dim=shape.head_dim, ffn=shape.ffn, blocks=shape.blocks,
            text_len=shape.text_len, img_len=shape.img_len, freq_dim=shape.freq_dim, theta=shape.theta,
            eps=shape.eps, qk_norm=int(getattr(shape, "qk_norm", False)),
            gelu_tanh=int(getattr(shape, "gelu_tanh", False)), fp8=int(getattr(shape, "fp8", 0)))
        up = lambda a, dt=self.tdtype: torch.from_numpy(np.ascontiguousarray(a)).to(device=device, dtype=dt)
        self.tensors = {k: up(v) for k, v in weights.items() if k != "blocks"}
        # In the 16-bit configuration the cross-attention query and output projections
        # are stored in fp16 (libwan runs that sub-layer in fp16, include/wan.h).
        f16 = {"cq_w", "co_w"} if self.tdtype == torch.bfloat16 else set()
        self.block_tensors = [{k: up(v, torch.float16 if k in f16 else self.tdtype) for k, v in blk.items()}
                              for blk in weights["blocks"]]
        if self.cfg.fp8 & 2:  # E4M3 codes + per-output-channel scales of the QKV and FFN-up weights
            for bt in self.block_tensors:
                for n in ("qkv_w", "f1_w"):
                    w = bt[n]
                    bt[n + "8"] = torch.empty(w.shape, dtype=torch.uint8, device=device)
                    bt[n[:-1] + "ws"] = torch.empty(w.shape[0], dtype=torch.float32, device=device)
                    wan_quant_rows_e4m3(w, bt[n + "8"], bt[n[:-1] + "ws"])
        self.blocks_c = (wan_block_weights * len(self.block_tensors))()
        for i, bt in enumerate(self.block_tensors):
            for n in _BLOCK_FIELDS:
                setattr(self.blocks_c[i], n, _p(bt.get(n)))
        self.weights_c = wan_dit_weights(**{n: _p(self.tensors[n]) for n in _GLOBAL_FIELDS})
        self.weights_c.blocks = C.cast(self.blocks_c, C.POINTER(wan_block_weights))
        self.ws = torch.empty(wan_dit_workspace_size(self.cfg) + 1024, dtype=torch.uint8, device=device)
        off = (-self.ws.data_ptr()) % 1024
        self.ws = self.ws[off:off + wan_dit_workspace_size(self.cfg)]
        if self.ws.numel() == 0:
            raise WanError(WAN_ERR_INVALID_ARG, "wan_dit_workspace_size")

    def text_embed(self, text, stream=None):
        B, Lt, _ = text.shape
        D = self.shape.dim
        ctx = torch.empty(B, Lt, D, dtype=self.tdtype, device=text.device)
        ws = torch.empty(wan_text_embed_workspace_size(B, Lt, D, self.cfg.dtype), dtype=torch.uint8,
                         device=text.device)
        t = self.tensors
        wan_text_embed(text, t["txt1_w"], t["txt1_b"], t["txt2_w"], t["txt2_b"], ctx, ws, stream)
        return ctx

    def time_embed(self, t, stream=None):
        s = self.shape
        e0 = torch.empty(s.batch, 6, s.dim, dtype=torch.float32, device=t.device)
        hm = torch.empty(s.batch, 2, s.dim, dtype=torch.float32, device=t.device)
        wan_time_embed(self.cfg, self.weights_c, t, e0, hm, 1 if t.numel() > 1 else 0, stream)
        return e0, hm

    def forward(self, latent, t, ctx_txt, ctx_img=None, latent_broadcast=False, v_out=None, txt_lens=None,
                stream=None):
        s = self.shape
        if v_out is None:
            v_out = torch.empty(s.batch, s.c_out, s.frames, s.height, s.width, dtype=torch.float32,
                                device=latent.device)
        wan_dit_forward(self.cfg, self.weights_c, latent, t, ctx_txt, ctx_img, v_out, self.ws, latent_broadcast,
                        txt_lens, stream)
        return v_out

    def guided_step(self, x, t_pair, guide_scale, ctx_txt, ctx_img=None, v_ws=None, txt_lens=None, stream=None):
        s = self.shape
        if v_ws is None:
            v_ws = torch.empty(2, s.c_out, s.frames, s.height, s.width, dtype=torch.float32, device=x.device)
        wan_dit_guided_step(self.cfg, self.weights_c, x, t_pair, guide_scale, ctx_txt, ctx_img, v_ws, self.ws,
                            txt_lens, stream)
        return v_ws

    def sample(self, x, steps, guide_scale, ctx_txt, ctx_img=None, txt_lens=None, stream=None):
        s = self.shape
        t_sched = torch.empty(steps + 1, dtype=torch.float32, device=x.device)
        v_ws = torch.empty(2, s.c_out, s.frames, s.height, s.width, dtype=torch.float32, device=x.device)
        n = wan_sample_workspace_size(self.cfg)
        ws = torch.empty(n + 1024, dtype=torch.uint8, device=x.device)
        off = (-ws.data_ptr()) % 1024
        wan_sample(self.cfg, self.weights_c, x, steps, guide_scale, ctx_txt, ctx_img, t_sched, v_ws, ws[off:off + n],
                   txt_lens, stream)
        return x

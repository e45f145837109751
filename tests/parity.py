"""Tolerances and conversions shared by the GPU parity tests.

bf16 configurations: max |g - o| <= 3e-2 * RMS(o) and sum|g - o| / sum|o| <= 5e-3.
fp32 configuration:  max_i |g_i - o_i| / max(|o_i|, RMS(o)) <= 1e-4 (relative error
floored at the RMS so near-zero elements do not dominate).
"""
import json
import os

import numpy as np

BF16_MAX_ABS_OVER_RMS = 3e-2
BF16_MEAN_REL = 5e-3
F32_MAX_REL = 1e-4


def to_dev(a, dtype, device="cuda"):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(device=device, dtype=dtype)


def to_np(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def bf16_errors(g, o):
    g = np.asarray(g, np.float64)
    o = np.asarray(o, np.float64)
    assert g.shape == o.shape, (g.shape, o.shape)
    assert np.all(np.isfinite(g)), "non-finite values in the GPU result"
    err = np.abs(g - o)
    rms = np.sqrt(np.mean(o ** 2))
    return float(err.max() / rms), float(err.sum() / np.abs(o).sum())


def _log(**rec):
    path = os.environ.get("WAN_PARITY_LOG")
    if path:
        with open(path, "a") as f:
            f.write(json.dumps(rec) + "\n")


def assert_bf16_close(g, o, what=""):
    mx, mr = bf16_errors(g, o)
    _log(what=what, kind="bf16", max_abs_over_rms=mx, mean_rel=mr, ok=bool(mx <= BF16_MAX_ABS_OVER_RMS and mr <= BF16_MEAN_REL))
    assert mx <= BF16_MAX_ABS_OVER_RMS and mr <= BF16_MEAN_REL, \
        f"{what}: max|err|/rms = {mx:.3e} (<= {BF16_MAX_ABS_OVER_RMS}), mean rel = {mr:.3e} (<= {BF16_MEAN_REL})"
    return mx, mr


def f32_error(g, o):
    g = np.asarray(g, np.float64)
    o = np.asarray(o, np.float64)
    assert g.shape == o.shape, (g.shape, o.shape)
    assert np.all(np.isfinite(g)), "non-finite values in the GPU result"
    rms = np.sqrt(np.mean(o ** 2))
    return float(np.max(np.abs(g - o) / np.maximum(np.abs(o), rms)))


def f32_error_unfloored(g, o):
    """max_i |g_i - o_i| / |o_i| over the elements with o_i != 0 (no RMS floor)."""
    g = np.asarray(g, np.float64)
    o = np.asarray(o, np.float64)
    nz = o != 0
    if not np.any(nz):
        return 0.0
    return float(np.max(np.abs(g[nz] - o[nz]) / np.abs(o[nz])))


def assert_f32_close(g, o, what="", tol=F32_MAX_REL):
    e = f32_error(g, o)
    _log(what=what, kind="f32", max_rel=e, max_rel_unfloored=f32_error_unfloored(g, o), tol=tol, ok=bool(e <= tol))
    assert e <= tol, f"{what}: max rel err {e:.3e} > {tol}"
    return e


def tokens_of(v):
    """[B, C, F, H, W] -> [B, L, C*4] in patch token order (layout only)."""
    B, C, F, H, W = v.shape
    t = v.reshape(B, C, F, H // 2, 2, W // 2, 2).transpose(0, 2, 3, 5, 1, 4, 6)
    return t.reshape(B, F * (H // 2) * (W // 2), C * 4)

"""CPU checks of the C ABI boundary: the library loads without a GPU, exports every
entry point include/wan.h declares, and its host-side validation and workspace
arithmetic behave as documented (no kernel is launched here)."""
import ctypes as C
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "wan.h")
LIB = os.path.join(ROOT, "video_diffusion_transformer_04_b300", "libwan.so")


def declared():
    txt = open(HEADER).read()
    txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
    return sorted(set(re.findall(r"\b(wan_[a-z0-9_]+)\s*\(", txt)))


@pytest.fixture(scope="module")
def wanlib():
    if not os.path.exists(LIB):
        from video_diffusion_transformer_04_b300 import _build
        _build.build()
    return C.CDLL(LIB)


def test_header_declares_the_seven_step_entry_points():
    names = declared()
    for n in ("wan_patchify", "wan_adaln_modulate", "wan_attn_rope3d", "wan_cross_attn", "wan_ffn",
              "wan_cfg_euler_step", "wan_dit_forward"):
        assert n in names


def test_library_exports_every_declared_symbol(wanlib):
    missing = [n for n in declared() if not hasattr(wanlib, n)]
    assert not missing, missing


def test_binding_covers_every_declared_symbol():
    from video_diffusion_transformer_04_b300 import wan
    assert sorted(wan.EXPORTED) == declared()


def test_library_has_no_driver_link_dependency():
    # The .so must load on a host without libcuda (the CPU suite runs without one).
    import subprocess
    out = subprocess.run(["ldd", LIB], capture_output=True, text=True).stdout
    assert "libcuda.so" not in out and "libcudart.so" not in out


def test_status_strings(wanlib):
    wanlib.wan_status_string.restype = C.c_char_p
    assert wanlib.wan_status_string(0) == b"ok"
    assert b"timed out" in wanlib.wan_status_string(-4)
    assert wanlib.wan_status_string(-99) == b"unknown status"


def test_host_validation_rejects_bad_arguments(wanlib):
    # Rejected before any CUDA call: NULL pointers, negative sizes, bad dtypes.
    f = wanlib.wan_cfg_euler_step
    f.argtypes = [C.c_void_p, C.c_void_p, C.c_void_p, C.c_longlong, C.c_float, C.c_float, C.c_int, C.c_void_p]
    assert f(None, None, None, 0, 5.0, -0.05, 0, None) == 0          # n == 0 is a no-op
    assert f(None, None, None, 16, 5.0, -0.05, 0, None) == -1       # NULL pointers
    assert f(None, None, None, -1, 5.0, -0.05, 0, None) == -1       # negative n
    assert f(None, None, None, 16, 5.0, -0.05, 7, None) == -1       # unknown dtype
    g = wanlib.wan_linear
    g.argtypes = [C.c_void_p] * 4 + [C.c_int] * 4 + [C.c_void_p, C.c_int, C.c_int, C.c_int, C.c_void_p]
    assert g(None, None, None, None, 8, 64, 64, 0, None, 0, 0, 0, None) == -1
    assert g(None, None, None, None, 8, 64, 64, 9, None, 0, 0, 0, None) == -1
    # fp16 storage is an output type of the bf16 GEMM only, and never the residual's type
    assert g(1 << 12, 1 << 12, None, 1 << 12, 8, 64, 64, 0, None, 0, 1, 2, None) == -2
    assert g(1 << 12, 1 << 12, None, 1 << 12, 8, 64, 64, 2, None, 0, 0, 2, None) == -2
    h = wanlib.wan_cross_attn
    h.argtypes = [C.c_void_p] * 7 + [C.c_int] * 8 + [C.c_void_p, C.c_size_t, C.c_void_p]
    # q/k in fp16 are accepted only next to bf16 v/o; unknown codes are invalid
    assert h(None, None, None, None, None, None, None, 1, 8, 8, 0, 1, 64, 1, 2, None, 0, None) == -2
    assert h(None, None, None, None, None, None, None, 1, 8, 8, 0, 1, 64, 0, 5, None, 0, None) == -1
    assert h(None, None, None, None, None, None, None, 1, 8, 8, 0, 1, 64, 0, 2, None, 0, None) == -1  # NULL q


def test_host_validation_of_the_fp16_and_qkv_rope_entry_points(wanlib):
    P, I, F, SZ = C.c_void_p, C.c_int, C.c_float, C.c_size_t
    A = 1 << 12
    h = wanlib.wan_cross_attn
    h.argtypes = [C.c_void_p] * 7 + [C.c_int] * 8 + [C.c_void_p, C.c_size_t, C.c_void_p]
    # fp16 v/o (the forward's cross-attention) need fp16 q/k
    assert h(A, A, A, None, None, None, A, 1, 8, 8, 0, 1, 64, 2, 0, None, 0, None) == -2
    assert h(None, A, A, None, None, None, A, 1, 8, 8, 0, 1, 64, 2, 2, None, 0, None) == -1
    g = wanlib.wan_linear
    g.argtypes = [C.c_void_p] * 4 + [C.c_int] * 4 + [C.c_void_p, C.c_int, C.c_int, C.c_int, C.c_void_p]
    assert g(None, A, None, A, 8, 64, 64, 0, None, 0, 2, 2, None) == -1   # fp16 operands: NULL x
    assert g(A, A, None, A, 8, 48, 64, 0, None, 0, 2, 2, None) == -2      # N % 32
    r = wanlib.wan_qkv_rope
    r.argtypes = [P] * 4 + [I] * 7 + [F, I, P, SZ, P]
    assert wanlib.wan_qkv_rope_workspace_size(128) >= 64 * 4
    ok = [A, A, A, A, 1, 60, 2, 128, 3, 4, 5, 10000.0, 0]
    assert r(None, *ok[1:], A, 1024, None) == -1                      # NULL y
    assert r(*ok[:8], 3, 4, 6, 10000.0, 0, A, 1024, None) == -1       # grid does not cover L
    assert r(*ok, None, 0, None) == -5                                # no workspace
    assert r(*ok[:12], 7, A, 1024, None) == -1                        # unknown dtype
    r8 = wanlib.wan_qkv_rope_e4m3
    r8.argtypes = [P] * 6 + [I] * 7 + [F, P, SZ, P]
    args8 = [A, A, A, A, A, A, 1, 60, 2, 128, 3, 4, 5, 10000.0]
    assert r8(A, None, *args8[2:], A, 1024, None) == -1               # missing row scales
    assert r8(*args8, A, 8, None) == -5                               # workspace too small


def test_dit_workspace_size_arithmetic():
    import synth
    from video_diffusion_transformer_04_b300 import wan
    s = synth.STEP_1P3B
    cfg = wan.wan_dit_config(dtype=wan.WAN_BF16, batch=2, c_in=16, c_out=16, frames=21, height=60, width=104,
                             dim=1536, heads=12, head_dim=128, ffn=8960, blocks=30, text_len=512, img_len=0,
                             freq_dim=256, theta=10000.0, eps=1e-6)
    n = wan.wan_dit_workspace_size(cfg)
    M, D = 2 * s.tokens, s.dim
    # at least x (fp32), y, q|k, v^T, o, cross q and the FFN hidden (bf16)
    lower = M * D * 4 + M * D * 2 * 5 + M * s.ffn * 2
    assert lower <= n <= lower * 1.2
    bad = wan.wan_dit_config(**{f: getattr(cfg, f) for f, _ in cfg._fields_})
    bad.heads = 7
    assert wan.wan_dit_workspace_size(bad) == 0
    bad = wan.wan_dit_config(**{f: getattr(cfg, f) for f, _ in cfg._fields_})
    bad.head_dim, bad.heads = 96, 16
    assert wan.wan_dit_workspace_size(bad) == 0       # bf16 attention takes d = 64 or 128


def test_host_validation_of_the_8bit_entry_points(wanlib):
    P, I, LL, SZ = C.c_void_p, C.c_int, C.c_longlong, C.c_size_t
    A = 1 << 12  # a 16-byte-aligned dummy address: only reached by the host checks
    q = wanlib.wan_quant_rows_e4m3
    q.argtypes = [P, I, LL, I, I, P, LL, P, P]
    assert q(None, 0, 64, 8, 64, A, 64, A, None) == -1           # NULL x
    assert q(A, 7, 64, 8, 64, A, 64, A, None) == -1              # unknown dtype
    assert q(A, 0, 64, 8, 62, A, 64, A, None) == -2              # K % 4
    qa = wanlib.wan_quant_attn_e4m3
    qa.argtypes = [P, P, P, I, I, I, I, I, I, P, P, P, P, P, P, P, SZ, P]
    args = [A, A, A, 2, 0, 1, 300, 2, 128, A, A, A, A, A, A]
    assert qa(*args, A, 1 << 20, None) != -1                      # well-formed (fails later, no GPU)
    assert qa(None, *args[1:], A, 1 << 20, None) == -1           # NULL q
    assert qa(*args[:3], 1, *args[4:], A, 1 << 20, None) == -1   # fp32 q/k are not a quantiser input
    assert qa(*args[:8], 64, *args[9:], A, 1 << 20, None) == -2  # d must be 128
    assert qa(*args, None, 0, None) == -5                        # no workspace
    assert qa(*args, A, 16, None) == -5                          # too small (needs B*H*d*4)
    at = wanlib.wan_attn_e4m3
    at.argtypes = [P] * 8 + [I] * 4 + [P]
    assert at(None, A, A, A, A, A, A, None, 1, 300, 2, 128, None) == -1
    assert at(A, A, A, A, A, A, A, None, 1, 300, 2, 64, None) == -2
    li = wanlib.wan_linear_e4m3
    li.argtypes = [P] * 6 + [I] * 4 + [P, I, P]
    assert li(None, A, A, A, None, A, 8, 64, 64, 0, None, 0, None) == -1
    assert li(A, A, A, A, None, A, 8, 64, 64, 9, None, 0, None) == -1   # unknown epilogue
    assert li(A, A, A, A, None, A, 8, 48, 64, 0, None, 0, None) == -2   # N % 32
    assert li(A, A, A, A, None, A, 8, 64, 56, 0, None, 0, None) == -2   # K % 16


def test_dit_workspace_size_of_the_8bit_variant():
    from video_diffusion_transformer_04_b300 import wan
    base = dict(dtype=wan.WAN_BF16, batch=2, c_in=16, c_out=16, frames=21, height=60, width=104, dim=1536,
                heads=12, head_dim=128, ffn=8960, blocks=30, text_len=512, img_len=0, freq_dim=256,
                theta=10000.0, eps=1e-6)
    n0 = wan.wan_dit_workspace_size(wan.wan_dit_config(**base))
    n3 = wan.wan_dit_workspace_size(wan.wan_dit_config(**base, fp8=3))
    M, D, H, d, L = 2 * 32760, 1536, 12, 128, 32760
    # y8 + sy, q8 + k8, v8t (+ scales): at least 4 M*D bytes more
    assert n3 - n0 >= 4 * M * D and n3 - n0 <= 4 * M * D + 16 * M * H + (1 << 20)
    assert wan.wan_dit_workspace_size(wan.wan_dit_config(**base, fp8=4)) == 0
    assert wan.wan_dit_workspace_size(wan.wan_dit_config(**dict(base, dtype=wan.WAN_F32), fp8=1)) == 0
    assert wan.wan_dit_workspace_size(wan.wan_dit_config(**dict(base, heads=24, head_dim=64), fp8=1)) == 0

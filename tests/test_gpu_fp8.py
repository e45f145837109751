"""GPU parity of the 8-bit variant (FP8 GEMMs + 8-bit self-attention) against the CPU oracle.

* Quantisers: E4M3 codes and scales bit for bit (both sides decide in fp32 on the same
  input values).
* 8-bit attention, fed the oracle's codes: the oracle computes softmax and products in
  fp64 on the dequantised operands; the kernel also rounds each probability to E4M3, so
  the test bound per output element is
      2^-4 * sum_j p_j |V_j| / sum_j p_j           (normal-range rounding of P)
    + 2^-18 * sum_{p_j < 2^-14} |V_j| / sum_j p_j  (probabilities in the subnormal range:
                                                     P' = 2^8 p >= 2^8 p_true)
    + 2^-8 |o|                                      (bf16 output rounding)
  with p_j the exact probabilities relative to the row max.
* FP8 GEMM, fed the oracle's codes: every product of two codes is exact, the sum is fp32,
  so the bf16 tolerances of the other GEMMs apply (fp32 tolerance for the residual form).
* The forward with the variant on, against the oracle's 8-bit forward, within the plain
  bf16 tolerances: the tiny configuration and the full 1.3B block.  At the full 1.3B
  block, where quantisation moves the result well beyond bf16 rounding, the GPU result
  must also lie closer to the 8-bit oracle than to the exact one: it computes the 8-bit
  method, not the bf16 one.  (At the tiny size the quantisation error is below the bf16
  rounding, so that comparison says nothing there.)  The 14B I2V block, where each side's
  own quantisation decisions on its own activations differ in a few percent of the codes,
  is checked in tests/test_gpu_block_fp8.py with the oracle fed the GPU's codes.
"""
import os

import numpy as np
import pytest
import torch

import synth
from oracle import wan_oracle as O
from tests.parity import _log, assert_bf16_close, assert_f32_close, to_dev, to_np, tokens_of

pytestmark = pytest.mark.gpu
BF, F16, F32, U8 = torch.bfloat16, torch.float16, torch.float32, torch.uint8
TD = {"bf16": BF, "f16": F16, "f32": F32}
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _round_to(a, dt):
    a = np.asarray(a, np.float64)
    if dt == "bf16":
        return synth.round_bf16(a)
    if dt == "f16":
        return a.astype(np.float16).astype(np.float64)
    return a.astype(np.float32).astype(np.float64)


def _u8(t):
    return t.cpu().numpy()


def _rel_rms(a, b):
    a, b = np.asarray(a, np.float64), np.asarray(b, np.float64)
    return float(np.sqrt(np.mean((a - b) ** 2) / np.mean(b ** 2)))


# ---------------------------------------------------------------- quantisers

@pytest.mark.parametrize("dt", ["bf16", "f16", "f32"])
def test_quant_rows_bit_exact(wan, dt):
    M, K = 37, 1540
    x = synth.normal(30, "q8.x", (M, K)) * np.exp(3.0 * synth.normal(30, "q8.s", (M, 1)))
    x[5] = 0.0
    x = _round_to(x, dt)
    x8 = torch.full((M, K), 0xFF, dtype=U8, device="cuda")
    s = torch.full((M,), float("nan"), dtype=F32, device="cuda")
    wan.wan_quant_rows_e4m3(to_dev(x, TD[dt]), x8, s)
    wan.wan_sync_status()
    codes, sc = O.quant_rows(x)
    assert np.array_equal(_u8(x8), codes)
    assert np.array_equal(s.cpu().numpy(), sc)


def _attn_inputs(seed, B, L, H, d, qkt):
    # Per-(token, head) and per-channel magnitudes spread over a few octaves.
    q = synth.normal(seed, "a8.q", (B, L, H, d)) * np.exp(0.5 * synth.normal(seed, "a8.qs", (B, L, H, 1)))
    k = synth.normal(seed, "a8.k", (B, L, H, d)) * np.exp(0.5 * synth.normal(seed, "a8.ks", (B, L, H, 1)))
    v = synth.normal(seed, "a8.v", (B, L, H, d)) * np.exp(synth.normal(seed, "a8.vs", (1, 1, H, d)))
    return _round_to(q, qkt), _round_to(k, qkt), _round_to(v, "bf16")


def _quant_gpu(wan, q, k, v, qkt):
    B, L, H, d = q.shape
    nkb, Lp = (L + 127) // 128, (L + 15) // 16 * 16
    dev = lambda shape, dt, fill: torch.full(shape, fill, dtype=dt, device="cuda")
    out = dict(q8=dev((B, L, H, d), U8, 0xFF), sq=dev((B, L, H), F32, float("nan")),
               k8=dev((B, L, H, d), U8, 0xFF), sk=dev((B, H, nkb), F32, float("nan")),
               v8t=dev((B, H, d, Lp), U8, 0xFF), sv=dev((B, H, d), F32, float("nan")))
    ws = torch.empty(wan.wan_quant_attn_workspace_size(B, H, d), dtype=U8, device="cuda")
    wan.wan_quant_attn_e4m3(to_dev(q, TD[qkt]), to_dev(k, TD[qkt]), to_dev(v, BF), out["q8"], out["sq"], out["k8"],
                            out["sk"], out["v8t"], out["sv"], ws)
    return out


@pytest.mark.parametrize("qkt", ["bf16", "f16"])
@pytest.mark.parametrize("L", [300, 128, 1])
def test_quant_attn_operands_bit_exact(wan, qkt, L):
    B, H, d = 2, 3, 128
    q, k, v = _attn_inputs(31, B, L, H, d, qkt)
    g = _quant_gpu(wan, q, k, v, qkt)
    wan.wan_sync_status()
    for b in range(B):
        q8, sq = O.quant_attn_q(q[b])
        k8, sk = O.quant_attn_k(k[b])
        v8, sv = O.quant_attn_v(v[b])
        assert np.array_equal(_u8(g["q8"][b]), q8) and np.array_equal(g["sq"][b].cpu().numpy(), sq)
        assert np.array_equal(_u8(g["k8"][b]), k8) and np.array_equal(g["sk"][b].cpu().numpy(), sk)
        v8t = _u8(g["v8t"][b])
        assert np.array_equal(v8t[:, :, :L], v8.transpose(1, 2, 0))
        assert np.all(v8t[:, :, L:] == 0)  # pad keys up to the 16-key row stride
        assert np.array_equal(g["sv"][b].cpu().numpy(), sv)


# ---------------------------------------------------------------- 8-bit attention

def _oracle_codes(q, k, v):
    """Per batch entry: the oracle's codes and scales in the ABI layouts."""
    B, L, H, d = q.shape
    Lp = (L + 15) // 16 * 16
    q8 = np.empty(q.shape, np.uint8); k8 = np.empty(k.shape, np.uint8)
    sq = np.empty((B, L, H), np.float32); sk = np.empty((B, H, (L + 127) // 128), np.float32)
    v8t = np.zeros((B, H, d, Lp), np.uint8); sv = np.empty((B, H, d), np.float32)
    for b in range(B):
        q8[b], sq[b] = O.quant_attn_q(q[b])
        k8[b], sk[b] = O.quant_attn_k(k[b])
        vc, sv[b] = O.quant_attn_v(v[b])
        v8t[b, :, :, :L] = vc.transpose(1, 2, 0)
    return q8, sq, k8, sk, v8t, sv


def _bound_8bit(Qd, Kd, Vd, ref):
    """Per-element bound of the kernel's E4M3 probability rounding (module docstring)."""
    L, H, d = Qd.shape
    bound = np.empty_like(ref)
    for h in range(H):
        s = Qd[:, h] @ Kd[:, h].T / np.sqrt(d)
        p = np.exp(s - s.max(axis=1, keepdims=True))
        l = p.sum(axis=1, keepdims=True)
        av = np.abs(Vd[:, h])
        bound[:, h] = (2.0 ** -4 * (p @ av) + 2.0 ** -18 * ((p < 2.0 ** -14) @ av)) / l
    return bound + 2.0 ** -8 * np.abs(ref) + 1e-7 * np.abs(Vd).max()


def _check_8bit(o_gpu, q8, sq, k8, sk, v8, sv, kv_len, what):
    ref = O.attention_8bit(q8, sq, k8, sk, v8, sv, kv_len=kv_len)
    blk = np.arange(k8.shape[0]) // 128
    Qd = O.dequant(q8, sq[..., None])
    Kd = O.e4m3_decode(k8) * np.asarray(sk, np.float64).T[blk][:, :, None]
    Vd = O.e4m3_decode(v8) * np.asarray(sv, np.float64)[None]
    n = kv_len or k8.shape[0]
    bound = _bound_8bit(Qd, Kd[:n], Vd[:n], ref)
    err = np.abs(o_gpu - ref)
    assert np.all(np.isfinite(o_gpu)), what
    worst = float((err / bound).max())
    _log(what=what, kind="attn8_bound", max_err_over_bound=worst,
         max_abs_over_rms=float(err.max() / np.sqrt(np.mean(ref ** 2))), ok=bool(worst <= 1.0))
    assert worst <= 1.0, f"{what}: max err / bound = {worst:.3f}"
    return worst


@pytest.mark.parametrize("B,L,H,lens,growth", [
    (1, 300, 2, None, False),      # ragged last key tile, two query tiles per CTA
    (2, 1000, 2, [1000, 517], False),  # k_lens
    (1, 4 * 128 + 37, 2, None, True),  # keys grow tile by tile: the lazy reference max moves
    (1, 128, 1, None, False),
    (1, 1, 1, None, False),
])
def test_attn_e4m3_vs_oracle(wan, B, L, H, lens, growth):
    d = 128
    q, k, v = _attn_inputs(32, B, L, H, d, "f16")
    if growth:
        k = _round_to(k * (0.2 + 1.2 * (np.arange(L) // 128))[None, :, None, None], "f16")
    q8, sq, k8, sk, v8t, sv = _oracle_codes(q, k, v)
    o = torch.full((B, L, H, d), float("nan"), dtype=BF, device="cuda")
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    kv = dev(np.array(lens, np.int32)) if lens else None
    wan.wan_attn_e4m3(dev(q8), dev(sq), dev(k8), dev(sk), dev(v8t), dev(sv), o, kv_lens=kv)
    wan.wan_sync_status()
    og = to_np(o)
    for b in range(B):
        n = lens[b] if lens else None
        _check_8bit(og[b], q8[b], sq[b], k8[b], sk[b], v8t[b].transpose(2, 0, 1)[:L], sv[b], n, f"attn8 b={b}")
    if growth:  # the rescale path ran: later tiles' row max far above the first tile's
        logits = np.einsum("lhd,mhd->hlm", q[0], k[0]) / np.sqrt(d)
        assert np.mean(logits.max(axis=2) - logits[:, :, :128].max(axis=2) > 1.0) > 0.5


def test_attn_8bit_full_size_sampled_rows(wan):
    # The 1.3B self-attention shape (32760 tokens, 12 heads of 128) through the composed
    # GPU path (quantisers + 8-bit attention); the oracle quantises the same values
    # itself and evaluates sampled query rows against every key.
    B, L, H, d = 1, 32760, 12, 128
    q, k, v = _attn_inputs(33, B, L, H, d, "f16")
    g = _quant_gpu(wan, q, k, v, "f16")
    o = torch.full((B, L, H, d), float("nan"), dtype=BF, device="cuda")
    wan.wan_attn_e4m3(g["q8"], g["sq"], g["k8"], g["sk"], g["v8t"], g["sv"], o)
    wan.wan_sync_status()
    rows = synth.sample_rows(L, 128, 33)
    q8, sq = O.quant_attn_q(q[0, rows])
    k8, sk = O.quant_attn_k(k[0])
    v8, sv = O.quant_attn_v(v[0])
    _check_8bit(to_np(o[0, rows]), q8, sq, k8, sk, v8, sv, None, "attn8 full size")


# ---------------------------------------------------------------- FP8 GEMM

@pytest.mark.parametrize("M,N,K", [(300, 384, 1536), (257, 256, 1552), (64, 96, 64)])
@pytest.mark.parametrize("epi", ["store", "gelu", "residual"])
def test_linear_e4m3_vs_oracle(wan, M, N, K, epi):
    a = synth.round_bf16(synth.normal(34, "l8.a", (M, K)) * np.exp(synth.normal(34, "l8.as", (M, 1))))
    w = synth.round_bf16(synth.normal(34, "l8.w", (N, K), std=K ** -0.5))
    b = synth.round_bf16(synth.normal(34, "l8.b", (N,), std=0.1))
    a8, sa = O.quant_rows(a)
    w8, sw = O.quant_rows(w)
    y = O.linear_fp8(a8, sa, w8, sw, b)
    dev = lambda x: torch.from_numpy(np.ascontiguousarray(x)).cuda()
    if epi == "residual":
        x0 = synth.normal(34, "l8.x0", (M, N))
        gate = synth.normal(34, "l8.g", (1, N))
        out = to_dev(x0, F32)
        wan.wan_linear_e4m3(dev(a8), dev(sa), dev(w8), dev(sw), to_dev(b, BF), out, wan.WAN_EPI_RESIDUAL,
                            gate=to_dev(gate, F32), rows_per_gate=M)
        wan.wan_sync_status()
        assert_f32_close(to_np(out), x0 + gate * y, f"fp8 linear residual {M}x{N}x{K}")
    else:
        out = torch.full((M, N), float("nan"), dtype=BF, device="cuda")
        kind = wan.WAN_EPI_GELU if epi == "gelu" else wan.WAN_EPI_STORE
        wan.wan_linear_e4m3(dev(a8), dev(sa), dev(w8), dev(sw), to_dev(b, BF), out, kind)
        wan.wan_sync_status()
        ref = O.gelu(y) if epi == "gelu" else y
        # rows span e^N(0,1) magnitudes: compare each row relative to its own RMS
        r = np.sqrt(np.mean(ref ** 2, axis=1, keepdims=True))
        assert_bf16_close(to_np(out) / r, ref / r, f"fp8 linear {epi} {M}x{N}x{K}")


# ---------------------------------------------------------------- forward with the variant

@pytest.mark.parametrize("bits", [1, 2, 3])
def test_tiny_forward_fp8_variant(wan, bits):
    s = synth.TINY.replace(dtype="bf16", dim=384, heads=3, head_dim=128, fp8=bits)
    w = synth.make_weights(s, 0)
    inp = synth.make_inputs(s, 0)
    m = wan.DiT(s, w)
    ctx = m.text_embed(to_dev(inp["text"], BF))
    lat = np.concatenate([inp["latent"], 0.5 * inp["latent"]], axis=0)
    t = np.array([0.3, 0.8], np.float32)
    v = m.forward(to_dev(lat, F32), to_dev(t, F32), ctx)
    wan.wan_sync_status()
    g = to_np(v)
    ctx_o = O.text_projection(inp["text"], w)
    o8 = O.dit_forward(lat, t, ctx_o, None, w, s)
    ex = O.dit_forward(lat, t, ctx_o, None, w, s.replace(fp8=0))
    e_gpu, e_q, e_exact = _rel_rms(g, o8), _rel_rms(o8, ex), _rel_rms(g, ex)
    _log(what=f"tiny fp8={bits}", kind="fp8_forward", gpu_vs_oracle8=e_gpu, oracle8_vs_exact=e_q, gpu_vs_exact=e_exact,
         ok=bool(e_gpu < e_exact))
    assert_bf16_close(g, o8, f"tiny forward fp8={bits}")
    # the GPU computes the 8-bit variant, not the exact forward: it lies closer to the
    # 8-bit oracle than to the exact one
    assert e_gpu < e_exact, f"|gpu - oracle8| {e_gpu:.3e}, |oracle8 - exact| {e_q:.3e}, |gpu - exact| {e_exact:.3e}"


@pytest.mark.parametrize("name", ["wan1.3b-block"])
def test_single_block_fp8_variant(wan, name):
    path8 = os.path.join(GOLDEN, f"{name}-fp8.npz")
    path = os.path.join(GOLDEN, f"{name}.npz")
    if not (os.path.exists(path8) and os.path.exists(path)):
        pytest.skip("golden not generated")
    g8, gx = np.load(path8), np.load(path)
    s = synth.WORKLOADS[name].replace(fp8=int(g8["fp8"]))
    w = synth.make_weights(s, 0)
    inp = synth.make_inputs(s, 0)
    m = wan.DiT(s, w)
    del w
    ctx = m.text_embed(to_dev(inp["text"], BF)) if s.text_dim else to_dev(inp["ctx_txt"], BF)
    ctx_img = to_dev(inp["ctx_img"], BF) if s.img_len else None
    v = m.forward(to_dev(inp["latent"], F32), to_dev(inp["t"], F32), ctx, ctx_img)
    wan.wan_sync_status()
    head = tokens_of(to_np(v))[0, g8["rows"]]
    assert np.array_equal(g8["rows"], gx["rows"])
    e_gpu, e_q = _rel_rms(head, g8["head"]), _rel_rms(g8["head"], gx["head"])
    e_exact = _rel_rms(head, gx["head"])
    _log(what=f"{name} fp8", kind="fp8_forward", gpu_vs_oracle8=e_gpu, oracle8_vs_exact=e_q, gpu_vs_exact=e_exact,
         ok=bool(e_gpu <= e_q and e_gpu < 0.5 * e_exact))
    assert_bf16_close(head, g8["head"], f"{name} fp8 head rows")
    assert e_gpu <= e_q and e_gpu < 0.5 * e_exact, \
        f"|gpu - oracle8| {e_gpu:.3e}, |oracle8 - exact| {e_q:.3e}, |gpu - exact| {e_exact:.3e}"

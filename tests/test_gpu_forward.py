"""GPU parity of the whole DiT forward, guided step and sampler against the CPU fp64
oracle on the benchmark workloads' seeded synthetic inputs.

* the tiny configuration (fp32 and bf16) is compared element by element with the
  oracle run live;
* the full-size configurations are compared at the positions stored by
  tests/golden/make_goldens.py (oracle output only).
"""
import os

import numpy as np
import pytest
import torch

import synth
from oracle import wan_oracle as O
from tests.parity import assert_bf16_close, assert_f32_close, to_dev, to_np, tokens_of

pytestmark = pytest.mark.gpu
BF, F32 = torch.bfloat16, torch.float32
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _model(wan, s, seed=0):
    w = synth.make_weights(s, seed)
    inp = synth.make_inputs(s, seed)
    return w, inp, wan.DiT(s, w)


def _golden(name):
    path = os.path.join(GOLDEN, f"{name}.npz")
    if not os.path.exists(path):
        pytest.skip(f"{path} not generated")
    return np.load(path)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_tiny_guided_step(wan, dtype):
    s = synth.TINY.replace(dtype=dtype)
    w, inp, m = _model(wan, s)
    tdt = m.tdtype
    ctx = m.text_embed(to_dev(inp["text"], tdt))
    x = to_dev(inp["latent"], F32)
    t = float(inp["t"][0])
    t_pair = torch.tensor([t, t + s.dt], dtype=F32, device="cuda")
    v = m.guided_step(x, t_pair, s.guide_scale, ctx)
    wan.wan_sync_status()
    ctx_o = O.text_projection(inp["text"], w)
    lat2 = np.concatenate([inp["latent"]] * 2, axis=0)
    v_o = O.dit_forward(lat2, np.array([t, t]), ctx_o, None, w, s)
    dt = float(np.float32(t + s.dt)) - float(np.float32(t))
    x_o = O.cfg_euler_step(inp["latent"], v_o[0:1], v_o[1:2], s.guide_scale, dt)
    if dtype == "f32":
        assert_f32_close(to_np(ctx), ctx_o, "ctx")
        assert_f32_close(to_np(v), v_o, "v")
        assert_f32_close(to_np(x), x_o, "x_next")
    else:
        assert_bf16_close(to_np(ctx), ctx_o, "ctx")
        assert_bf16_close(to_np(v), v_o, "v")
        assert_bf16_close(to_np(x), x_o, "x_next")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("dims", [(128, 2, 64), (384, 3, 128)])
def test_tiny_forward_qk_norm_gelu_tanh_variant(wan, dtype, dims):
    # The checkpoint-fidelity variant: RMSNorm on q and k before RoPE, tanh-form GELU.
    D, H, hd = dims
    s = synth.TINY.replace(dtype=dtype, dim=D, heads=H, head_dim=hd, qk_norm=True, gelu_tanh=True)
    w, inp, m = _model(wan, s)
    ctx = m.text_embed(to_dev(inp["text"], m.tdtype))
    lat = np.concatenate([inp["latent"], 0.5 * inp["latent"]], axis=0)
    t = np.array([0.3, 0.8], np.float32)
    v = m.forward(to_dev(lat, F32), to_dev(t, F32), ctx)
    wan.wan_sync_status()
    v_o = O.dit_forward(lat, t, O.text_projection(inp["text"], w), None, w, s)
    if dtype == "f32":
        assert_f32_close(to_np(v), v_o, "v (qk_norm, gelu_tanh)")
    else:
        assert_bf16_close(to_np(v), v_o, "v (qk_norm, gelu_tanh)")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_tiny_forward_padded_text(wan, dtype):
    # Padded text contexts with per-entry valid lengths (k_lens of the cross-attention):
    # the result must equal the oracle run on each entry's unpadded context.
    s = synth.TINY.replace(dtype=dtype)
    w, inp, m = _model(wan, s)
    tdt = m.tdtype
    ctx = m.text_embed(to_dev(inp["text"], tdt))
    lens = np.array([5, 16], np.int32)
    lat = np.concatenate([inp["latent"], 0.5 * inp["latent"]], axis=0)
    t = np.array([0.3, 0.8], np.float32)
    v = m.forward(to_dev(lat, F32), to_dev(t, F32), ctx, txt_lens=torch.from_numpy(lens).cuda())
    wan.wan_sync_status()
    ctx_o = O.text_projection(inp["text"], w)
    v_o = O.dit_forward(lat, t, [ctx_o[b, :lens[b]] for b in range(2)], None, w, s)
    if dtype == "f32":
        assert_f32_close(to_np(v), v_o, "v with padded text")
    else:
        assert_bf16_close(to_np(v), v_o, "v with padded text")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_sampler_context_cache_is_exact(wan, dtype):
    # wan_sample projects the cross-attention keys/values once and reuses them; stepping
    # by hand with wan_dit_guided_step projects them at every step.  Same arithmetic on
    # the same operands: the results must agree bit for bit.
    s = synth.TINY.replace(dtype=dtype)
    w, inp, m = _model(wan, s)
    ctx = m.text_embed(to_dev(inp["text"], m.tdtype))
    steps = 3
    x_a = to_dev(inp["latent"], F32)
    m.sample(x_a, steps, s.guide_scale, ctx)
    x_b = to_dev(inp["latent"], F32)
    ts = torch.tensor(1.0 - np.arange(steps + 1, dtype=np.float32) / steps, device="cuda")
    for k in range(steps):
        m.guided_step(x_b, ts[k:k + 2].contiguous(), s.guide_scale, ctx)
    wan.wan_sync_status()
    assert torch.equal(x_a, x_b)


def test_tiny_forward_batch_permutation(wan):
    # Permuting the batch (latents, timesteps, contexts) permutes the outputs.
    s = synth.TINY
    w, inp, m = _model(wan, s)
    ctx = m.text_embed(to_dev(inp["text"], F32))
    lat = torch.cat([to_dev(inp["latent"], F32), 0.5 * to_dev(inp["latent"], F32)])
    t = torch.tensor([0.3, 0.8], dtype=F32, device="cuda")
    v1 = m.forward(lat, t, ctx).clone()
    v2 = m.forward(lat.flip(0).contiguous(), t.flip(0).contiguous(), ctx.flip(0).contiguous())
    wan.wan_sync_status()
    assert_f32_close(to_np(v2), to_np(v1)[::-1], "permuted batch", tol=1e-6)


def _check_single_block(wan, name):
    g = _golden(name)
    s = synth.WORKLOADS[name]
    w, inp, m = _model(wan, s)
    if s.text_dim:
        ctx = m.text_embed(to_dev(inp["text"], BF))
        assert_bf16_close(to_np(ctx[0])[g["ctx_rows"]], g["ctx"], "ctx rows")
    else:
        ctx = to_dev(inp["ctx_txt"], BF)
    ctx_img = to_dev(inp["ctx_img"], BF) if s.img_len else None
    v = m.forward(to_dev(inp["latent"], F32), to_dev(inp["t"], F32), ctx, ctx_img)
    wan.wan_sync_status()
    head = tokens_of(to_np(v))[0, g["rows"]]
    assert_bf16_close(head, g["head"], f"{name} head rows")


def test_wan13b_block(wan):
    _check_single_block(wan, "wan1.3b-block")


def test_wan14b_i2v_block(wan):
    _check_single_block(wan, "wan14b-i2v-block")


def test_wan13b_30blk_guided_step(wan):
    g = _golden("wan1.3b-30blk-guided-step")
    s = synth.STEP_1P3B
    w, inp, m = _model(wan, s)
    del w
    ctx = m.text_embed(to_dev(inp["text"], BF))
    x = to_dev(inp["latent"], F32)
    t = float(inp["t"][0])
    t_pair = torch.tensor([t, t + s.dt], dtype=F32, device="cuda")
    v = m.guided_step(x, t_pair, s.guide_scale, ctx)
    wan.wan_sync_status()
    vt = tokens_of(to_np(v))
    rows = g["rows"]
    assert_bf16_close(vt[0, rows], g["v_cond"], "v_cond")
    assert_bf16_close(vt[1, rows], g["v_uncond"], "v_uncond")
    assert_bf16_close(tokens_of(to_np(x))[0, rows], g["x_next"], "x_next")


def test_wan13b_20step_sampler_shrunk(wan):
    g = _golden("wan1.3b-20step-sampler-shrunk")
    Fr, H, W = (int(a) for a in g["shape"])
    s = synth.SAMPLER_1P3B.replace(frames=Fr, height=H, width=W)
    w, inp, m = _model(wan, s)
    del w
    ctx = m.text_embed(to_dev(inp["text"], BF))
    x = to_dev(inp["latent"], F32)
    m.sample(x, s.steps, s.guide_scale, ctx)
    wan.wan_sync_status()
    assert_bf16_close(to_np(x), g["x_final"], "sampled x0")

"""One DiT block composed from the per-op entry points (wan_patchify, wan_time_embed,
wan_adaln_modulate, wan_linear, wan_attn_rope3d, wan_cross_attn, wan_ffn) at the
full 1.3B and 14B block sizes, checked after every sub-layer against the oracle's
intermediates stored at sampled rows (tests/golden/wan1.3b-block.npz, wan14b-i2v-block.npz)."""
import os

import numpy as np
import pytest
import torch

import synth
from tests.parity import assert_bf16_close, to_dev, to_np

pytestmark = pytest.mark.gpu
BF, F16, F32 = torch.bfloat16, torch.float16, torch.float32
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


@pytest.mark.parametrize("name", ["wan1.3b-block", "wan14b-i2v-block"])
def test_block_composed_from_ops(wan, name):
    path = os.path.join(GOLDEN, f"{name}.npz")
    if not os.path.exists(path):
        pytest.skip("golden not generated")
    g = np.load(path)
    s = synth.WORKLOADS[name]
    w = synth.make_weights(s, 0)
    inp = synth.make_inputs(s, 0)
    m = wan.DiT(s, w)
    blk = m.block_tensors[0]
    t = m.tensors
    D, H, d, L = s.dim, s.heads, s.head_dim, s.tokens
    rows = g["rows"][:len(g["x0"])]
    dev = "cuda"

    def check(key, tensor):
        assert_bf16_close(to_np(tensor)[0, rows], g[key], f"{name} {key}")

    lat = to_dev(inp["latent"], F32)
    x = torch.empty(1, L, D, dtype=F32, device=dev)
    ws = torch.empty(wan.wan_patchify_workspace_size(1, s.c_in, s.frames, s.height, s.width, wan.WAN_BF16),
                     dtype=torch.uint8, device=dev)
    wan.wan_patchify(lat, t["patch_w"], t["patch_b"], x, ws)
    check("x0", x)

    e0, _ = m.time_embed(to_dev(inp["t"], F32))
    mod = e0[0] + blk["mod"].float()          # [6, D]: the block's six modulation vectors
    sh1, sc1, g1, sh2, sc2, g2 = (mod[i].reshape(1, D).contiguous() for i in range(6))

    y = torch.empty(1, L, D, dtype=BF, device=dev)
    wan.wan_adaln_modulate(x, sh1, sc1, y)
    check("y1", y)

    # q and k in fp16 (as the fused forward stores them for the QK^T product), v in bf16
    qk = torch.empty(L, 2 * D, dtype=F16, device=dev)
    wan.wan_linear(y.view(L, D), blk["qkv_w"][:2 * D], blk["qkv_b"][:2 * D], qk)
    v = torch.empty(1, L, H, d, dtype=BF, device=dev)
    wan.wan_linear(y.view(L, D), blk["qkv_w"][2 * D:], blk["qkv_b"][2 * D:], v.view(L, D))
    q, k = (qk[:, i * D:(i + 1) * D].contiguous().view(1, L, H, d) for i in range(2))
    o = torch.empty(1, L, H, d, dtype=BF, device=dev)
    aws = torch.empty(wan.wan_attn_workspace_size(1, L, H, d, wan.WAN_BF16) + 1024, dtype=torch.uint8, device=dev)
    aws = aws[(-aws.data_ptr()) % 1024:]
    wan.wan_attn_rope3d(q, k, v, o, s.grid, ws=aws)
    check("attn", o.view(1, L, D))
    wan.wan_linear(o.view(L, D), blk["o_w"], blk["o_b"], x.view(L, D), wan.WAN_EPI_RESIDUAL, g1, L)
    check("x_sa", x)

    # The cross-attention sub-layer in fp16 storage, as the fused forward runs it: LN
    # output, q, k, v, o and the query / output projection weights.
    y16 = torch.empty(1, L, D, dtype=F16, device=dev)
    wan.wan_adaln_modulate(x, None, None, y16)
    qc = torch.empty(1, L, H, d, dtype=F16, device=dev)
    wan.wan_linear(y16.view(L, D), blk["cq_w"], blk["cq_b"], qc.view(L, D))
    if s.text_dim:
        ctx = m.text_embed(to_dev(inp["text"], BF))
    else:
        ctx = to_dev(inp["ctx_txt"], BF)
    Lt = s.text_len

    def kv_of(c, wname, bname, Lk):
        kb = torch.empty(1, Lk, H, d, dtype=F16, device=dev)
        vb = torch.empty(1, Lk, H, d, dtype=F16, device=dev)
        wan.wan_linear(c.view(Lk, D), blk[wname][:D], blk[bname][:D], kb.view(Lk, D))
        wan.wan_linear(c.view(Lk, D), blk[wname][D:], blk[bname][D:], vb.view(Lk, D))
        return kb, vb

    kt, vt = kv_of(ctx[:1], "ckv_w", "ckv_b", Lt)
    ki = vi = None
    if s.img_len:
        ki, vi = kv_of(to_dev(inp["ctx_img"][:1], BF), "ckvi_w", "ckvi_b", s.img_len)
    oc = torch.empty(1, L, H, d, dtype=F16, device=dev)
    wan.wan_cross_attn(qc, kt, vt, ki, vi, oc)
    wan.wan_linear(oc.view(L, D), blk["co_w"], blk["co_b"], x.view(L, D), wan.WAN_EPI_RESIDUAL)
    check("x_ca", x)

    wan.wan_adaln_modulate(x, sh2, sc2, y)
    check("y2", y)
    hbuf = torch.empty(1, L, s.ffn, dtype=BF, device=dev)
    wan.wan_ffn(y, blk["f1_w"], blk["f1_b"], blk["f2_w"], blk["f2_b"], g2, x, hbuf)
    wan.wan_sync_status()
    check("x_blk", x)

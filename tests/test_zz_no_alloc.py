"""The text projection entry point that allocates nothing (wan_text_embed_noalloc).

It serves callers that cannot allocate device memory: its scratch is a static device
array inside libwan.  Checked through the C ABI against wan_text_embed (which takes a
caller-allocated workspace) on two calls in a row with different inputs: both run the
same kernels on the same inputs, so the results must be bit-identical, and a stale
scratch left by the first call would show up in the second.  One call is also compared
with the CPU oracle under the bf16 tolerance, and sizes beyond the static maximum must
be rejected before any launch.  This file is collected last on purpose.
"""
import pytest
import torch

import synth
from oracle import wan_oracle as O
from tests.parity import assert_bf16_close, to_dev, to_np

pytestmark = pytest.mark.gpu
BF = torch.bfloat16


def _weights(seed, Ct, D):
    rb = synth.round_bf16
    return [rb(synth.normal(seed, n, shp) * 0.02) for n, shp in
            (("na.w1", (D, Ct)), ("na.b1", (D,)), ("na.w2", (D, D)), ("na.b2", (D,)))]


def test_text_embed_noalloc_matches_workspace_version(wan):
    B, Lt, Ct, D = 2, 512, 4096, 1536
    wh = _weights(21, Ct, D)
    w = [to_dev(a, BF) for a in wh]
    ws = torch.empty(wan.wan_text_embed_workspace_size(B, Lt, D, wan.WAN_BF16), dtype=torch.uint8, device="cuda")
    for call in range(2):
        text_h = synth.round_bf16(synth.normal(21 + call, "na.text", (B, Lt, Ct)))
        text = to_dev(text_h, BF)
        ref = torch.empty(B, Lt, D, dtype=BF, device="cuda")
        wan.wan_text_embed(text, *w, ref, ws)
        out = torch.full((B, Lt, D), float("nan"), dtype=BF, device="cuda")
        wan.wan_text_embed_noalloc(text, *w, out)
        wan.wan_sync_status()
        assert torch.equal(out, ref), f"noalloc call {call} differs from the workspace version"
        if call == 1:  # one direct comparison with the oracle (first batch entry, 64 rows)
            o = O.linear(O.gelu(O.linear(text_h[0, :64], wh[0], wh[1])), wh[2], wh[3])
            assert_bf16_close(to_np(out[0, :64]), o, "noalloc text projection vs oracle")


def test_text_embed_noalloc_rejects_oversize(wan):
    # B * Lt * D * 2 bytes beyond the static scratch: rejected on the host, nothing launched.
    B, Lt, Ct, D = 4, 1024, 128, 4096
    assert wan.wan_text_embed_workspace_size(B, Lt, D, wan.WAN_BF16) > wan.wan_text_embed_noalloc_max_bytes()
    st = wan.lib.wan_text_embed_noalloc(None, None, None, None, None, None, B, Lt, Ct, D, wan.WAN_BF16, None)
    assert st == wan.WAN_ERR_WORKSPACE

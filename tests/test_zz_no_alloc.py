"""The text projection entry point that allocates nothing (wan_text_embed_noalloc).

It serves callers that cannot allocate device memory: its scratch is a static device
array inside libwan.  Checked through the C ABI against wan_text_embed (which takes a
caller-allocated workspace) on two calls in a row with different inputs, so a stale
scratch from the first call would show up in the second; and sizes beyond the static
maximum must be rejected before any launch.  This file is collected last on purpose.
"""
import pytest
import torch

import synth
from tests.parity import assert_bf16_close, to_dev, to_np

pytestmark = pytest.mark.gpu
BF = torch.bfloat16


def _weights(seed, Ct, D):
    rb = synth.round_bf16
    return [to_dev(rb(synth.normal(seed, n, shp) * 0.02), BF) for n, shp in
            (("na.w1", (D, Ct)), ("na.b1", (D,)), ("na.w2", (D, D)), ("na.b2", (D,)))]


def test_text_embed_noalloc_matches_workspace_version(wan):
    B, Lt, Ct, D = 2, 512, 4096, 1536
    w = _weights(21, Ct, D)
    ws = torch.empty(wan.wan_text_embed_workspace_size(B, Lt, D, wan.WAN_BF16), dtype=torch.uint8, device="cuda")
    for call in range(2):
        text = to_dev(synth.round_bf16(synth.normal(21 + call, "na.text", (B, Lt, Ct))), BF)
        ref = torch.empty(B, Lt, D, dtype=BF, device="cuda")
        wan.wan_text_embed(text, *w, ref, ws)
        out = torch.full((B, Lt, D), float("nan"), dtype=BF, device="cuda")
        wan.wan_text_embed_noalloc(text, *w, out)
        wan.wan_sync_status()
        assert_bf16_close(to_np(out), to_np(ref), f"noalloc call {call}")


def test_text_embed_noalloc_rejects_oversize(wan):
    # B * Lt * D * 2 bytes beyond the static scratch: rejected on the host, nothing launched.
    B, Lt, Ct, D = 4, 1024, 128, 4096
    assert wan.wan_text_embed_workspace_size(B, Lt, D, wan.WAN_BF16) > wan.wan_text_embed_noalloc_max_bytes()
    st = wan.lib.wan_text_embed_noalloc(None, None, None, None, None, None, B, Lt, Ct, D, wan.WAN_BF16, None)
    assert st == wan.WAN_ERR_WORKSPACE

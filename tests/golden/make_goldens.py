"""Write the stored expected values of the full-size parity tests.

Every value here is computed by the CPU fp64 oracle (``oracle/wan_oracle.py``)
from the seeded synthetic inputs (``synth``); nothing comes from the CUDA path.
The GPU tests regenerate the same inputs from the same seeds and compare the
kernels' outputs with these values at the stored positions.

    python tests/golden/make_goldens.py --workload wan1.3b-block               # one 1.3B block (minutes)
    python tests/golden/make_goldens.py --workload wan1.3b-30blk-guided-step   # 30 blocks x 2 branches (~3 h on 8 cores)
    python tests/golden/make_goldens.py --workload wan14b-i2v-block            # one 14B I2V block
    python tests/golden/make_goldens.py --workload wan1.3b-20step-sampler      # 20 steps on a shrunk latent
    python tests/golden/make_goldens.py --workload wan1.3b-block --fp8 3       # the 8-bit variant of one block
    python tests/golden/make_goldens.py --workload wan14b-i2v-block --fp8 3    # the same at the 14B I2V shape

Outputs ``tests/golden/<workload>.npz`` (``-shrunk`` for the sampler, ``-fp8`` for the
8-bit variant; float32 values, int64 indices).
"""
import argparse
import os
import sys
import time

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import synth  # noqa: E402
from oracle import wan_oracle as O  # noqa: E402

SEED = 0
N_TRACE = 8   # sampled rows whose block intermediates are stored
# The 20-step sampler is checked on a shrunk latent with the full 30-block widths.
SHRUNK_SAMPLER = dict(frames=5, height=16, width=16)


def f32(a):
    return np.asarray(a, np.float32)


def single_block(name, n_rows, fp8=0):
    s = synth.WORKLOADS[name].replace(fp8=fp8)
    w = synth.make_weights(s, SEED)
    inp = synth.make_inputs(s, SEED)
    if s.text_dim:
        ctx = O.text_projection(inp["text"], w)
    else:
        ctx = np.asarray(inp["ctx_txt"], np.float64)
    ctx_img = inp.get("ctx_img")
    rows = synth.sample_rows(s.tokens, n_rows, SEED)
    trace = {}
    tok, xb = O.dit_forward(inp["latent"], inp["t"], ctx, ctx_img, w, s, rows=rows, trace=trace)
    tr = trace["per_batch"][0]
    # Head outputs at every sampled token; intermediates at the first N_TRACE of them.
    out = dict(rows=rows.astype(np.int64), head=f32(tok[0]), x_blk=f32(xb[0][:N_TRACE]),
               ctx_rows=np.arange(0, s.text_len, s.text_len // 8).astype(np.int64))
    out["ctx"] = f32(ctx[0][out["ctx_rows"]])
    for key in ("x0", "y1", "q", "k", "v", "attn", "x_sa", "x_ca", "y2"):
        out[key] = f32(tr[key][:N_TRACE])
    _, e0, hm = O.time_embedding(inp["t"], w, s.dim, s.freq_dim)
    out["e0"], out["hm"] = f32(e0[0]), f32(hm[0])
    return out


def guided_step_full(n_rows):
    s = synth.STEP_1P3B
    w = synth.make_weights(s, SEED)
    inp = synth.make_inputs(s, SEED)
    ctx = O.text_projection(inp["text"], w)
    t = float(inp["t"][0])
    lat = np.concatenate([inp["latent"]] * 2, axis=0)
    v = O.dit_forward(lat, np.array([t, t]), ctx, None, w, s)
    x_next = O.cfg_euler_step(inp["latent"], v[0:1], v[1:2], s.guide_scale, s.dt)
    rows = synth.sample_rows(s.tokens, n_rows, SEED)
    vt = O.patchify_tokens(v)
    xt = O.patchify_tokens(x_next)
    return dict(rows=rows.astype(np.int64), v_cond=f32(vt[0, rows]), v_uncond=f32(vt[1, rows]),
                x_next=f32(xt[0, rows]))


def sampler_shrunk():
    s = synth.SAMPLER_1P3B.replace(**SHRUNK_SAMPLER)
    w = synth.make_weights(s, SEED)
    inp = synth.make_inputs(s, SEED)
    ctx = O.text_projection(inp["text"], w)
    x = O.sample(inp["latent"], ctx, None, w, s, s.steps)
    return dict(x_final=f32(x), shape=np.array([s.frames, s.height, s.width], np.int64))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--workload", required=True, choices=["wan1.3b-block", "wan1.3b-30blk-guided-step",
                                                          "wan14b-i2v-block", "wan1.3b-20step-sampler"])
    ap.add_argument("--fp8", type=int, default=0, help="8-bit variant bits (single-block workloads)")
    a = ap.parse_args()
    t0 = time.time()
    name = a.workload
    if a.fp8 and name not in ("wan1.3b-block", "wan14b-i2v-block"):
        ap.error("--fp8 applies to the single-block workloads")
    if name in ("wan1.3b-block", "wan14b-i2v-block"):
        out = single_block(name, 512 if name == "wan1.3b-block" else 256, a.fp8)
        if a.fp8:
            name += "-fp8"
            out["fp8"] = np.array(a.fp8, np.int64)
    elif name == "wan1.3b-30blk-guided-step":
        out = guided_step_full(512)
    else:
        out = sampler_shrunk()
        name += "-shrunk"
    path = os.path.join(HERE, f"{name}.npz")
    np.savez_compressed(path, **out)
    print(f"wrote {path} in {time.time() - t0:.1f} s")


if __name__ == "__main__":
    main()

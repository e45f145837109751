"""B300-native (sm_103a) Wan video-DiT denoising step.

The compute lives in libwan.so (hand-written CUDA: tcgen05/TMEM GEMMs fed by TMA,
a tcgen05 flash-attention kernel, fused elementwise passes) behind the C ABI in
include/wan.h.  ``video_diffusion_transformer_04_b300.wan`` is the thin ctypes
binding; build the library with ``python -m video_diffusion_transformer_04_b300._build``.
"""

__all__ = ["wan"]

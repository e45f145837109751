/*
 * wan.h - C ABI of libwan: the Wan video-DiT denoising step on one B300 (sm_103a).
 *
 * Sources of the operations (cited by page title and section):
 *   [Method]  hyper.ai summary of "Wan: Open and Advanced Large-Scale Video Generative
 *             Models" (arXiv 2503.20314), section "方法" (Method): patchify by a (1,2,2)
 *             3D conv into (B, L, D); transformer blocks with text cross-attention; an MLP
 *             of Linear + SiLU on the time embedding predicting six modulation
 *             parameters; a depatchify module; flow matching on the linear path between
 *             data x1 and noise x0.
 *   [Code]    zizhi168.cn "阿里Wan 2.1视频生成模型深度剖析", section "核心代码实现亮点":
 *             the classifier-free guidance combination, DiT-style modulation, self- and
 *             cross-attention per block, rope_apply(q|k, grid_sizes, freqs) before
 *             flash_attention, CLIP context concatenated ahead of the text context.
 *   [I2V]     x-humanoid.csdn.net notes on the Wan report, section 1.1 "模型设计": noise,
 *             condition latent and mask concatenated on channels, zero-initialised extra
 *             projection, decoupled cross-attention to CLIP image features.
 *   [Sampler] kwkr.cn hands-on article, sections 3.2 and 4.4: Euler integration,
 *             about 20 steps, latent = latent + v*dt.
 *
 * Conventions shared by every entry point:
 *   - Every tensor argument is a DEVICE pointer owned by the caller.  libwan never
 *     allocates, frees or retains device memory; the only scratch is the caller's
 *     workspace (ws, ws_bytes), sized by the matching *_workspace_size function.
 *   - Layouts are dense row-major (C order), 16-byte aligned; the workspace 1024-byte
 *     aligned.  Token order inside a sample is (f, i, j) with j fastest, i.e. token
 *     l = (f*Hp + i)*Wp + j on the patch grid (Fg, Hp, Wp) = (F, H/2, W/2).
 *   - Weights use the nn.Linear layout [out, in].  With dtype WAN_BF16 every weight,
 *     bias and activation argument is bf16 (fp32 accumulation); with WAN_F32 they are
 *     fp32 (the parity path).  The residual stream x, the latent and the velocity are
 *     always fp32.
 *   - Everything is enqueued asynchronously on `stream` (NULL = legacy default stream).
 *   - Return value: WAN_OK (0) or a negative status.  Arguments are validated on the
 *     host before anything is launched; on an error nothing, or only a prefix of the
 *     work, has been enqueued and the outputs are undefined.  Kernels never trap: a
 *     pipeline wait that exceeds its time limit sets a device status word that
 *     wan_sync_status() reports as WAN_ERR_TIMEOUT.  There is no CPU fallback.
 */
#ifndef WAN_H_
#define WAN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* wan_stream_t; /* identical to cudaStream_t */

enum wan_status_code {
  WAN_OK = 0,
  WAN_ERR_INVALID_ARG = -1, /* NULL pointer, non-positive size, inconsistent shape */
  WAN_ERR_UNSUPPORTED = -2, /* shape/alignment/dtype the kernels do not handle */
  WAN_ERR_CUDA = -3,        /* a CUDA runtime call or launch failed */
  WAN_ERR_TIMEOUT = -4,     /* a device pipeline wait ran out of time */
  WAN_ERR_WORKSPACE = -5    /* ws NULL, misaligned or smaller than required */
};

/* Storage types.  WAN_F16 (fp16) is accepted only where an entry point says so: for the
 * q and k operands of the attention calls next to bf16 v and o (fp16 keeps 3 more
 * mantissa bits in the logits q.k than bf16), for the whole cross-attention sub-layer
 * (wan_adaln_modulate's output, wan_linear's operands and output, wan_cross_attn's v and
 * o), and as the output of wan_linear. */
enum wan_dtype { WAN_BF16 = 0, WAN_F32 = 1, WAN_F16 = 2 };

/* Epilogues of wan_linear: y = x W^T + b followed by ... */
enum wan_epilogue {
  WAN_EPI_STORE = 0,    /* store y in out_dtype */
  WAN_EPI_GELU = 1,     /* store GELU(y) (erf form) in out_dtype */
  WAN_EPI_RESIDUAL = 2, /* x_f32[m, n] += gate[m / rows_per_gate, n] * y (gate NULL: 1) */
  WAN_EPI_GELU_TANH = 3 /* store GELU(y) in its tanh form, 0.5 y (1 + tanh(sqrt(2/pi)(y + 0.044715 y^3))) */
};

/* Human-readable text of a status code (static storage). */
const char* wan_status_string(int status);

/* Synchronise `stream`, then read and clear the device status word of the current
 * device.  Returns WAN_ERR_TIMEOUT if any kernel since the last call gave up on a
 * pipeline wait, WAN_ERR_CUDA if the synchronisation failed, else WAN_OK. */
int wan_sync_status(wan_stream_t stream);

/* Number of libwan kernels launched by this process so far (all devices). */
long long wan_launch_count(void);

/* Failure-path self-test (no counterpart in the pages): enqueues one kernel whose only
 * pipeline wait is on a barrier nothing arrives on.  The bounded wait gives up after
 * limit_ms (1..1000) and records a timeout in the device status word, exactly as a
 * stalled pipeline would; the next wan_sync_status returns WAN_ERR_TIMEOUT and clears
 * it.  Nothing faults, traps or hangs; the context stays usable. */
int wan_watchdog_selftest(int limit_ms, wan_stream_t stream);

/* ------------------------------------------------------------------ patchify
 * [Method] patchify: a 3D conv with kernel = stride = (1,2,2) maps the latent
 * [B, C, F, H, W] to the token sequence x [B, L, D], L = F*(H/2)*(W/2):
 *   x[b, l, :] = bias + sum_{c,di,dj} w[:, c*4 + di*2 + dj] * latent[b, c, f, 2i+di, 2j+dj].
 * latent: fp32 [B, C, F, H, W] (H, W even).  w: [D, C*4], b: [D] (dtype).
 * x: fp32 [B, L, D] (the residual stream; overwritten).
 * ws: >= wan_patchify_workspace_size(...) bytes (the gathered patches).
 * Needs D % 32 == 0. */
size_t wan_patchify_workspace_size(int B, int C, int F, int H, int W, int dtype);
int wan_patchify(const float* latent, const void* w, const void* b, float* x, int B, int C, int F,
                 int H, int W, int D, int dtype, void* ws, size_t ws_bytes, wan_stream_t stream);

/* ------------------------------------------------------------------ AdaLN
 * [Code] DiT-style modulation: y = LN(x) * (1 + scale[b]) + shift[b], LN over D with
 * biased variance, no affine, epsilon eps.  x: fp32 [B, L, D]; shift, scale: fp32 [B, D]
 * (both NULL: plain LN).  y: [B, L, D] in dtype (WAN_BF16, WAN_F16 or WAN_F32; fp16 is
 * meant for the unmodulated LN of the cross-attention query, whose rows have norm
 * sqrt(D)).  Needs D % 4 == 0, D <= 8192. */
int wan_adaln_modulate(const float* x, const float* shift, const float* scale, void* y, int B, int L,
                       int D, float eps, int dtype, wan_stream_t stream);

/* ------------------------------------------------------------------ self-attention
 * [Code] x = flash_attention(q=rope_apply(q, grid_sizes, freqs), k=rope_apply(k, ...), v):
 * full bidirectional softmax(q k^T / sqrt(d)) v per (batch, head), no mask.
 * 3D RoPE: the head dim splits into [frame | height | width] parts of sizes
 * (d - 4*floor(d/6), 2*floor(d/6), 2*floor(d/6)); adjacent pairs (2m, 2m+1) of part a
 * rotate by pos_a * theta^(-2j/d_a), pos = the token's (f, i, j) on the grid
 * (Fg, Hg, Wg), Fg*Hg*Wg == L.
 * v, o: [B, L, H, d] in dtype; q, k: [B, L, H, d] in qk_dtype (= dtype, or WAN_F16 with
 * dtype WAN_BF16).  apply_rope = 0 treats q and k as already rotated.  With dtype
 * WAN_BF16 the rotated q and k enter the QK^T product in fp16.
 * kv_lens: DEVICE int [B] or NULL.  [Code] flash_attention(..., k_lens=seq_lens): entry b
 * attends to its first kv_lens[b] keys only (values outside [1, L] are clamped to that
 * range); keys past that length must hold finite values (they get weight exactly 0).
 * NULL: every entry attends to all L keys.
 * ws (the rotated q and k): >= wan_attn_workspace_size(...) bytes, 1024-byte aligned;
 * unused (may be NULL) when apply_rope = 0.  d must be 64 or 128 (bf16 path); d <= 128
 * and even (fp32 path). */
size_t wan_attn_workspace_size(int B, int L, int H, int d, int dtype);
int wan_attn_rope3d(const void* q, const void* k, const void* v, void* o, const int* kv_lens, int B,
                    int L, int H, int d, int Fg, int Hg, int Wg, float theta, int apply_rope, int dtype,
                    int qk_dtype, void* ws, size_t ws_bytes, wan_stream_t stream);

/* ------------------------------------------------------------------ QKV projection + 3D RoPE
 * [Code] q, k, v = projections of the modulated input, then rope_apply(q | k, grid_sizes,
 * freqs): the self-attention's QKV projection with the rotation fused into its epilogue
 * (the same kernel as inside wan_dit_forward).
 *   qkv[b, l, :] = [q | k | v] = y[b, l, :] w^T + b, then q and k of every head rotated
 *   as described for wan_attn_rope3d (grid (Fg, Hg, Wg), Fg*Hg*Wg == L, base theta).
 * y: [B, L, D] (dtype: WAN_BF16 or WAN_F32), D = H*d; w: [3D, D]; b: [3D] or NULL (dtype).
 * qkv: [B, L, 3D]; with WAN_BF16 the q and k columns [0, 2D) hold fp16 values and the v
 * columns bf16 (the storage the attention kernels take); with WAN_F32 all fp32.
 * ws: >= wan_qkv_rope_workspace_size(d) bytes, 16-byte aligned (the pair frequencies).
 * wan_qkv_rope_e4m3: the FP8 form of the 8-bit variant: y8 [B*L, D] E4M3 codes with row
 * scales sy [B*L], w8 [3D, D] codes with row scales sw [3D] (as wan_quant_rows_e4m3
 * writes them), b bf16; output as for WAN_BF16.  Needs D % 32 == 0 (and d % 32 == 0
 * with 16-bit output). */
size_t wan_qkv_rope_workspace_size(int d);
int wan_qkv_rope(const void* y, const void* w, const void* b, void* qkv, int B, int L, int H, int d, int Fg,
                 int Hg, int Wg, float theta, int dtype, void* ws, size_t ws_bytes, wan_stream_t stream);
int wan_qkv_rope_e4m3(const void* y8, const float* sy, const void* w8, const float* sw, const void* b,
                      void* qkv, int B, int L, int H, int d, int Fg, int Hg, int Wg, float theta, void* ws,
                      size_t ws_bytes, wan_stream_t stream);

/* ------------------------------------------------------------------ cross-attention
 * [Method] text conditioning by cross-attention; [I2V] decoupled cross-attention to the
 * CLIP image context: o = softmax(q kt^T/sqrt(d)) vt + softmax(q ki^T/sqrt(d)) vi
 * (the second term only when ki != NULL).  Both softmaxes run in one launch; the two
 * terms are summed in fp32 and rounded once (in the 16-bit formats the text term is
 * parked in o between the two segments, so it is rounded to o's type once more).
 * o: [B, L, H, d]; vt: [B, Lt, H, d]; vi: [B, Li, H, d] or NULL (dtype: WAN_BF16, WAN_F16
 * or WAN_F32).
 * q: [B, L, H, d]; kt: [B, Lt, H, d]; ki: [B, Li, H, d] or NULL (qk_dtype: dtype, or
 * WAN_F16 with dtype WAN_BF16; WAN_F16 with dtype WAN_F16).
 * kt_lens: DEVICE int [B] or NULL: valid text tokens per entry of a padded context (the
 * k_lens of [Code]; clamped to [1, Lt]; padded keys must be finite); the image segment
 * is always fully valid.
 * ws, ws_bytes: unused (wan_cross_attn_workspace_size returns 0; q, k, v are read in
 * place), kept so a caller can pass the same workspace to every attention call. */
size_t wan_cross_attn_workspace_size(int B, int Lt, int Li, int H, int d, int dtype);
int wan_cross_attn(const void* q, const void* kt, const void* vt, const int* kt_lens, const void* ki,
                   const void* vi, void* o, int B, int L, int Lt, int Li, int H, int d, int dtype,
                   int qk_dtype, void* ws, size_t ws_bytes, wan_stream_t stream);

/* ------------------------------------------------------------------ FFN
 * FFN sub-layer with gated residual: x += gate[b] * (W2 GELU(W1 y + b1) + b2).
 * y: [B, L, D] modulated input (dtype); w1: [F, D], b1: [F]; w2: [D, F], b2: [D];
 * gate: fp32 [B, D] (NULL: 1); x_inout: fp32 [B, L, D]; h_ws: [B, L, F] (dtype) scratch.
 * Needs D % 32 == 0, F % 32 == 0. */
int wan_ffn(const void* y, const void* w1, const void* b1, const void* w2, const void* b2,
            const float* gate, float* x_inout, void* h_ws, int B, int L, int D, int F, int dtype,
            wan_stream_t stream);

/* ------------------------------------------------------------------ linear
 * One projection y = x W^T + b with an epilogue (enum wan_epilogue); the GEMM under every
 * projection of the block.  x: [M, K] and w: [N, K] in dtype (WAN_BF16, WAN_F16 or
 * WAN_F32; x and w share it); b: [N] or NULL (bf16 with the 16-bit dtypes, else fp32).
 * WAN_EPI_STORE / WAN_EPI_GELU write out [M, N] in out_dtype (WAN_BF16 or WAN_F16 only
 * with a 16-bit dtype).  WAN_EPI_RESIDUAL accumulates into the fp32 out [M, N] with the
 * optional fp32 gate [M / rows_per_gate, N] (out_dtype WAN_F32).  Needs K % 8 == 0,
 * N % 32 == 0. */
int wan_linear(const void* x, const void* w, const void* b, void* out, int M, int N, int K,
               int epilogue, const float* gate, int rows_per_gate, int dtype, int out_dtype,
               wan_stream_t stream);

/* ------------------------------------------------------------------ 8-bit variant
 * [Method] (hyper.ai summary of the Wan report, section 方法, the inference paragraph):
 * FP8 GEMMs and an 8-bit FlashAttention speed up the DiT.  READING (the pages fix no
 * format or scaling): OCP FP8 E4M3 codes, round to nearest even, saturating at +-448;
 * one scale per group, decided in fp32: amax = max |x|, inv = 448 / amax,
 * code = e4m3(x * inv), dequantisation scale s = amax / 448 (an all-zero group: s = 0).
 * Groups: GEMM activations per row (token), GEMM weights per row (output channel);
 * attention q per (token, head), k per (head, block of 128 keys), v per (head, channel)
 * over all keys.  Codes are plain bytes (no device type in these signatures).
 *
 * wan_quant_rows_e4m3: x [M, K] in dtype (WAN_BF16, WAN_F16 or WAN_F32; row stride ldx
 *   elements, 16-byte aligned rows) -> x8 [M, K] codes (row stride ld8 bytes), s [M] fp32.
 *   K, ldx and ld8 multiples of 4. */
int wan_quant_rows_e4m3(const void* x, int dtype, long long ldx, int M, int K, void* x8, long long ld8,
                        float* s, wan_stream_t stream);

/* wan_quant_attn_e4m3: the 8-bit operands of self-attention.
 *   q, k: [B, L, H*d] in qk_dtype; v: [B, L, H*d] in v_dtype (WAN_BF16 or WAN_F16 each).
 *   Outputs (device, caller-owned): q8 [B, L, H*d] codes, sq [B, L, H];
 *   k8 [B, L, H*d], sk [B, H, ceil(L/128)]; v8t [B, H, d, Lp] (v transposed, keys
 *   contiguous, Lp = L rounded up to 16, pad keys zero), sv [B, H, d].
 *   ws: >= wan_quant_attn_workspace_size(B, H, d) bytes (per-channel |max| of v).
 *   d must be 128; all pointers 16-byte aligned. */
size_t wan_quant_attn_workspace_size(int B, int H, int d);
int wan_quant_attn_e4m3(const void* q, const void* k, const void* v, int qk_dtype, int v_dtype, int B, int L,
                        int H, int d, void* q8, float* sq, void* k8, float* sk, void* v8t, float* sv,
                        void* ws, size_t ws_bytes, wan_stream_t stream);

/* wan_attn_e4m3: o = softmax(Q K^T / sqrt(d)) V with Q, K, V the dequantised operands in
 *   the layouts wan_quant_attn_e4m3 writes; both products run on 8-bit tensor cores with
 *   fp32 accumulation, the probabilities are rounded to E4M3 inside the kernel (relative
 *   error <= 2^-4 each in the normal range).  o: bf16 [B, L, H*d]; kv_lens as for
 *   wan_attn_rope3d.  d must be 128. */
int wan_attn_e4m3(const void* q8, const float* sq, const void* k8, const float* sk, const void* v8t,
                  const float* sv, void* o, const int* kv_lens, int B, int L, int H, int d, wan_stream_t stream);

/* wan_linear_e4m3: out = (x8 sx)(w8 sw)^T + b, every product of two codes exact, fp32
 *   accumulation, with an epilogue as for wan_linear: WAN_EPI_STORE / WAN_EPI_GELU /
 *   WAN_EPI_GELU_TANH write bf16 out [M, N]; WAN_EPI_RESIDUAL accumulates into fp32 out
 *   with the optional gate.  x8 [M, K] codes, sx [M]; w8 [N, K] codes, sw [N] (16-byte
 *   aligned); b [N] bf16 or NULL.  K % 16 == 0, N % 32 == 0. */
int wan_linear_e4m3(const void* x8, const float* sx, const void* w8, const float* sw, const void* b, void* out,
                    int M, int N, int K, int epilogue, const float* gate, int rows_per_gate, wan_stream_t stream);

/* ------------------------------------------------------------------ text projection
 * Projection of the text-encoder output (umT5 width Ct) to the DiT width D.
 * READING (pages silent on its form): ctx = W2 GELU(W1 text + b1) + b2.
 * text: [B, Lt, Ct]; w1: [D, Ct], b1: [D]; w2: [D, D], b2: [D]; ctx: [B, Lt, D] (dtype). */
size_t wan_text_embed_workspace_size(int B, int Lt, int D, int dtype);
int wan_text_embed(const void* text, const void* w1, const void* b1, const void* w2, const void* b2,
                   void* ctx, int B, int Lt, int Ct, int D, int dtype, void* ws, size_t ws_bytes,
                   wan_stream_t stream);

/* ------------------------------------------------------------------ text projection without allocation
 * No counterpart in the paper: a library convenience.  Same computation and result as
 * wan_text_embed, for callers that cannot allocate device memory (a host that owns the
 * whole allocator and passes only fixed input/output buffers, or a latency-critical path
 * where an allocation may stall or fail).  The scratch (the hidden activations between
 * the two linear layers) lives in a static device array of
 * wan_text_embed_noalloc_max_bytes() = 16 MiB inside libwan, held by every GPU that
 * loads the library until the process exits; nothing is allocated per call.
 *   - Sizes whose scratch, wan_text_embed_workspace_size(B, Lt, D, dtype), exceeds the
 *     maximum are rejected with WAN_ERR_WORKSPACE before anything is launched (bf16: up
 *     to B*Lt*D = 8 Mi elements).
 *   - Every call looks up the array's device address on the current device
 *     (cudaGetSymbolAddress, no allocation); the first lookup on a device may load the
 *     library's module there, so make the first call on each device outside stream
 *     capture.
 *   - Every call on a device shares the one array, which keeps the last call's contents
 *     (the scratch is fully written before it is read, so nothing needs clearing).
 *     Calls whose work overlaps on the GPU (different streams, concurrent graphs) race on
 *     the array: serialise them.
 * Arguments as for wan_text_embed, without ws / ws_bytes. */
int wan_text_embed_noalloc(const void* text, const void* w1, const void* b1, const void* w2, const void* b2,
                           void* ctx, int B, int Lt, int Ct, int D, int dtype, wan_stream_t stream);
size_t wan_text_embed_noalloc_max_bytes(void);

/* ------------------------------------------------------------------ CFG + Euler
 * [Code] noise_pred = uncond + s * (cond - uncond); [Sampler 4.4] x <- x + v * dt, with
 * t running from 1 (noise) to 0 (data) and dt = t_next - t:
 *   x[i] <- x[i] + dt * (v_uncond[i] + guide_scale * (v_cond[i] - v_uncond[i])).
 * x: fp32 [n] in place; v_cond, v_uncond: [n] in v_dtype (WAN_BF16 or WAN_F32).
 * n == 0 is a no-op. */
int wan_cfg_euler_step(float* x, const void* v_cond, const void* v_uncond, long long n,
                       float guide_scale, float dt, int v_dtype, wan_stream_t stream);

/* ------------------------------------------------------------------ whole DiT forward */
/* With dtype WAN_BF16 the cross-attention sub-layer runs in fp16 storage: its LN output,
 * q, k, v, probabilities and o, and therefore its two square weights cq_w and co_w, which
 * the caller stores in fp16 (every other weight, bias and activation is bf16).  Its
 * values are bounded (an unmodulated LN row has norm sqrt(D); the probabilities stay
 * below 2^15), and fp16's 3 extra mantissa bits keep the error of wide models' peaked
 * softmaxes at the level of the narrow ones. */
typedef struct wan_dit_config {
  int dtype;       /* WAN_BF16 or WAN_F32 */
  int batch;       /* B */
  int c_in, c_out; /* latent channels in (16; 36 for I2V) and predicted (16) */
  int frames, height, width; /* latent F, H, W (H, W even) */
  int dim, heads, head_dim, ffn, blocks;
  int text_len;    /* Lt */
  int img_len;     /* Li (0: text-to-video) */
  int freq_dim;    /* sinusoid width of the time embedding (256) */
  float theta;     /* RoPE base (10000) */
  float eps;       /* LayerNorm epsilon (1e-6) */
  /* Variants the pages do not describe, off (0) by default, for fidelity with released
   * checkpoints: RMSNorm with a learned weight (epsilon eps) on the full-width q and k
   * before RoPE, and the tanh form of GELU in the FFN. */
  int qk_norm;
  int gelu_tanh;
  /* 8-bit variant (bf16 path, head_dim 128), off (0) by default: bit 0 = 8-bit
   * self-attention, bit 1 = FP8 QKV and FFN-up GEMMs (their activations leave the
   * LayerNorm + modulation pass as per-token E4M3 codes; the weights come quantised per
   * output channel in wan_block_weights). */
  int fp8;
} wan_dit_config;

typedef struct wan_block_weights {
  const void* mod;                  /* [6, D]  learned bias added to the shared e0 */
  const void *qkv_w, *qkv_b;        /* [3D, D], [3D] */
  const void *o_w, *o_b;            /* [D, D], [D] */
  const void *cq_w, *cq_b;          /* [D, D], [D]   cross-attention query (cq_w fp16 with WAN_BF16) */
  const void *ckv_w, *ckv_b;        /* [2D, D], [2D] text key|value */
  const void *ckvi_w, *ckvi_b;      /* [2D, D], [2D] image key|value (NULL when img_len == 0) */
  const void *co_w, *co_b;          /* [D, D], [D]   cross-attention output (co_w fp16 with WAN_BF16) */
  const void *f1_w, *f1_b;          /* [F, D], [F] */
  const void *f2_w, *f2_b;          /* [D, F], [D] */
  const void *norm_q_w, *norm_k_w;  /* [D], [D] RMSNorm weights (only with qk_norm) */
  /* only with fp8 bit 1: E4M3 codes of qkv_w and f1_w and their per-row scales, as
   * written by wan_quant_rows_e4m3 */
  const void* qkv_w8;
  const float* qkv_ws;              /* [3D] */
  const void* f1_w8;
  const float* f1_ws;               /* [F] */
} wan_block_weights;

typedef struct wan_dit_weights {
  const void *patch_w, *patch_b;    /* [D, c_in*4], [D] */
  const void *t1_w, *t1_b;          /* [D, freq_dim], [D] */
  const void *t2_w, *t2_b;          /* [D, D], [D] */
  const void *m_w, *m_b;            /* [6D, D], [6D]  block modulation (shift1,scale1,gate1,shift2,scale2,gate2) */
  const void *hm_w, *hm_b;          /* [2D, D], [2D]  head modulation (shift, scale) */
  const void *head_w, *head_b;      /* [c_out*4, D], [c_out*4] */
  const wan_block_weights* blocks;  /* HOST array of `blocks` entries (device pointers inside) */
} wan_dit_weights;

/* Bytes of workspace wan_dit_forward / wan_dit_guided_step / wan_sample need. */
size_t wan_dit_workspace_size(const wan_dit_config* cfg);

/* [Method] time conditioning: an MLP of Linear and SiLU layers on the sinusoidal time
 * embedding, shared by all blocks, predicting the six modulation vectors.
 * READING (pages silent on the exact form): s = [cos(1000 t w_k), sin(1000 t w_k)],
 * w_k = 10000^(-k/(freq_dim/2)); e = t2(SiLU(t1(s))); e0 = m(SiLU(e)) -> [B, 6, D]
 * (shift1, scale1, gate1, shift2, scale2, gate2); hm = hm(SiLU(e)) -> [B, 2, D]
 * (head shift, scale).  t: fp32 DEVICE, t[b * t_stride]; e0, hm: fp32 outputs.
 * Uses the t1/t2/m/hm weights of `w` only.  ws: >= wan_time_embed_workspace_size(cfg). */
size_t wan_time_embed_workspace_size(const wan_dit_config* cfg);
int wan_time_embed(const wan_dit_config* cfg, const wan_dit_weights* w, const float* t, int t_stride, float* e0,
                   float* hm, void* ws, size_t ws_bytes, wan_stream_t stream);

/* [Method] + [Code]: the DiT velocity prediction.  patchify -> `blocks` transformer
 * blocks (AdaLN-modulated self-attention with 3D RoPE, cross-attention to ctx_txt (and
 * decoupled ctx_img), AdaLN-modulated GELU FFN, gated residuals) -> head -> depatchify.
 * latent: fp32 [B, c_in, F, H, W], or [1, ...] broadcast to every batch entry when
 * latent_broadcast != 0; t: fp32 [B] DEVICE timesteps in [0, 1]; ctx_txt: [B, Lt, D];
 * txt_lens: DEVICE int [B] valid text tokens per entry of a padded ctx_txt, or NULL (all
 * Lt valid); ctx_img: [B, Li, D] or NULL (dtype); v_out: fp32 [B, c_out, F, H, W].
 * ws: >= wan_dit_workspace_size(cfg) bytes, 1024-byte aligned. */
int wan_dit_forward(const wan_dit_config* cfg, const wan_dit_weights* w, const float* latent,
                    int latent_broadcast, const float* t, const void* ctx_txt, const int* txt_lens,
                    const void* ctx_img, float* v_out, void* ws, size_t ws_bytes, wan_stream_t stream);

/* One guided denoising step (cfg->batch must be 2: cond, uncond).  Runs the DiT on
 * [cond; uncond] with the shared latent x and timestep, then fuses CFG and the Euler
 * update into x's first c_out channels.  x: fp32 [1, c_in, F, H, W] in/out;
 * t_pair: fp32 DEVICE {t, t_next}; ctx_txt: [2, Lt, D] (cond first); txt_lens: DEVICE int
 * [2] or NULL; ctx_img: [2, Li, D] or NULL.  v_ws: fp32 [2, c_out, F, H, W] receives the
 * two velocity predictions. */
int wan_dit_guided_step(const wan_dit_config* cfg, const wan_dit_weights* w, float* x,
                        const float* t_pair, float guide_scale, const void* ctx_txt,
                        const int* txt_lens, const void* ctx_img, float* v_ws, void* ws,
                        size_t ws_bytes, wan_stream_t stream);

/* [Sampler 3.2, 4.4] End-to-end Euler sampling: `steps` guided steps on the uniform
 * schedule t_k = 1 - k/steps, from noise x (t = 1) to the data estimate (t = 0).
 * The contexts do not depend on t, so every block's cross-attention keys and values are
 * projected once, into the workspace, and reused by all steps (the same result as
 * projecting them at every step).  ws: >= wan_sample_workspace_size(cfg) bytes,
 * 1024-byte aligned.  t_sched: fp32 DEVICE scratch of steps+1 floats; other arguments as
 * for wan_dit_guided_step. */
size_t wan_sample_workspace_size(const wan_dit_config* cfg);
int wan_sample(const wan_dit_config* cfg, const wan_dit_weights* w, float* x, int steps,
               float guide_scale, const void* ctx_txt, const int* txt_lens, const void* ctx_img,
               float* t_sched, float* v_ws, void* ws, size_t ws_bytes, wan_stream_t stream);

/* ------------------------------------------------------------------ profiling
 * Kernel timing with CUDA events recorded around every libwan launch while enabled.
 * wan_profile_begin(capacity) starts recording (at most `capacity` launches);
 * wan_profile_end(names, ms, counts, n_kinds) synchronises the recorded events and
 * writes, per kernel kind, the total milliseconds and launch count; returns the number
 * of kinds written (or a negative status).  names receives static strings. */
int wan_profile_begin(int capacity);
int wan_profile_end(const char** names, double* ms, int* counts, int max_kinds);

#ifdef __cplusplus
}
#endif

#endif /* WAN_H_ */

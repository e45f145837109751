// C ABI of libwan (include/wan.h): argument validation, tensor-map creation, workspace
// planning, the orchestration of the DiT forward / guided step / sampler, and the
// launch counter and event profiler.  No entry point allocates device memory.
#include <atomic>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <vector>

#include <cudaTypedefs.h>

#include "kernels.h"

// Device status word (per device context): kernels record pipeline-wait timeouts here.
__device__ int g_wan_status = 0;

namespace wan {

// ------------------------------------------------------------------ launch bookkeeping
static std::atomic<long long> g_launches{0};

struct ProfRec {
  const char* kind;
  cudaEvent_t a, b;
};
static std::mutex g_prof_mu;
static bool g_prof_on = false;
static bool g_prof_open = false;
static std::vector<ProfRec> g_recs;
static std::vector<cudaEvent_t> g_pool;
static size_t g_cap = 0;

void count_launch(const char* kind, cudaStream_t stream, bool begin) {
  if (begin) g_launches.fetch_add(1, std::memory_order_relaxed);
  if (!g_prof_on) return;
  std::lock_guard<std::mutex> lk(g_prof_mu);
  if (begin) {
    g_prof_open = false;
    if (g_recs.size() < g_cap) {
      const size_t i = g_recs.size();
      ProfRec r{kind, g_pool[2 * i], g_pool[2 * i + 1]};
      if (cudaEventRecord(r.a, stream) == cudaSuccess) {
        g_recs.push_back(r);
        g_prof_open = true;
      }
    }
  } else if (g_prof_open) {
    cudaEventRecord(g_recs.back().b, stream);
    g_prof_open = false;
  }
}

struct DevInfo {
  int* status = nullptr;
  int num_sms = 0;
};
static std::mutex g_dev_mu;
static DevInfo g_dev[64];

int launch_ctx(cudaStream_t stream, LaunchCtx* ctx) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return WAN_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_dev_mu);
  DevInfo& d = g_dev[dev];
  if (!d.status) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_wan_status) != cudaSuccess) return WAN_ERR_CUDA;
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return WAN_ERR_CUDA;
    d.status = static_cast<int*>(p);
    d.num_sms = sms;
  }
  ctx->stream = stream;
  ctx->dev_status = d.status;
  ctx->num_sms = d.num_sms;
  return WAN_OK;
}

int set_smem_limit_once(const void* func, int bytes, std::atomic<unsigned long long>* done) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return WAN_ERR_CUDA;
  const unsigned long long bit = 1ull << dev;
  if (done->load(std::memory_order_acquire) & bit) return WAN_OK;
  if (cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess)
    return WAN_ERR_CUDA;
  done->fetch_or(bit, std::memory_order_release);  // racing threads set the same value
  return WAN_OK;
}

// ------------------------------------------------------------------ tensor maps
static PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
static std::once_flag g_encode_once;

static PFN_cuTensorMapEncodeTiled_v12000 encoder() {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  return g_encode;
}

static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

int make_tmap_2d(CUtensorMap* m, const void* base, CUtensorMapDataType dt, int elem_bytes, uint64_t d0, uint64_t d1,
                 uint64_t stride1_bytes, uint32_t box0, uint32_t box1) {
  auto enc = encoder();
  if (!enc) return WAN_ERR_CUDA;
  if (!aligned16(base) || stride1_bytes % 16 != 0 || box0 * (uint32_t)elem_bytes != 128) return WAN_ERR_UNSUPPORTED;
  cuuint64_t dims[2] = {d0, d1};
  cuuint64_t strides[1] = {stride1_bytes};
  cuuint32_t box[2] = {box0, box1};
  cuuint32_t es[2] = {1, 1};
  CUresult r = enc(m, dt, 2, const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? WAN_OK : WAN_ERR_UNSUPPORTED;
}

int make_tmap_3d(CUtensorMap* m, const void* base, CUtensorMapDataType dt, int elem_bytes, uint64_t d0, uint64_t d1,
                 uint64_t d2, uint64_t stride1_bytes, uint64_t stride2_bytes, uint32_t box0, uint32_t box1) {
  auto enc = encoder();
  if (!enc) return WAN_ERR_CUDA;
  if (!aligned16(base) || stride1_bytes % 16 != 0 || stride2_bytes % 16 != 0 || box0 * (uint32_t)elem_bytes != 128)
    return WAN_ERR_UNSUPPORTED;
  cuuint64_t dims[3] = {d0, d1, d2};
  cuuint64_t strides[2] = {stride1_bytes, stride2_bytes};
  cuuint32_t box[3] = {box0, box1, 1};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = enc(m, dt, 3, const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? WAN_OK : WAN_ERR_UNSUPPORTED;
}

// ------------------------------------------------------------------ helpers
#define WAN_TRY(expr)          \
  do {                         \
    const int _st = (expr);    \
    if (_st != WAN_OK) return _st; \
  } while (0)

static inline long long round_up(long long v, long long a) { return (v + a - 1) / a * a; }

struct Bump {
  uint8_t* base;
  size_t off = 0;
  explicit Bump(void* b) : base(static_cast<uint8_t*>(b)) {}
  template <typename T>
  T* take(size_t count, size_t elem = sizeof(T)) {
    off = (size_t)round_up((long long)off, 1024);
    T* p = base ? reinterpret_cast<T*>(base + off) : nullptr;
    off += count * elem;
    return p;
  }
};

static EpiParams epi_base(int kind, int M, int N, int rows_per_batch, const void* bias, int f32) {
  EpiParams e;
  memset(&e, 0, sizeof(e));
  e.kind = kind;
  e.M = M;
  e.N = N;
  e.rows_per_batch = rows_per_batch > 0 ? rows_per_batch : (M > 0 ? M : 1);
  e.bias = bias;
  e.bias_f32 = f32;
  return e;
}

// y = A W^T (+ epilogue) in the call's dtype (fp32 SIMT, or 16-bit tensor cores with A
// and W both bf16, or both fp16 when ab_f16).
static int proj(const LaunchCtx& c, int f32, const void* A, long long lda, int a_cols, const void* W, long long ldw,
                int w_cols, int M, int N, int K, int kb_period, const EpiParams& ep, const char* tag,
                bool ab_f16 = false) {
  if (f32) return gemm_f32(c, static_cast<const float*>(A), lda, static_cast<const float*>(W), ldw, M, N, K, ep, tag);
  return gemm_bf16(c, A, lda, a_cols, W, ldw, w_cols, M, N, K, kb_period, ep, tag, ab_f16);
}

static int attend(const LaunchCtx& c, int f32, const AttnArgs& a) {
  return f32 ? attention_f32(c, a) : attention_bf16(c, a);
}

static int check_dtype(int dtype) { return (dtype == WAN_BF16 || dtype == WAN_F32) ? WAN_OK : WAN_ERR_INVALID_ARG; }

// q/k storage of an attention call: the call's dtype, or fp16 alongside bf16 v/o.
static int check_qk_dtype(int dtype, int qk_dtype) {
  if (qk_dtype == dtype) return WAN_OK;
  if (dtype == WAN_BF16 && qk_dtype == WAN_F16) return WAN_OK;
  return (qk_dtype == WAN_BF16 || qk_dtype == WAN_F32 || qk_dtype == WAN_F16) ? WAN_ERR_UNSUPPORTED
                                                                               : WAN_ERR_INVALID_ARG;
}

// ------------------------------------------------------------------ patchify
static long long patch_kpad(int C, int f32) { return f32 ? 4LL * C : round_up(4LL * C, 64); }

static size_t patch_ws_bytes(int B, int C, int F, int H, int W, int f32) {
  const long long M = (long long)B * F * (H / 2) * (W / 2);
  return f32 ? (size_t)(M * 4 * C * 4) : (size_t)(M * 2 * patch_kpad(C, 0) * 2);
}

static int patchify_impl(const LaunchCtx& c, const float* latent, long long lat_bstride, const void* w, const void* b,
                         float* x, int B, int C, int F, int H, int W, int D, int f32, void* A) {
  const int L = F * (H / 2) * (W / 2);
  const int M = B * L;
  const long long kpad = patch_kpad(C, f32);
  WAN_TRY(launch_patch_gather(c, latent, lat_bstride, A, f32, B, C, F, H, W, (int)kpad));
  EpiParams ep = epi_base(EPI_STORE, M, D, L, b, f32);
  ep.out = x;
  ep.ldo = D;
  ep.out_type = OUT_F32;
  if (f32) return proj(c, 1, A, 4LL * C, 4 * C, w, 4LL * C, 4 * C, M, D, 4 * C, 0, ep, "gemm_patchify");
  return proj(c, 0, A, 2 * kpad, (int)(2 * kpad), w, 4LL * C, 4 * C, M, D, (int)(2 * kpad), (int)(kpad / 64), ep,
              "gemm_patchify");
}

// ------------------------------------------------------------------ forward workspace plan
struct FwdWs {
  float* x;
  void *y, *qkv, *o, *qc, *kvc, *kvci, *h, *patchA;
  float *tsin, *h1, *e, *e0, *hm, *mods;
  float* rope;  // RoPE pair frequencies [head_dim / 2]
  // 8-bit variant: LN output codes + row scales; attention operands (see Attn8Operands)
  uint8_t *y8, *q8, *k8, *v8t;
  float *sy, *sq, *sk, *sv;
  unsigned int* vamax;
  size_t bytes;
};

static FwdWs plan_forward(const wan_dit_config* cfg, void* ws) {
  const int f32 = cfg->dtype == WAN_F32;
  const size_t es = f32 ? 4 : 2;
  const long long B = cfg->batch, D = cfg->dim, hd = cfg->head_dim;
  const long long L = (long long)cfg->frames * (cfg->height / 2) * (cfg->width / 2);
  const long long M = B * L;
  Bump bp(ws);
  FwdWs w;
  w.x = bp.take<float>(M * D);
  w.y = bp.take<uint8_t>(M * D * es);
  w.qkv = bp.take<uint8_t>(M * 3 * D * es);  // rows q | k | v
  w.o = bp.take<uint8_t>(M * D * es);
  w.qc = bp.take<uint8_t>(M * D * es);
  w.kvc = bp.take<uint8_t>(B * cfg->text_len * 2 * D * es);  // rows k | v
  w.kvci = cfg->img_len ? bp.take<uint8_t>(B * cfg->img_len * 2 * D * es) : nullptr;
  w.h = bp.take<uint8_t>(M * (long long)cfg->ffn * es);
  w.patchA = bp.take<uint8_t>(patch_ws_bytes((int)B, cfg->c_in, cfg->frames, cfg->height, cfg->width, f32));
  w.tsin = bp.take<float>(B * cfg->freq_dim);
  w.h1 = bp.take<float>(B * D);
  w.e = bp.take<float>(B * D);
  w.e0 = bp.take<float>(B * 6 * D);
  w.hm = bp.take<float>(B * 2 * D);
  w.mods = bp.take<float>((long long)cfg->blocks * B * 6 * D);
  w.rope = bp.take<float>((size_t)hd / 2);
  w.y8 = w.q8 = w.k8 = w.v8t = nullptr;
  w.sy = w.sq = w.sk = w.sv = nullptr;
  w.vamax = nullptr;
  if (cfg->fp8 & 2) {
    w.y8 = bp.take<uint8_t>(M * D);
    w.sy = bp.take<float>(M);
  }
  if (cfg->fp8 & 1) {
    const long long H = cfg->heads, nkb = (L + 127) / 128, Lp = round_up(L, 16);
    w.q8 = bp.take<uint8_t>(M * D);
    w.k8 = bp.take<uint8_t>(M * D);
    w.v8t = bp.take<uint8_t>(B * H * hd * Lp);
    w.sq = bp.take<float>(M * H);
    w.sk = bp.take<float>(B * H * nkb);
    w.sv = bp.take<float>(B * H * hd);
    w.vamax = bp.take<unsigned int>(B * H * hd);
  }
  w.bytes = (size_t)round_up((long long)bp.off, 1024);
  return w;
}

// Cross-attention keys/values of every block for a fixed context (the text and image
// contexts do not depend on t, so a sampler computes them once): per block, text rows
// [B*Lt, 2D] (k | v) then image rows [B*Li, 2D].
static size_t ctx_cache_block_bytes(const wan_dit_config* cfg) {
  const size_t es = cfg->dtype == WAN_F32 ? 4 : 2;
  return (size_t)round_up((long long)cfg->batch * (cfg->text_len + cfg->img_len) * 2 * cfg->dim * es, 1024);
}
static size_t ctx_cache_bytes(const wan_dit_config* cfg) { return ctx_cache_block_bytes(cfg) * cfg->blocks; }

static int validate_cfg(const wan_dit_config* cfg) {
  if (!cfg) return WAN_ERR_INVALID_ARG;
  WAN_TRY(check_dtype(cfg->dtype));
  if (cfg->batch <= 0 || cfg->c_in <= 0 || cfg->c_out <= 0 || cfg->frames <= 0 || cfg->height <= 0 ||
      cfg->width <= 0 || cfg->dim <= 0 || cfg->heads <= 0 || cfg->head_dim <= 0 || cfg->ffn <= 0 ||
      cfg->blocks <= 0 || cfg->text_len <= 0 || cfg->img_len < 0 || cfg->freq_dim <= 0 || cfg->freq_dim % 2)
    return WAN_ERR_INVALID_ARG;
  if (cfg->height % 2 || cfg->width % 2 || cfg->heads * cfg->head_dim != cfg->dim) return WAN_ERR_INVALID_ARG;
  if (cfg->dim % 32 || cfg->ffn % 32 || cfg->c_out * 4 % 32 || cfg->dim > 8192) return WAN_ERR_UNSUPPORTED;
  if (cfg->dtype == WAN_BF16 && cfg->head_dim != 64 && cfg->head_dim != 128) return WAN_ERR_UNSUPPORTED;
  if (cfg->dtype == WAN_F32 && (cfg->head_dim > 128 || cfg->head_dim % 2)) return WAN_ERR_UNSUPPORTED;
  if (cfg->freq_dim % 8) return WAN_ERR_UNSUPPORTED;
  if (cfg->fp8 < 0 || cfg->fp8 > 3) return WAN_ERR_INVALID_ARG;
  if (cfg->fp8 && (cfg->dtype != WAN_BF16 || cfg->head_dim != 128)) return WAN_ERR_UNSUPPORTED;
  return WAN_OK;
}

static int validate_weights(const wan_dit_config* cfg, const wan_dit_weights* w) {
  if (!w || !w->blocks) return WAN_ERR_INVALID_ARG;
  const void* g[] = {w->patch_w, w->patch_b, w->t1_w, w->t1_b, w->t2_w, w->t2_b, w->m_w,
                     w->m_b,     w->hm_w,    w->hm_b, w->head_w, w->head_b};
  for (const void* p : g)
    if (!p || !aligned16(p)) return WAN_ERR_INVALID_ARG;
  for (int i = 0; i < cfg->blocks; ++i) {
    const wan_block_weights& b = w->blocks[i];
    const void* q[] = {b.mod, b.qkv_w, b.qkv_b, b.o_w, b.o_b, b.cq_w, b.cq_b, b.ckv_w,
                       b.ckv_b, b.co_w, b.co_b, b.f1_w, b.f1_b, b.f2_w, b.f2_b};
    for (const void* p : q)
      if (!p || !aligned16(p)) return WAN_ERR_INVALID_ARG;
    if (cfg->img_len && (!b.ckvi_w || !b.ckvi_b)) return WAN_ERR_INVALID_ARG;
    if (cfg->qk_norm && (!b.norm_q_w || !b.norm_k_w || !aligned16(b.norm_q_w) || !aligned16(b.norm_k_w)))
      return WAN_ERR_INVALID_ARG;
    if (cfg->fp8 & 2) {
      const void* f[] = {b.qkv_w8, b.qkv_ws, b.f1_w8, b.f1_ws};
      for (const void* p : f)
        if (!p || !aligned16(p)) return WAN_ERR_INVALID_ARG;
    }
  }
  return WAN_OK;
}

// s = sinusoid(t); e = t2(SiLU(t1(s))); e0 = m(SiLU(e)); hm = hm(SiLU(e)).
static int time_embed_impl(const LaunchCtx& c, const wan_dit_config* cfg, const wan_dit_weights* w, const float* t,
                           int t_stride, float* tsin, float* h1, float* e, float* e0, float* hm) {
  const int f32 = cfg->dtype == WAN_F32;
  const int B = cfg->batch, D = cfg->dim;
  WAN_TRY(launch_sinusoid(c, t, t_stride, tsin, B, cfg->freq_dim));
  WAN_TRY(launch_small_linear(c, tsin, w->t1_w, w->t1_b, f32, h1, B, D, cfg->freq_dim, 0, 1));
  WAN_TRY(launch_small_linear(c, h1, w->t2_w, w->t2_b, f32, e, B, D, D, 0, 0));
  WAN_TRY(launch_small_linear(c, e, w->m_w, w->m_b, f32, e0, B, 6 * D, D, 1, 0));
  return launch_small_linear(c, e, w->hm_w, w->hm_b, f32, hm, B, 2 * D, D, 1, 0);
}

// Cross-attention keys/values of block i into kv_txt [B*Lt, 2D] and kv_img [B*Li, 2D].
static int cross_kv_impl(const LaunchCtx& c, const wan_dit_config* cfg, const wan_block_weights& bw,
                         const void* ctx_txt, const void* ctx_img, void* kv_txt, void* kv_img) {
  const int f32 = cfg->dtype == WAN_F32;
  const int B = cfg->batch, D = cfg->dim;
  for (int seg = 0; seg < (cfg->img_len ? 2 : 1); ++seg) {
    const int Lk = seg ? cfg->img_len : cfg->text_len;
    EpiParams ep = epi_base(EPI_QKV, B * Lk, 2 * D, Lk, seg ? bw.ckvi_b : bw.ckv_b, f32);
    ep.out = seg ? kv_img : kv_txt;
    ep.ldo = 2LL * D;
    ep.out_type = f32 ? OUT_F32 : OUT_BF16;
    ep.n_rot = 0;
    ep.n_f16 = f32 ? 0 : 2 * D;  // k and v in fp16: the cross-attention sub-layer computes in fp16
    ep.head_dim = cfg->head_dim;
    WAN_TRY(proj(c, f32, seg ? ctx_img : ctx_txt, D, D, seg ? bw.ckvi_w : bw.ckv_w, D, D, B * Lk, 2 * D, D, 0, ep,
                 "gemm_cross_kv"));
  }
  return WAN_OK;
}

// kv_cache: NULL (each block projects its cross-attention keys/values from the context),
// or a filled cache of ctx_cache_bytes(cfg) for this context (then no context projection
// runs).
static int dit_forward_impl(const wan_dit_config* cfg, const wan_dit_weights* w, const float* latent,
                            long long lat_bstride, const float* t, int t_stride, const void* ctx_txt,
                            const int* txt_lens, const void* ctx_img, const uint8_t* kv_cache, float* v_out,
                            void* ws, size_t ws_bytes, cudaStream_t stream) {
  WAN_TRY(validate_cfg(cfg));
  WAN_TRY(validate_weights(cfg, w));
  if (!latent || !t || !ctx_txt || !v_out || (cfg->img_len && !ctx_img)) return WAN_ERR_INVALID_ARG;
  if (!aligned16(latent) || !aligned16(ctx_txt) || !aligned16(v_out) || (ctx_img && !aligned16(ctx_img)))
    return WAN_ERR_UNSUPPORTED;
  FwdWs W = plan_forward(cfg, nullptr);
  if (!ws || ws_bytes < W.bytes || (reinterpret_cast<uintptr_t>(ws) & 1023)) return WAN_ERR_WORKSPACE;
  W = plan_forward(cfg, ws);
  LaunchCtx c;
  WAN_TRY(launch_ctx(stream, &c));

  const int f32 = cfg->dtype == WAN_F32;
  const int B = cfg->batch, D = cfg->dim, H = cfg->heads, hd = cfg->head_dim, Fh = cfg->ffn;
  const int Lt = cfg->text_len, Li = cfg->img_len;
  const int Fg = cfg->frames, Hg = cfg->height / 2, Wg = cfg->width / 2;
  const int L = Fg * Hg * Wg;
  const int M = B * L;

  // 3D RoPE table and the shared time embedding -> six modulation vectors per block.
  WAN_TRY(launch_rope_table(c, W.rope, hd, cfg->theta));
  const RopeGeom rg = rope_geom(W.rope, Fg, Hg, Wg, hd);
  WAN_TRY(time_embed_impl(c, cfg, w, t, t_stride, W.tsin, W.h1, W.e, W.e0, W.hm));
  {
    std::vector<const void*> mp(cfg->blocks);
    for (int i = 0; i < cfg->blocks; ++i) mp[i] = w->blocks[i].mod;
    WAN_TRY(launch_block_mods(c, W.e0, mp.data(), cfg->blocks, f32, W.mods, B, D));
  }

  WAN_TRY(patchify_impl(c, latent, lat_bstride, w->patch_w, w->patch_b, W.x, B, cfg->c_in, cfg->frames,
                        cfg->height, cfg->width, D, f32, W.patchA));

  for (int i = 0; i < cfg->blocks; ++i) {
    const wan_block_weights& bw = w->blocks[i];
    const float* mod = W.mods + (long long)i * B * 6 * D;  // [B][6][D]

    // --- self-attention: y = LN(x)(1+sc1)+sh1; q,k (RoPE), v; attention; x += g1 (o Wo^T + bo)
    const bool fp8_gemm = (cfg->fp8 & 2) != 0, fp8_attn = (cfg->fp8 & 1) != 0;
    if (fp8_gemm)
      WAN_TRY(launch_ln_mod_e4m3(c, W.x, mod + 0 * D, mod + 1 * D, 6LL * D, W.y8, W.sy, M, L, D, cfg->eps));
    else
      WAN_TRY(launch_ln_mod(c, W.x, mod + 0 * D, mod + 1 * D, 6LL * D, W.y, f32 ? OUT_F32 : OUT_BF16, M, L, D, cfg->eps));
    {
      EpiParams ep = epi_base(EPI_QKV, M, 3 * D, L, bw.qkv_b, f32);
      ep.out = W.qkv;
      ep.ldo = 3LL * D;
      ep.out_type = f32 ? OUT_F32 : OUT_BF16;
      ep.n_rot = cfg->qk_norm ? 0 : 2 * D;  // with q/k RMSNorm, RoPE follows the norm below
      ep.n_f16 = f32 ? 0 : 2 * D;           // q, k feed the QK^T MMA in fp16
      ep.head_dim = hd;
      ep.rope = rg;
      if (fp8_gemm)
        WAN_TRY(gemm_e4m3(c, W.y8, D, D, W.sy, static_cast<const uint8_t*>(bw.qkv_w8), D, D, bw.qkv_ws, M, 3 * D,
                          D, ep, "gemm_qkv_rope_e4m3"));
      else
        WAN_TRY(proj(c, f32, W.y, D, D, bw.qkv_w, D, D, M, 3 * D, D, 0, ep, "gemm_qkv_rope"));
      if (cfg->qk_norm)
        WAN_TRY(launch_qk_rmsnorm_rope(c, W.qkv, 3LL * D, bw.norm_q_w, bw.norm_k_w, rg, M, L, D, hd, cfg->eps, f32));
    }
    if (fp8_attn) {
      Attn8Operands qa;
      memset(&qa, 0, sizeof(qa));
      qa.q = W.qkv; qa.ldq = 3LL * D; qa.q_col = 0;
      qa.k = W.qkv; qa.ldk = 3LL * D; qa.k_col = D;
      qa.v = W.qkv; qa.ldv = 3LL * D; qa.v_col = 2 * D;
      qa.qk_type = OUT_F16; qa.v_type = OUT_BF16;
      qa.B = B; qa.L = L; qa.H = H; qa.head_dim = hd;
      qa.nkb = (L + 127) / 128; qa.Lp = (int)round_up(L, 16);
      qa.q8 = W.q8; qa.sq = W.sq; qa.k8 = W.k8; qa.sk = W.sk; qa.v8t = W.v8t; qa.sv = W.sv; qa.v_amax = W.vamax;
      WAN_TRY(quant_attn_e4m3(c, qa));
      Attn8Args a;
      memset(&a, 0, sizeof(a));
      a.q8 = W.q8; a.sq = W.sq; a.k8 = W.k8; a.sk = W.sk; a.v8t = W.v8t; a.sv = W.sv;
      a.o = W.o; a.ldo = D; a.o_col = 0;
      a.B = B; a.L = L; a.H = H; a.head_dim = hd; a.Lp = qa.Lp;
      a.tag = "attn_self_e4m3";
      WAN_TRY(attention_e4m3(c, a));
    } else {
      AttnArgs a;
      memset(&a, 0, sizeof(a));
      a.q = W.qkv; a.ldq = 3LL * D; a.q_row_len = 3 * D; a.q_col = 0;
      a.k = W.qkv; a.ldk = 3LL * D; a.k_row_len = 3 * D; a.k_col = D;
      a.v = W.qkv; a.ldv = 3LL * D; a.v_row_len = 3 * D; a.v_col = 2 * D;
      a.o = W.o; a.ldo = D; a.o_col = 0;
      a.B = B; a.Lq = L; a.Lkv = L; a.H = H; a.head_dim = hd;
      a.tag = "attn_self";
      a.qk_f16 = !f32;
      WAN_TRY(attend(c, f32, a));
    }
    {
      EpiParams ep = epi_base(EPI_RESID, M, D, L, bw.o_b, f32);
      ep.resid = W.x;
      ep.ldr = D;
      ep.gate = mod + 2 * D;
      ep.ld_gate = 6LL * D;
      WAN_TRY(proj(c, f32, W.o, D, D, bw.o_w, D, D, M, D, D, 0, ep, "gemm_o_gate"));
    }

    // --- cross-attention: q = LN(x) Wq^T; k,v from the context; x += o Wo^T + bo.
    // 16-bit path: the whole sub-layer runs in fp16 storage (LN output, q, k, v, the
    // probabilities, o, and the weights cq_w / co_w): its values are bounded (an
    // unmodulated LN row has norm sqrt(D); probabilities stay below 2^15), and fp16's 3
    // extra mantissa bits cut the error of the peaked softmaxes of wide models.
    WAN_TRY(launch_ln_mod(c, W.x, nullptr, nullptr, 0, W.y, f32 ? OUT_F32 : OUT_F16, M, L, D, cfg->eps));
    {
      EpiParams ep = epi_base(EPI_STORE, M, D, L, bw.cq_b, f32);
      ep.out = W.qc;
      ep.ldo = D;
      ep.out_type = f32 ? OUT_F32 : OUT_F16;
      WAN_TRY(proj(c, f32, W.y, D, D, bw.cq_w, D, D, M, D, D, 0, ep, "gemm_cross_q", true));
    }
    void* kv_txt = W.kvc;
    void* kv_img = W.kvci;
    if (kv_cache) {
      kv_txt = const_cast<uint8_t*>(kv_cache) + (size_t)i * ctx_cache_block_bytes(cfg);
      kv_img = static_cast<uint8_t*>(kv_txt) + (size_t)B * Lt * 2 * D * (f32 ? 4 : 2);
    } else {
      WAN_TRY(cross_kv_impl(c, cfg, bw, ctx_txt, ctx_img, kv_txt, kv_img));
    }
    if (f32) {
      for (int seg = 0; seg < (Li ? 2 : 1); ++seg) {
        const int Lk = seg ? Li : Lt;
        void* kv = seg ? kv_img : kv_txt;
        AttnArgs a;
        memset(&a, 0, sizeof(a));
        a.q = W.qc; a.ldq = D; a.q_row_len = D; a.q_col = 0;
        a.k = kv; a.ldk = 2LL * D; a.k_row_len = 2 * D; a.k_col = 0;
        a.v = kv; a.ldv = 2LL * D; a.v_row_len = 2 * D; a.v_col = D;
        a.o = W.o; a.ldo = D; a.o_col = 0;
        a.B = B; a.Lq = L; a.Lkv = Lk; a.H = H; a.head_dim = hd;
        a.accumulate = seg;
        a.kv_lens = seg ? nullptr : txt_lens;  // text keys may be padded; the image tokens are all valid
        a.tag = "attn_cross";
        WAN_TRY(attention_f32(c, a));
      }
    } else {
      CrossArgs a;
      memset(&a, 0, sizeof(a));
      a.q = W.qc; a.ldq = D; a.q_row_len = D; a.q_col = 0;
      a.kt = kv_txt; a.vt = kv_txt; a.ldkt = a.ldvt = 2LL * D; a.kt_row_len = a.vt_row_len = 2 * D;
      a.kt_col = 0; a.vt_col = D;
      if (Li) {
        a.ki = kv_img; a.vi = kv_img; a.ldki = a.ldvi = 2LL * D; a.ki_row_len = a.vi_row_len = 2 * D;
        a.ki_col = 0; a.vi_col = D;
      }
      a.o = W.o; a.ldo = D; a.o_col = 0;
      a.B = B; a.L = L; a.Lt = Lt; a.Li = Li; a.H = H; a.head_dim = hd;
      a.kt_lens = txt_lens;  // text keys may be padded; the image tokens are all valid
      a.qk_f16 = 1;
      a.pv_f16 = 1;
      a.tag = "attn_cross";
      WAN_TRY(cross_attention_tc(c, a));
    }
    {
      EpiParams ep = epi_base(EPI_RESID, M, D, L, bw.co_b, f32);
      ep.resid = W.x;
      ep.ldr = D;
      WAN_TRY(proj(c, f32, W.o, D, D, bw.co_w, D, D, M, D, D, 0, ep, "gemm_cross_o", true));
    }

    // --- FFN: y = LN(x)(1+sc2)+sh2; h = GELU(y W1^T + b1); x += g2 (h W2^T + b2)
    if (fp8_gemm)
      WAN_TRY(launch_ln_mod_e4m3(c, W.x, mod + 3 * D, mod + 4 * D, 6LL * D, W.y8, W.sy, M, L, D, cfg->eps));
    else
      WAN_TRY(launch_ln_mod(c, W.x, mod + 3 * D, mod + 4 * D, 6LL * D, W.y, f32 ? OUT_F32 : OUT_BF16, M, L, D, cfg->eps));
    {
      EpiParams ep = epi_base(cfg->gelu_tanh ? EPI_GELU_TANH : EPI_GELU, M, Fh, L, bw.f1_b, f32);
      ep.out = W.h;
      ep.ldo = Fh;
      ep.out_type = f32 ? OUT_F32 : OUT_BF16;
      if (fp8_gemm)
        WAN_TRY(gemm_e4m3(c, W.y8, D, D, W.sy, static_cast<const uint8_t*>(bw.f1_w8), D, D, bw.f1_ws, M, Fh, D,
                          ep, "gemm_ffn1_gelu_e4m3"));
      else
        WAN_TRY(proj(c, f32, W.y, D, D, bw.f1_w, D, D, M, Fh, D, 0, ep, "gemm_ffn1_gelu"));
    }
    {
      EpiParams ep = epi_base(EPI_RESID, M, D, L, bw.f2_b, f32);
      ep.resid = W.x;
      ep.ldr = D;
      ep.gate = mod + 5 * D;
      ep.ld_gate = 6LL * D;
      WAN_TRY(proj(c, f32, W.h, Fh, Fh, bw.f2_w, Fh, Fh, M, D, Fh, 0, ep, "gemm_ffn2_gate"));
    }
  }

  // head: LN(x)(1+sc_h)+sh_h -> Linear D -> c_out*4 -> depatchify
  WAN_TRY(launch_ln_mod(c, W.x, W.hm, W.hm + D, 2LL * D, W.y, f32 ? OUT_F32 : OUT_BF16, M, L, D, cfg->eps));
  {
    EpiParams ep = epi_base(EPI_HEAD, M, cfg->c_out * 4, L, w->head_b, f32);
    ep.vout = v_out;
    ep.C = cfg->c_out;
    ep.F = cfg->frames;
    ep.H = cfg->height;
    ep.W = cfg->width;
    WAN_TRY(proj(c, f32, W.y, D, D, w->head_w, D, D, M, cfg->c_out * 4, D, 0, ep, "gemm_head"));
  }
  return WAN_OK;
}

}  // namespace wan

using namespace wan;

// ====================================================================== C ABI
extern "C" {

const char* wan_status_string(int status) {
  switch (status) {
    case WAN_OK: return "ok";
    case WAN_ERR_INVALID_ARG: return "invalid argument";
    case WAN_ERR_UNSUPPORTED: return "unsupported shape, alignment or dtype";
    case WAN_ERR_CUDA: return "CUDA runtime error";
    case WAN_ERR_TIMEOUT: return "device pipeline wait timed out";
    case WAN_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    default: return "unknown status";
  }
}

int wan_sync_status(wan_stream_t stream) {
  LaunchCtx c;
  WAN_TRY(launch_ctx(stream, &c));
  if (cudaStreamSynchronize(stream) != cudaSuccess) return WAN_ERR_CUDA;
  int v = 0;
  if (cudaMemcpy(&v, c.dev_status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return WAN_ERR_CUDA;
  if (v != 0) {
    const int zero = 0;
    cudaMemcpy(c.dev_status, &zero, sizeof(int), cudaMemcpyHostToDevice);
    return WAN_ERR_TIMEOUT;
  }
  return WAN_OK;
}

long long wan_launch_count(void) { return g_launches.load(); }

int wan_watchdog_selftest(int limit_ms, wan_stream_t stream) {
  if (limit_ms < 1 || limit_ms > 1000) return WAN_ERR_INVALID_ARG;
  LaunchCtx c;
  WAN_TRY(launch_ctx(stream, &c));
  return launch_watchdog_selftest(c, (unsigned long long)limit_ms * 1000000ull);
}

size_t wan_patchify_workspace_size(int B, int C, int F, int H, int W, int dtype) {
  if (B <= 0 || C <= 0 || F <= 0 || H <= 0 || W <= 0) return 0;
  return patch_ws_bytes(B, C, F, H, W, dtype == WAN_F32);
}

int wan_patchify(const float* latent, const void* w, const void* b, float* x, int B, int C, int F, int H, int W,
                 int D, int dtype, void* ws, size_t ws_bytes, wan_stream_t stream) {
  WAN_TRY(check_dtype(dtype));
  if (!latent || !w || !b || !x || B <= 0 || C <= 0 || F <= 0 || H <= 0 || W <= 0 || D <= 0 || H % 2 || W % 2)
    return WAN_ERR_INVALID_ARG;
  if (D % 32 || !aligned16(latent) || !aligned16(w) || !aligned16(b) || !aligned16(x)) return WAN_ERR_UNSUPPORTED;
  if (!ws || ws_bytes < patch_ws_bytes(B, C, F, H, W, dtype == WAN_F32) || !aligned16(ws)) return WAN_ERR_WORKSPACE;
  LaunchCtx c;
  WAN_TRY(launch_ctx(stream, &c));
  return patchify_impl(c, latent, (long long)C * F * H * W, w, b, x, B, C, F, H, W, D, dtype == WAN_F32, ws);
}

int wan_adaln_modulate(const float* x, const float* shift, const float* scale, void* y, int B, int L, int D,
                       float eps, int dtype, wan_stream_t stream) {
  if (dtype != WAN_F16) WAN_TRY(check_dtype(dtype));
  if (!x || !y || B <= 0 || L <= 0 || D <= 0 || (!shift) != (!scale)) return WAN_ERR_INVALID_ARG;
  if (D % 4 || D > 8192 || !aligned16(x) || !aligned16(y) || (shift && (!aligned16(shift) || !aligned16(scale))))
    return WAN_ERR_UNSUPPORTED;
  LaunchCtx c;
  WAN_TRY(launch_ctx(stream, &c));
  return launch_ln_mod(c, x, shift, scale, D, y, dtype == WAN_F32 ? OUT_F32 : (dtype == WAN_F16 ? OUT_F16 : OUT_BF16),
                       B * L, L, D, eps);
}

size_t wan_attn_workspace_size(int B, int L, int H, int d, int dtype) {
  if (B <= 0 || L <= 0 || H <= 0 || d <= 0) return 0;
  const size_t es = dtype == WAN_F32 ? 4 : 2;
  Bump bp(nullptr);
  bp.take<float>((size_t)d / 2);   // RoPE pair frequencies
  bp.take<uint8_t>((size_t)B * L * H * d * es);  // rotated q
  bp.take<uint8_t>((size_t)B * L * H * d * es);  // rotated k
  return (size_t)round_up((long long)bp.off, 1024);
}

int wan_attn_rope3d(const void* q, const void* k, const void* v, void* o, const int* kv_lens, int B, int L, int H,
                    int d, int Fg, int Hg, int Wg, float theta, int apply_rope, int dtype, int qk_dtype, void* ws,
                    size_t ws_bytes, wan_stream_t stream) {
  WAN_TRY(check_dtype(dtype));
  WAN_TRY(check_qk_dtype(dtype, qk_dtype));
  const int f32 = dtype == WAN_F32;
  if (!q || !k || !v || !o || B <= 0 || L <= 0 || H <= 0 || d <= 0) return WAN_ERR_INVALID_ARG;
  if (apply_rope && (Fg <= 0 || Hg <= 0 || Wg <= 0 || (long long)Fg * Hg * Wg != L)) return WAN_ERR_INVALID_ARG;
  if ((!f32 && d != 64 && d != 128) || (f32 && (d > 128 || d % 2))) return WAN_ERR_UNSUPPORTED;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o)) return WAN_ERR_UNSUPPORTED;
  if (apply_rope && (!ws || ws_bytes < wan_attn_workspace_size(B, L, H, d, dtype) ||
                     (reinterpret_cast<uintptr_t>(ws) & 1023)))
    return WAN_ERR_WORKSPACE;
  LaunchCtx c;
  WAN_TRY(launch_ctx(stream, &c));
  const void* qa = q;
  const void* ka = k;
  if (apply_rope) {
    const size_t es = f32 ? 4 : 2;
    Bump bp(ws);
    float* tab = bp.take<float>((size_t)d / 2);
    void* qr = bp.take<uint8_t>((size_t)B * L * H * d * es);
    void* kr = bp.take<uint8_t>((size_t)B * L * H * d * es);
    WAN_TRY(launch_rope_table(c, tab, d, theta));
    const RopeGeom g = rope_geom(tab, Fg, Hg, Wg, d);
    const int in_type = f32 ? OUT_F32 : (qk_dtype == WAN_F16 ? OUT_F16 : OUT_BF16);
    WAN_TRY(launch_rope_apply(c, q, qr, g, B, L, H, d, in_type));
    WAN_TRY(launch_rope_apply(c, k, kr, g, B, L, H, d, in_type));
    qa = qr;
    ka = kr;
  }
  AttnArgs a;
  memset(&a, 0, sizeof(a));
  const int D = H * d;
  a.q = qa; a.ldq = D; a.q_row_len = D;
  a.k = ka; a.ldk = D; a.k_row_len = D;
  a.v = v; a.ldv = D; a.v_row_len = D;
  a.o = o; a.ldo = D;
  a.B = B; a.Lq = L; a.Lkv = L; a.H = H; a.head_dim = d;
  a.kv_lens = kv_lens;
  a.tag = "attn_self";
  a.qk_f16 = !f32 && (apply_rope || qk_dtype == WAN_F16);  // rotated q, k are written in fp16
  return attend(c, f32, a);
}

size_t wan_qkv_rope_workspace_size(int d) {
  if (d <= 0) return 0;
  return (size_t)round_up((long long)d / 2 * 4, 1024);
}

// The QKV projection of the forward with its fused epilogue: bias, 3D RoPE on q and k,
// q and k stored in fp16 (16-bit path) next to v in the call's type.
static int qkv_rope_common(const void* y, const float* sy, const void* w, const float* sw, const void* b, void* qkv,
                           int B, int L, int H, int d, int Fg, int Hg, int Wg, float theta, int dtype, bool e4m3,
                           void* ws, size_t ws_bytes, cudaStream_t stream) {
  const int f32 = dtype == WAN_F32;
  if (!y || !w || !qkv || B <= 0 || L <= 0 || H <= 0 || d <= 0 || d % 2) return WAN_ERR_INVALID_ARG;
  if (Fg <= 0 || Hg <= 0 || Wg <= 0 || (long long)Fg * Hg * Wg != L) return WAN_ERR_INVALID_ARG;
  if (e4m3 && (!sy || !sw)) return WAN_ERR_INVALID_ARG;
  const int D = H * d;
  if (D % 32 || (!f32 && d % 32) || !aligned16(y) || !aligned16(w) || !aligned16(qkv) || (b && !aligned16(b)) ||
      (sw && !aligned16(sw)))
    return WAN_ERR_UNSUPPORTED;
  if (!ws || ws_bytes < wan_qkv_rope_workspace_size(d) || !aligned16(ws)) return WAN_ERR_WORKSPACE;
  LaunchCtx c;
  WAN_TRY(launch_ctx(stream, &c));
  float* tab = static_cast<float*>(ws);
  WAN_TRY(launch_rope_table(c, tab, d, theta));
  const int M = B * L;
  EpiParams ep = epi_base(EPI_QKV, M, 3 * D, L, b, f32);
  ep.out = qkv;
  ep.ldo = 3LL * D;
  ep.out_type = f32 ? OUT_F32 : OUT_BF16;
  ep.n_rot = 2 * D;
  ep.n_f16 = f32 ? 0 : 2 * D;
  ep.head_dim = d;
  ep.rope = rope_geom(tab, Fg, Hg, Wg, d);
  if (e4m3)
    return gemm_e4m3(c, static_cast<const uint8_t*>(y), D, D, sy, static_cast<const uint8_t*>(w), D, D, sw, M, 3 * D,
                     D, ep, "gemm_qkv_rope_e4m3");
  return proj(c, f32, y, D, D, w, D, D, M, 3 * D, D, 0, ep, "gemm_qkv_rope");
}

int wan_qkv_rope(const void* y, const void* w, const void* b, void* qkv, int B, int L, int H, int d, int Fg, int Hg,
                 int Wg, float theta, int dtype, void* ws, size_t ws_bytes, wan_stream_t stream) {
  WAN_TRY(check_dtype(dtype));
  return qkv_rope_common(y, nullptr, w, nullptr, b, qkv, B, L, H, d, Fg, Hg, Wg, theta, dtype, false, ws, ws_bytes,
                         stream);
}

int wan_qkv_rope_e4m3(const void* y8, const float* sy, const void* w8, const float* sw, const void* b, void* qkv,
                      int B, int L, int H, int d, int Fg, int Hg, int Wg, float theta, void* ws, size_t ws_bytes,
                      wan_stream_t stream) {
  if ((long long)H * d % 16) return WAN_ERR_UNSUPPORTED;
  return qkv_rope_common(y8, sy, w8, sw, b, qkv, B, L, H, d, Fg, Hg, Wg, theta, WAN_BF16, true, ws, ws_bytes,
                         stream);
}

size_t wan_cross_attn_workspace_size(int B, int Lt, int Li, int H, int d, int dtype) {
  (void)B, (void)Lt, (void)Li, (void)H, (void)d, (void)dtype;
  return 0;  // the kernels read q, k and v in place
}

int wan_cross_attn(const void* q, const void* kt, const void* vt, const int* kt_lens, const void* ki, const void* vi,
                   void* o, int B, int L, int Lt, int Li, int H, int d, int dtype, int qk_dtype, void* ws,
                   size_t ws_bytes, wan_stream_t stream) {
  (void)ws, (void)ws_bytes;
  // dtype (v and o): WAN_F32 with fp32 q/k; WAN_BF16 with bf16 or fp16 q/k; WAN_F16 with fp16 q/k.
  if (dtype == WAN_F16) {
    if (qk_dtype != WAN_F16)
      return (qk_dtype == WAN_BF16 || qk_dtype == WAN_F32) ? WAN_ERR_UNSUPPORTED : WAN_ERR_INVALID_ARG;
  } else {
    WAN_TRY(check_dtype(dtype));
    WAN_TRY(check_qk_dtype(dtype, qk_dtype));
  }
  const int f32 = dtype == WAN_F32;
  if (!q || !kt || !vt || !o || B <= 0 || L <= 0 || Lt <= 0 || Li < 0 || H <= 0 || d <= 0) return WAN_ERR_INVALID_ARG;
  if (Li > 0 && (!ki || !vi)) return WAN_ERR_INVALID_ARG;
  if ((!f32 && d != 64 && d != 128) || (f32 && (d > 128 || d % 2))) return WAN_ERR_UNSUPPORTED;
  if (!aligned16(q) || !aligned16(kt) || !aligned16(vt) || !aligned16(o) || (Li && (!aligned16(ki) || !aligned16(vi))))
    return WAN_ERR_UNSUPPORTED;
  LaunchCtx c;
  WAN_TRY(launch_ctx(stream, &c));
  const int D = H * d;
  if (f32) {
    for (int seg = 0; seg < (Li ? 2 : 1); ++seg) {
      const int Lk = seg ? Li : Lt;
      AttnArgs a;
      memset(&a, 0, sizeof(a));
      a.q = q; a.ldq = D; a.q_row_len = D;
      a.k = seg ? ki : kt; a.ldk = D; a.k_row_len = D;
      a.v = seg ? vi : vt; a.ldv = D; a.v_row_len = D;
      a.o = o; a.ldo = D;
      a.B = B; a.Lq = L; a.Lkv = Lk; a.H = H; a.head_dim = d;
      a.accumulate = seg;
      a.kv_lens = seg ? nullptr : kt_lens;
      a.tag = "attn_cross";
      WAN_TRY(attention_f32(c, a));
    }
    return WAN_OK;
  }
  CrossArgs a;
  memset(&a, 0, sizeof(a));
  a.q = q; a.ldq = D; a.q_row_len = D;
  a.kt = kt; a.vt = vt; a.ldkt = a.ldvt = D; a.kt_row_len = a.vt_row_len = D;
  if (Li) {
    a.ki = ki; a.vi = vi; a.ldki = a.ldvi = D; a.ki_row_len = a.vi_row_len = D;
  }
  a.o = o; a.ldo = D;
  a.B = B; a.L = L; a.Lt = Lt; a.Li = Li; a.H = H; a.head_dim = d;
  a.kt_lens = kt_lens;
  a.qk_f16 = qk_dtype == WAN_F16;
  a.pv_f16 = dtype == WAN_F16;
  a.tag = "attn_cross";
  return cross_attention_tc(c, a);
}

int wan_ffn(const void* y, const void* w1, const void* b1, const void* w2, const void* b2, const float* gate,
            float* x_inout, void* h_ws, int B, int L, int D, int F, int dtype, wan_stream_t stream) {
  WAN_TRY(check_dtype(dtype));
  const int f32 = dtype == WAN_F32;
  if (!y || !w1 || !w2 || !x_inout || !h_ws || B <= 0 || L <= 0 || D <= 0 || F <= 0) return WAN_ERR_INVALID_ARG;
  if (D % 32 || F % 32 || !aligned16(y) || !aligned16(w1) || !aligned16(w2) || !aligned16(x_inout) ||
      !aligned16(h_ws) || (gate && !aligned16(gate)) || (b1 && !aligned16(b1)) || (b2 && !aligned16(b2)))
    return WAN_ERR_UNSUPPORTED;
  LaunchCtx c;
  WAN_TRY(launch_ctx(stream, &c));
  const int M = B * L;
  EpiParams e1 = epi_base(EPI_GELU, M, F, L, b1, f32);
  e1.out = h_ws;
  e1.ldo = F;
  e1.out_type = f32 ? OUT_F32 : OUT_BF16;
  WAN_TRY(proj(c, f32, y, D, D, w1, D, D, M, F, D, 0, e1, "gemm_ffn1_gelu"));
  EpiParams e2 = epi_base(EPI_RESID, M, D, L, b2, f32);
  e2.resid = x_inout;
  e2.ldr = D;
  e2.gate = gate;
  e2.ld_gate = D;
  return proj(c, f32, h_ws, F, F, w2, F, F, M, D, F, 0, e2, "gemm_ffn2_gate");
}

int wan_linear(const void* x, const void* w, const void* b, void* out, int M, int N, int K, int epilogue,
               const float* gate, int rows_per_gate, int dtype, int out_dtype, wan_stream_t stream) {
  if (dtype != WAN_F16) WAN_TRY(check_dtype(dtype));
  if (out_dtype != WAN_BF16 && out_dtype != WAN_F32 && out_dtype != WAN_F16) return WAN_ERR_INVALID_ARG;
  const int f32 = dtype == WAN_F32;
  if (!x || !w || !out || M <= 0 || N <= 0 || K <= 0) return WAN_ERR_INVALID_ARG;
  if (epilogue != WAN_EPI_STORE && epilogue != WAN_EPI_GELU && epilogue != WAN_EPI_RESIDUAL &&
      epilogue != WAN_EPI_GELU_TANH)
    return WAN_ERR_INVALID_ARG;
  if (gate && rows_per_gate <= 0) return WAN_ERR_INVALID_ARG;
  if (f32 && out_dtype != WAN_F32) return WAN_ERR_UNSUPPORTED;
  if (epilogue == WAN_EPI_RESIDUAL && out_dtype != WAN_F32) return WAN_ERR_UNSUPPORTED;
  if (N % 32 || K % 8 || !aligned16(x) || !aligned16(w) || !aligned16(out) || (gate && !aligned16(gate)) ||
      (b && !aligned16(b)))
    return WAN_ERR_UNSUPPORTED;
  LaunchCtx c;
  WAN_TRY(launch_ctx(stream, &c));
  const int kind = epilogue == WAN_EPI_STORE ? EPI_STORE
                   : epilogue == WAN_EPI_GELU ? EPI_GELU
                   : epilogue == WAN_EPI_GELU_TANH ? EPI_GELU_TANH
                                                   : EPI_RESID;
  EpiParams ep = epi_base(kind, M, N, gate ? rows_per_gate : M, b, f32);
  if (kind == EPI_RESID) {
    ep.resid = static_cast<float*>(out);
    ep.ldr = N;
    ep.gate = gate;
    ep.ld_gate = N;
  } else {
    ep.out = out;
    ep.ldo = N;
    ep.out_type = out_dtype == WAN_F32 ? OUT_F32 : (out_dtype == WAN_F16 ? OUT_F16 : OUT_BF16);
  }
  return proj(c, f32, x, K, K, w, K, K, M, N, K, 0, ep, "gemm_linear", dtype == WAN_F16);
}

static int out_type_of(int dtype) {
  return dtype == WAN_F32 ? OUT_F32 : (dtype == WAN_F16 ? OUT_F16 : OUT_BF16);
}

int wan_quant_rows_e4m3(const void* x, int dtype, long long ldx, int M, int K, void* x8, long long ld8, float* s,
                        wan_stream_t stream) {
  if (dtype != WAN_BF16 && dtype != WAN_F16 && dtype != WAN_F32) return WAN_ERR_INVALID_ARG;
  if (!x || !x8 || !s || M < 0 || K <= 0 || ldx < K || ld8 < K) return WAN_ERR_INVALID_ARG;
  if (K % 4 || ldx % 4 || ld8 % 4 || !aligned16(x) || (reinterpret_cast<uintptr_t>(x8) & 3)) return WAN_ERR_UNSUPPORTED;
  LaunchCtx c;
  WAN_TRY(launch_ctx(stream, &c));
  return launch_quant_rows_e4m3(c, x, out_type_of(dtype), ldx, M, K, static_cast<uint8_t*>(x8), ld8, s);
}

size_t wan_quant_attn_workspace_size(int B, int H, int d) {
  if (B <= 0 || H <= 0 || d <= 0) return 0;
  return (size_t)round_up((long long)B * H * d * 4, 1024);
}

int wan_quant_attn_e4m3(const void* q, const void* k, const void* v, int qk_dtype, int v_dtype, int B, int L, int H,
                        int d, void* q8, float* sq, void* k8, float* sk, void* v8t, float* sv, void* ws,
                        size_t ws_bytes, wan_stream_t stream) {
  if ((qk_dtype != WAN_BF16 && qk_dtype != WAN_F16) || (v_dtype != WAN_BF16 && v_dtype != WAN_F16))
    return WAN_ERR_INVALID_ARG;
  if (!q || !k || !v || !q8 || !sq || !k8 || !sk || !v8t || !sv || B <= 0 || L <= 0 || H <= 0)
    return WAN_ERR_INVALID_ARG;
  if (d != 128) return WAN_ERR_UNSUPPORTED;
  const void* ptrs[] = {q, k, v, q8, k8, v8t};
  for (const void* p : ptrs)
    if (!aligned16(p)) return WAN_ERR_UNSUPPORTED;
  if (!ws || ws_bytes < wan_quant_attn_workspace_size(B, H, d) || (reinterpret_cast<uintptr_t>(ws) & 3))
    return WAN_ERR_WORKSPACE;
  LaunchCtx c;
  WAN_TRY(launch_ctx(stream, &c));
  Attn8Operands a;
  memset(&a, 0, sizeof(a));
  const int D = H * d;
  a.q = q; a.ldq = D; a.q_col = 0;
  a.k = k; a.ldk = D; a.k_col = 0;
  a.v = v; a.ldv = D; a.v_col = 0;
  a.qk_type = out_type_of(qk_dtype);
  a.v_type = out_type_of(v_dtype);
  a.B = B; a.L = L; a.H = H; a.head_dim = d;
  a.nkb = (L + 127) / 128;
  a.Lp = (int)round_up(L, 16);
  a.q8 = static_cast<uint8_t*>(q8); a.sq = sq;
  a.k8 = static_cast<uint8_t*>(k8); a.sk = sk;
  a.v8t = static_cast<uint8_t*>(v8t); a.sv = sv;
  a.v_amax = static_cast<unsigned int*>(ws);
  return quant_attn_e4m3(c, a);
}

int wan_attn_e4m3(const void* q8, const float* sq, const void* k8, const float* sk, const void* v8t, const float* sv,
                  void* o, const int* kv_lens, int B, int L, int H, int d, wan_stream_t stream) {
  if (!q8 || !sq || !k8 || !sk || !v8t || !sv || !o || B <= 0 || L <= 0 || H <= 0) return WAN_ERR_INVALID_ARG;
  if (d != 128) return WAN_ERR_UNSUPPORTED;
  if (!aligned16(q8) || !aligned16(k8) || !aligned16(v8t) || !aligned16(sv) || !aligned16(o))
    return WAN_ERR_UNSUPPORTED;
  LaunchCtx c;
  WAN_TRY(launch_ctx(stream, &c));
  Attn8Args a;
  memset(&a, 0, sizeof(a));
  a.q8 = static_cast<const uint8_t*>(q8); a.sq = sq;
  a.k8 = static_cast<const uint8_t*>(k8); a.sk = sk;
  a.v8t = static_cast<const uint8_t*>(v8t); a.sv = sv;
  a.o = o; a.ldo = (long long)H * d; a.o_col = 0;
  a.B = B; a.L = L; a.H = H; a.head_dim = d; a.Lp = (int)round_up(L, 16);
  a.kv_lens = kv_lens;
  a.tag = "attn_self_e4m3";
  return attention_e4m3(c, a);
}

int wan_linear_e4m3(const void* x8, const float* sx, const void* w8, const float* sw, const void* b, void* out, int M,
                    int N, int K, int epilogue, const float* gate, int rows_per_gate, wan_stream_t stream) {
  if (!x8 || !sx || !w8 || !sw || !out || M <= 0 || N <= 0 || K <= 0) return WAN_ERR_INVALID_ARG;
  if (epilogue != WAN_EPI_STORE && epilogue != WAN_EPI_GELU && epilogue != WAN_EPI_RESIDUAL &&
      epilogue != WAN_EPI_GELU_TANH)
    return WAN_ERR_INVALID_ARG;
  if (gate && rows_per_gate <= 0) return WAN_ERR_INVALID_ARG;
  if (N % 32 || K % 16 || !aligned16(x8) || !aligned16(w8) || !aligned16(sw) || !aligned16(out) ||
      (gate && !aligned16(gate)) || (b && !aligned16(b)))
    return WAN_ERR_UNSUPPORTED;
  LaunchCtx c;
  WAN_TRY(launch_ctx(stream, &c));
  const int kind = epilogue == WAN_EPI_STORE ? EPI_STORE
                   : epilogue == WAN_EPI_GELU ? EPI_GELU
                   : epilogue == WAN_EPI_GELU_TANH ? EPI_GELU_TANH
                                                   : EPI_RESID;
  EpiParams ep = epi_base(kind, M, N, gate ? rows_per_gate : M, b, 0);
  if (kind == EPI_RESID) {
    ep.resid = static_cast<float*>(out);
    ep.ldr = N;
    ep.gate = gate;
    ep.ld_gate = N;
  } else {
    ep.out = out;
    ep.ldo = N;
    ep.out_type = OUT_BF16;
  }
  return gemm_e4m3(c, static_cast<const uint8_t*>(x8), K, K, sx, static_cast<const uint8_t*>(w8), K, K, sw, M, N, K,
                   ep, "gemm_linear_e4m3");
}

size_t wan_text_embed_workspace_size(int B, int Lt, int D, int dtype) {
  if (B <= 0 || Lt <= 0 || D <= 0) return 0;
  return (size_t)round_up((long long)B * Lt * D * (dtype == WAN_F32 ? 4 : 2), 1024);
}

int wan_text_embed(const void* text, const void* w1, const void* b1, const void* w2, const void* b2, void* ctx, int B,
                   int Lt, int Ct, int D, int dtype, void* ws, size_t ws_bytes, wan_stream_t stream) {
  WAN_TRY(check_dtype(dtype));
  const int f32 = dtype == WAN_F32;
  if (!text || !w1 || !w2 || !ctx || B <= 0 || Lt <= 0 || Ct <= 0 || D <= 0) return WAN_ERR_INVALID_ARG;
  if (D % 32 || Ct % 8 || !aligned16(text) || !aligned16(w1) || !aligned16(w2) || !aligned16(ctx) ||
      (b1 && !aligned16(b1)) || (b2 && !aligned16(b2)))
    return WAN_ERR_UNSUPPORTED;
  if (!ws || ws_bytes < wan_text_embed_workspace_size(B, Lt, D, dtype) || !aligned16(ws)) return WAN_ERR_WORKSPACE;
  LaunchCtx c;
  WAN_TRY(launch_ctx(stream, &c));
  const int M = B * Lt;
  EpiParams e1 = epi_base(EPI_GELU, M, D, Lt, b1, f32);
  e1.out = ws;
  e1.ldo = D;
  e1.out_type = f32 ? OUT_F32 : OUT_BF16;
  WAN_TRY(proj(c, f32, text, Ct, Ct, w1, Ct, Ct, M, D, Ct, 0, e1, "gemm_text1_gelu"));
  EpiParams e2 = epi_base(EPI_STORE, M, D, Lt, b2, f32);
  e2.out = ctx;
  e2.ldo = D;
  e2.out_type = f32 ? OUT_F32 : OUT_BF16;
  return proj(c, f32, ws, D, D, w2, D, D, M, D, D, 0, e2, "gemm_text2");
}

int wan_cfg_euler_step(float* x, const void* v_cond, const void* v_uncond, long long n, float guide_scale, float dt,
                       int v_dtype, wan_stream_t stream) {
  WAN_TRY(check_dtype(v_dtype));
  if (n < 0) return WAN_ERR_INVALID_ARG;
  if (n == 0) return WAN_OK;
  if (!x || !v_cond || !v_uncond) return WAN_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(v_cond) || !aligned16(v_uncond)) return WAN_ERR_UNSUPPORTED;
  LaunchCtx c;
  WAN_TRY(launch_ctx(stream, &c));
  return launch_cfg_euler(c, x, v_cond, v_uncond, n, guide_scale, dt, nullptr, v_dtype == WAN_F32);
}

size_t wan_dit_workspace_size(const wan_dit_config* cfg) {
  if (validate_cfg(cfg) != WAN_OK) return 0;
  return plan_forward(cfg, nullptr).bytes;
}

size_t wan_time_embed_workspace_size(const wan_dit_config* cfg) {
  if (validate_cfg(cfg) != WAN_OK) return 0;
  Bump bp(nullptr);
  bp.take<float>((size_t)cfg->batch * cfg->freq_dim);
  bp.take<float>((size_t)cfg->batch * cfg->dim);
  bp.take<float>((size_t)cfg->batch * cfg->dim);
  return (size_t)round_up((long long)bp.off, 1024);
}

int wan_time_embed(const wan_dit_config* cfg, const wan_dit_weights* w, const float* t, int t_stride, float* e0,
                   float* hm, void* ws, size_t ws_bytes, wan_stream_t stream) {
  WAN_TRY(validate_cfg(cfg));
  if (!w || !w->t1_w || !w->t1_b || !w->t2_w || !w->t2_b || !w->m_w || !w->m_b || !w->hm_w || !w->hm_b || !t || !e0 ||
      !hm || t_stride < 0)
    return WAN_ERR_INVALID_ARG;
  if (!ws || ws_bytes < wan_time_embed_workspace_size(cfg) || (reinterpret_cast<uintptr_t>(ws) & 1023))
    return WAN_ERR_WORKSPACE;
  LaunchCtx c;
  WAN_TRY(launch_ctx(stream, &c));
  Bump bp(ws);
  float* tsin = bp.take<float>((size_t)cfg->batch * cfg->freq_dim);
  float* h1 = bp.take<float>((size_t)cfg->batch * cfg->dim);
  float* e = bp.take<float>((size_t)cfg->batch * cfg->dim);
  return time_embed_impl(c, cfg, w, t, t_stride, tsin, h1, e, e0, hm);
}

int wan_dit_forward(const wan_dit_config* cfg, const wan_dit_weights* w, const float* latent, int latent_broadcast,
                    const float* t, const void* ctx_txt, const int* txt_lens, const void* ctx_img, float* v_out,
                    void* ws, size_t ws_bytes, wan_stream_t stream) {
  if (!cfg) return WAN_ERR_INVALID_ARG;
  const long long bstride = latent_broadcast ? 0 : (long long)cfg->c_in * cfg->frames * cfg->height * cfg->width;
  return dit_forward_impl(cfg, w, latent, bstride, t, 1, ctx_txt, txt_lens, ctx_img, nullptr, v_out, ws, ws_bytes,
                          stream);
}

static int guided_step_impl(const wan_dit_config* cfg, const wan_dit_weights* w, float* x, const float* t_pair,
                            float guide_scale, const void* ctx_txt, const int* txt_lens, const void* ctx_img,
                            const uint8_t* kv_cache, float* v_ws, void* ws, size_t ws_bytes, cudaStream_t stream) {
  if (!cfg || !x || !t_pair || !v_ws) return WAN_ERR_INVALID_ARG;
  if (cfg->batch != 2) return WAN_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(v_ws)) return WAN_ERR_UNSUPPORTED;
  WAN_TRY(dit_forward_impl(cfg, w, x, 0, t_pair, 0, ctx_txt, txt_lens, ctx_img, kv_cache, v_ws, ws, ws_bytes, stream));
  LaunchCtx c;
  WAN_TRY(launch_ctx(stream, &c));
  const long long n = (long long)cfg->c_out * cfg->frames * cfg->height * cfg->width;
  return launch_cfg_euler(c, x, v_ws, v_ws + n, n, guide_scale, 0.f, t_pair, 1);
}

int wan_dit_guided_step(const wan_dit_config* cfg, const wan_dit_weights* w, float* x, const float* t_pair,
                        float guide_scale, const void* ctx_txt, const int* txt_lens, const void* ctx_img, float* v_ws,
                        void* ws, size_t ws_bytes, wan_stream_t stream) {
  return guided_step_impl(cfg, w, x, t_pair, guide_scale, ctx_txt, txt_lens, ctx_img, nullptr, v_ws, ws, ws_bytes,
                          stream);
}

size_t wan_sample_workspace_size(const wan_dit_config* cfg) {
  if (validate_cfg(cfg) != WAN_OK) return 0;
  return plan_forward(cfg, nullptr).bytes + ctx_cache_bytes(cfg);
}

int wan_sample(const wan_dit_config* cfg, const wan_dit_weights* w, float* x, int steps, float guide_scale,
               const void* ctx_txt, const int* txt_lens, const void* ctx_img, float* t_sched, float* v_ws, void* ws,
               size_t ws_bytes, wan_stream_t stream) {
  if (!cfg || !x || !t_sched || steps <= 0) return WAN_ERR_INVALID_ARG;
  WAN_TRY(validate_cfg(cfg));
  WAN_TRY(validate_weights(cfg, w));
  if (!ctx_txt || (cfg->img_len && !ctx_img)) return WAN_ERR_INVALID_ARG;
  const size_t fwd = plan_forward(cfg, nullptr).bytes;
  if (!ws || ws_bytes < fwd + ctx_cache_bytes(cfg) || (reinterpret_cast<uintptr_t>(ws) & 1023)) return WAN_ERR_WORKSPACE;
  LaunchCtx c;
  WAN_TRY(launch_ctx(stream, &c));
  WAN_TRY(launch_schedule(c, t_sched, steps));
  // The context is the same for every step: project every block's cross-attention keys
  // and values once, after the forward workspace, and let every step read them.
  uint8_t* cache = static_cast<uint8_t*>(ws) + fwd;
  const size_t es = cfg->dtype == WAN_F32 ? 4 : 2;
  for (int i = 0; i < cfg->blocks; ++i) {
    uint8_t* kt = cache + (size_t)i * ctx_cache_block_bytes(cfg);
    uint8_t* ki = kt + (size_t)cfg->batch * cfg->text_len * 2 * cfg->dim * es;
    WAN_TRY(cross_kv_impl(c, cfg, w->blocks[i], ctx_txt, ctx_img, kt, ki));
  }
  for (int k = 0; k < steps; ++k)
    WAN_TRY(guided_step_impl(cfg, w, x, t_sched + k, guide_scale, ctx_txt, txt_lens, ctx_img, cache, v_ws, ws, fwd,
                             stream));
  return WAN_OK;
}

int wan_profile_begin(int capacity) {
  if (capacity <= 0) return WAN_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lk(g_prof_mu);
  while (g_pool.size() < 2 * (size_t)capacity) {
    cudaEvent_t e;
    if (cudaEventCreate(&e) != cudaSuccess) return WAN_ERR_CUDA;
    g_pool.push_back(e);
  }
  g_recs.clear();
  g_cap = (size_t)capacity;
  g_prof_open = false;
  g_prof_on = true;
  return WAN_OK;
}

int wan_profile_end(const char** names, double* ms, int* counts, int max_kinds) {
  std::vector<ProfRec> recs;
  {
    std::lock_guard<std::mutex> lk(g_prof_mu);
    g_prof_on = false;
    recs.swap(g_recs);
  }
  int nk = 0;
  for (const ProfRec& r : recs) {
    if (cudaEventSynchronize(r.b) != cudaSuccess) return WAN_ERR_CUDA;
    float t = 0.f;
    if (cudaEventElapsedTime(&t, r.a, r.b) != cudaSuccess) return WAN_ERR_CUDA;
    int k = 0;
    while (k < nk && strcmp(names[k], r.kind) != 0) ++k;
    if (k == nk) {
      if (nk == max_kinds) continue;
      names[nk] = r.kind;
      ms[nk] = 0.0;
      counts[nk] = 0;
      ++nk;
    }
    ms[k] += t;
    counts[k] += 1;
  }
  return nk;
}

}  // extern "C"

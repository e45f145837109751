// Internal interface between the kernel files and the C-ABI layer (api.cu).
#pragma once

#include <atomic>

#include "epilogue.cuh"
#include "wan_common.cuh"

namespace wan {

// ------------------------------------------------------------------ launch attributes (api.cu)
// Raise `func`'s dynamic shared-memory limit to `bytes` on the current device.  The
// attribute belongs to the device that is current when it is set, so `done` keeps one
// bit per device ordinal (0..63) and the call is made once per device.
int set_smem_limit_once(const void* func, int bytes, std::atomic<unsigned long long>* done);

// ------------------------------------------------------------------ tensor maps (api.cu)
// 2D / 3D tiled maps with 128-byte swizzle and zero fill outside the tensor.
int make_tmap_2d(CUtensorMap* m, const void* base, CUtensorMapDataType dt, int elem_bytes, uint64_t d0,
                 uint64_t d1, uint64_t stride1_bytes, uint32_t box0, uint32_t box1);
int make_tmap_3d(CUtensorMap* m, const void* base, CUtensorMapDataType dt, int elem_bytes, uint64_t d0,
                 uint64_t d1, uint64_t d2, uint64_t stride1_bytes, uint64_t stride2_bytes, uint32_t box0,
                 uint32_t box1);

// ------------------------------------------------------------------ GEMMs
// 16-bit tcgen05 GEMM: C = A[M, K] * B[N, K]^T -> epilogue, A and B both bf16 (or both
// fp16 when ab_f16).  a_cols / b_cols: valid columns of A / B (TMA zero-fills beyond);
// lda / ldb: row strides in elements.  kb_period > 0: the B k-block index wraps modulo
// kb_period (A = [hi | lo] split).
int gemm_bf16(const LaunchCtx& c, const void* A, long long lda, int a_cols, const void* B, long long ldb,
              int b_cols, int M, int N, int K, int kb_period, const EpiParams& ep, const char* tag,
              bool ab_f16 = false);
// FP8 (E4M3) tcgen05 GEMM: C = (A8 sa) (B8 sb)^T -> epilogue, with per-row scales sa [M]
// of A and per-row scales sb [N] of B (per output channel) applied to the fp32
// accumulator before the epilogue.  lda / ldb: row strides in bytes (multiples of 16).
int gemm_e4m3(const LaunchCtx& c, const uint8_t* A, long long lda, int a_cols, const float* sa, const uint8_t* B,
              long long ldb, int b_cols, const float* sb, int M, int N, int K, const EpiParams& ep, const char* tag);
// fp32 SIMT GEMM (parity path): same contract, fp32 operands.
int gemm_f32(const LaunchCtx& c, const float* A, long long lda, const float* B, long long ldb, int M, int N, int K,
             const EpiParams& ep, const char* tag);

// ------------------------------------------------------------------ attention
struct AttnArgs {
  const void* q;
  long long ldq;   // row stride of q (elements)
  int q_row_len;   // valid elements per q row
  int q_col;       // column of head 0
  const void* k;
  long long ldk;
  int k_row_len;
  int k_col;
  const void* v;   // [B, Lkv, ldv] rows; head h at columns v_col + h*d
  long long ldv;
  int v_row_len;
  int v_col;
  void* o;
  long long ldo;
  int o_col;
  int B, Lq, Lkv, H, head_dim;
  const int* kv_lens;  // device [B]: valid keys per batch entry (clamped to [1, Lkv]), or NULL = Lkv
  int accumulate;  // o += result
  int qk_f16;      // bf16 path: q and k are fp16 (else bf16); v and o are bf16
  const char* tag; // profiler label of the launch
};
int attention_bf16(const LaunchCtx& c, const AttnArgs& a);

// Decoupled cross-attention in one persistent launch (attn_cross.cu):
//   o = softmax(q kt^T / sqrt(d)) vt [+ softmax(q ki^T / sqrt(d)) vi]
// Rows are [B, len, ld*] with head h at columns *_col + h * d.  q and k are bf16 or fp16
// (qk_f16); v and o are both bf16 or both fp16 (pv_f16, which needs qk_f16).
struct CrossArgs {
  const void* q;
  long long ldq;
  int q_row_len, q_col;
  const void *kt, *vt;  // text keys / values [B, Lt, ld]
  long long ldkt, ldvt;
  int kt_row_len, vt_row_len, kt_col, vt_col;
  const void *ki, *vi;  // image keys / values [B, Li, ld], or NULL when Li == 0
  long long ldki, ldvi;
  int ki_row_len, vi_row_len, ki_col, vi_col;
  void* o;
  long long ldo;
  int o_col;
  int B, L, Lt, Li, H, head_dim;
  const int* kt_lens;  // device [B]: valid text keys per batch entry (clamped to [1, Lt]), or NULL
  int qk_f16, pv_f16;
  const char* tag;
};
int cross_attention_tc(const LaunchCtx& c, const CrossArgs& a);
int attention_f32(const LaunchCtx& c, const AttnArgs& a);

// ------------------------------------------------------------------ 8-bit operands and attention
// Quantiser inputs (q, k, v rows of the QKV projection, bf16 or fp16) and outputs.
struct Attn8Operands {
  const void* q;
  long long ldq;  // row stride (elements)
  int q_col;      // column of head 0
  const void* k;
  long long ldk;
  int k_col;
  const void* v;
  long long ldv;
  int v_col;
  int qk_type, v_type;  // OutType of the inputs: OUT_BF16 or OUT_F16
  int B, L, H, head_dim;
  int nkb;  // ceil(L / 128)
  int Lp;   // L rounded up to 16
  uint8_t* q8;  // [B*L, H*d]
  float* sq;    // [B*L, H]
  uint8_t* k8;  // [B*L, H*d]
  float* sk;    // [B, H, nkb]
  uint8_t* v8t; // [B, H, d, Lp]
  float* sv;    // [B, H, d]
  unsigned int* v_amax;  // [B, H, d] scratch
};
int quant_attn_e4m3(const LaunchCtx& c, const Attn8Operands& a);
struct Attn8Args {
  const uint8_t* q8;
  const float* sq;
  const uint8_t* k8;
  const float* sk;
  const uint8_t* v8t;
  const float* sv;
  void* o;  // bf16 [B, L, ldo], head h at columns o_col + h*d
  long long ldo;
  int o_col;
  int B, L, H, head_dim, Lp;
  const int* kv_lens;  // device [B] or NULL
  const char* tag;
};
int attention_e4m3(const LaunchCtx& c, const Attn8Args& a);
// x8[r, :] = E4M3 codes of row r of x (in_type OutType), s[r] its dequantisation scale.
int launch_quant_rows_e4m3(const LaunchCtx& c, const void* x, int in_type, long long ldx, int rows, int K,
                           uint8_t* x8, long long ld8, float* s);
// LN + modulation (as launch_ln_mod) written as per-row E4M3 codes y8 [rows, D] and scales sy [rows].
int launch_ln_mod_e4m3(const LaunchCtx& c, const float* x, const float* shift, const float* scale,
                       long long mod_bstride, uint8_t* y8, float* sy, int rows, int L, int D, float eps);

// ------------------------------------------------------------------ elementwise / small kernels
// y = LN(x)(1 + scale) + shift per row, stored as out_type (OutType: bf16, fp16 or fp32).
int launch_ln_mod(const LaunchCtx& c, const float* x, const float* shift, const float* scale, long long mod_bstride,
                  void* y, int out_type, int rows, int L, int D, float eps);
int launch_cfg_euler(const LaunchCtx& c, float* x, const void* vc, const void* vu, long long n, float s, float dt,
                     const float* t_pair, int v_f32);
int launch_patch_gather(const LaunchCtx& c, const float* latent, long long latent_bstride, void* A, int out_f32,
                        int B, int C, int F, int H, int W, int kpad);
// omega[j] = theta^(-2 j_a / d_a) for the head's d/2 rotation pairs (axis parts f | h | w).
int launch_rope_table(const LaunchCtx& c, float* omega, int head_dim, float theta);
// t[b * t_stride] (t_stride 0: one timestep shared by the batch).
int launch_sinusoid(const LaunchCtx& c, const float* t, int t_stride, float* s, int B, int dim);
// out[b, n] = act_out(sum_k W[n, k] * act_in(x[b, k]) + bias[n]); act: 0 none, 1 SiLU.
int launch_small_linear(const LaunchCtx& c, const float* x, const void* W, const void* bias, int w_f32, float* out,
                        int B, int N, int K, int act_in, int act_out);
// mods[blk][b][k][n] = e0[b][k*D + n] + mod_blk[k][n] for `nblk` blocks.
int launch_block_mods(const LaunchCtx& c, const float* e0, const void* const* mod_ptrs, int nblk, int w_f32,
                      float* mods, int B, int D);
// Rotate q [B, L, H*d] into out (same layout) with the 3D-RoPE table.  in_type (OutType):
// bf16 or fp16 input is written out in fp16, fp32 stays fp32.
int launch_rope_apply(const LaunchCtx& c, const void* in, void* out, const RopeGeom& g, int B, int L, int H, int d,
                      int in_type);
int launch_schedule(const LaunchCtx& c, float* ts, int steps);
// In place on the q | k | v rows (row stride ld): q and k <- RoPE(RMSNorm(.) * w) over D.
int launch_qk_rmsnorm_rope(const LaunchCtx& c, void* qkv, long long ld, const void* wq, const void* wk,
                           const RopeGeom& g, int rows, int L, int D, int hd, float eps, int f32);
// A kernel whose only wait never completes: it gives up after limit_ns (status word set).
int launch_watchdog_selftest(const LaunchCtx& c, unsigned long long limit_ns);

// RoPE table geometry for head_dim d on grid (Fg, Hg, Wg).
inline RopeGeom rope_geom(const float* omega, int Fg, int Hg, int Wg, int d) {
  RopeGeom g;
  const int dh = 2 * (d / 6);
  const int df = d - 2 * dh;
  g.omega = omega;
  g.Fg = Fg;
  g.Hg = Hg;
  g.Wg = Wg;
  g.nf = df / 2;
  g.nh = dh / 2;
  g.nw = dh / 2;
  return g;
}

}  // namespace wan

// GEMM epilogues of the DiT block: every projection's bias, activation, 3D RoPE,
// gated residual and layout change is applied to a row chunk of the accumulator
// right where it leaves the tensor core (or the SIMT accumulator), so no extra pass
// over HBM is needed for them.
#pragma once

#include <cuda_fp16.h>

#include "wan_common.cuh"

namespace wan {

enum EpiKind : int {
  EPI_STORE = 0,  // out[m, n] = acc + bias
  EPI_GELU = 1,   // out[m, n] = GELU(acc + bias)
  EPI_RESID = 2,  // resid[m, n] += gate[b, n] * (acc + bias)   (gate NULL: 1)
  EPI_QKV = 3,    // cols [0, n_qk): (RoPE on [0, n_rot)) -> qk[m, n]; cols [n_qk, N): -> vt
  EPI_HEAD = 4,   // depatchify: vout[b, c, f, 2i+di, 2j+dj] = acc + bias, n = c*4 + di*2 + dj
};

struct RopeGeom {
  const float2* tab;  // [Fg*nf | Hg*nh | Wg*nw] (cos, sin)
  int Fg, Hg, Wg;     // token grid
  int nf, nh, nw;     // rotation pairs per axis
};

// Storage types of epilogue outputs.
enum OutType : int { OUT_BF16 = 0, OUT_F32 = 1, OUT_F16 = 2 };

struct EpiParams {
  int kind;
  int M, N;
  int rows_per_batch;  // L (tokens per sample): b = m / L, l = m % L
  const void* bias;    // [N] or NULL
  int bias_f32;
  // EPI_STORE / EPI_GELU
  void* out;
  long long ldo;
  int out_type;  // OutType
  // EPI_RESID
  float* resid;
  long long ldr;
  const float* gate;
  long long ld_gate;  // gate batch stride (elements)
  // EPI_QKV
  void* qk;
  long long ldqk;
  int qk_type;  // OutType of q|k
  int vt_type;  // OutType of v^T (OUT_BF16 or OUT_F32)
  int n_qk, n_rot;
  void* vt;            // [(b*H + h)*hd + dd] rows of ld_vt elements
  long long ld_vt;
  int head_dim, heads;
  RopeGeom rope;
  // EPI_HEAD
  float* vout;
  int C, F, H, W;
};

__device__ __forceinline__ float epi_bias(const EpiParams& p, int n) {
  if (p.bias_f32) return static_cast<const float*>(p.bias)[n];
  return bf2f(static_cast<const bf16*>(p.bias)[n]);
}

// Store CNT consecutive values (CNT % 4 == 0, 16-byte aligned destinations for CNT >= 8).
__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
  __half2 p = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&p);
}

template <int CNT>
__device__ __forceinline__ void epi_store_row(void* base, int type, long long off, const float* v) {
  if (type == OUT_F32) {
    float4* d = reinterpret_cast<float4*>(static_cast<float*>(base) + off);
#pragma unroll
    for (int i = 0; i < CNT / 4; ++i) d[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
    return;
  }
  uint16_t* d = static_cast<uint16_t*>(base) + off;
  const bool h = type == OUT_F16;
  if constexpr (CNT % 8 == 0) {
#pragma unroll
    for (int i = 0; i < CNT / 8; ++i) {
      uint4 u;
      u.x = h ? pack_half2(v[8 * i + 0], v[8 * i + 1]) : pack_bf16x2(v[8 * i + 0], v[8 * i + 1]);
      u.y = h ? pack_half2(v[8 * i + 2], v[8 * i + 3]) : pack_bf16x2(v[8 * i + 2], v[8 * i + 3]);
      u.z = h ? pack_half2(v[8 * i + 4], v[8 * i + 5]) : pack_bf16x2(v[8 * i + 4], v[8 * i + 5]);
      u.w = h ? pack_half2(v[8 * i + 6], v[8 * i + 7]) : pack_bf16x2(v[8 * i + 6], v[8 * i + 7]);
      reinterpret_cast<uint4*>(d)[i] = u;
    }
  } else {
#pragma unroll
    for (int i = 0; i < CNT / 4; ++i) {
      uint2 u;
      u.x = h ? pack_half2(v[4 * i + 0], v[4 * i + 1]) : pack_bf16x2(v[4 * i + 0], v[4 * i + 1]);
      u.y = h ? pack_half2(v[4 * i + 2], v[4 * i + 3]) : pack_bf16x2(v[4 * i + 2], v[4 * i + 3]);
      reinterpret_cast<uint2*>(d)[i] = u;
    }
  }
}

// Rotate the adjacent pairs of v (CNT values starting at head-dim index dd0, even) by
// the 3D-RoPE angles of token l.
template <int CNT>
__device__ __forceinline__ void epi_rope(const RopeGeom& g, int head_dim, int dd0, int l, float* v) {
  const int pf = l / (g.Hg * g.Wg);
  const int ph = (l / g.Wg) % g.Hg;
  const int pw = l % g.Wg;
  const float2* tf = g.tab + pf * g.nf;
  const float2* th = g.tab + g.Fg * g.nf + ph * g.nh;
  const float2* tw = g.tab + g.Fg * g.nf + g.Hg * g.nh + pw * g.nw;
#pragma unroll
  for (int i = 0; i < CNT / 2; ++i) {
    const int pair = (dd0 >> 1) + i;  // pair index within the head
    float2 cs;
    if (pair < g.nf) cs = tf[pair];
    else if (pair < g.nf + g.nh) cs = th[pair - g.nf];
    else cs = tw[pair - g.nf - g.nh];
    const float x0 = v[2 * i], x1 = v[2 * i + 1];
    v[2 * i] = x0 * cs.x - x1 * cs.y;
    v[2 * i + 1] = x0 * cs.y + x1 * cs.x;
  }
  (void)head_dim;
}

// Gated-residual update values of row m, columns n0..n0+CNT-1: v <- gate[b, n] * (v + bias[n])
// (gate NULL: 1).  Rows at or past M (a tile's ragged tail) get 0 and read no gate.
template <int CNT>
__device__ __forceinline__ void epi_resid_values(const EpiParams& p, int m, int n0, float* v) {
  if (m >= p.M) {
#pragma unroll
    for (int i = 0; i < CNT; ++i) v[i] = 0.f;
    return;
  }
  if (p.bias) {
#pragma unroll
    for (int i = 0; i < CNT; ++i) v[i] += epi_bias(p, n0 + i);
  }
  if (p.gate) {
    const float* g = p.gate + (long long)(m / p.rows_per_batch) * p.ld_gate + n0;
#pragma unroll
    for (int i = 0; i < CNT / 4; ++i) {
      const float4 gg = *reinterpret_cast<const float4*>(g + 4 * i);
      v[4 * i] *= gg.x;
      v[4 * i + 1] *= gg.y;
      v[4 * i + 2] *= gg.z;
      v[4 * i + 3] *= gg.w;
    }
  }
}

// Apply the epilogue to values v[0..CNT) of row m, columns n0..n0+CNT-1 (all valid;
// n0 % CNT == 0 and the chunk never straddles a section or head boundary).
template <int CNT>
__device__ __forceinline__ void epilogue_chunk(const EpiParams& p, int m, int n0, float* v) {
  if (p.bias) {
#pragma unroll
    for (int i = 0; i < CNT; ++i) v[i] += epi_bias(p, n0 + i);
  }
  const int b = m / p.rows_per_batch;
  const int l = m - b * p.rows_per_batch;
  switch (p.kind) {
    case EPI_GELU:
#pragma unroll
      for (int i = 0; i < CNT; ++i) v[i] = gelu_erf(v[i]);
      // fallthrough
    case EPI_STORE:
      epi_store_row<CNT>(p.out, p.out_type, (long long)m * p.ldo + n0, v);
      break;
    case EPI_RESID: {
      float4* x = reinterpret_cast<float4*>(p.resid + (long long)m * p.ldr + n0);
      const float* g = p.gate ? p.gate + (long long)b * p.ld_gate + n0 : nullptr;
#pragma unroll
      for (int i = 0; i < CNT / 4; ++i) {
        float4 a = x[i];
        float4 gg = g ? *reinterpret_cast<const float4*>(g + 4 * i) : make_float4(1.f, 1.f, 1.f, 1.f);
        a.x += gg.x * v[4 * i + 0];
        a.y += gg.y * v[4 * i + 1];
        a.z += gg.z * v[4 * i + 2];
        a.w += gg.w * v[4 * i + 3];
        x[i] = a;
      }
      break;
    }
    case EPI_QKV: {
      if (n0 < p.n_qk) {
        if (n0 < p.n_rot) epi_rope<CNT>(p.rope, p.head_dim, n0 % p.head_dim, l, v);
        epi_store_row<CNT>(p.qk, p.qk_type, (long long)m * p.ldqk + n0, v);
      } else {
        const int c = n0 - p.n_qk;
        const int h = c / p.head_dim;
        const int dd0 = c - h * p.head_dim;
        const long long row0 = ((long long)b * p.heads + h) * p.head_dim + dd0;
        if (p.vt_type == OUT_F32) {
          float* vt = static_cast<float*>(p.vt);
#pragma unroll
          for (int i = 0; i < CNT; ++i) vt[(row0 + i) * p.ld_vt + l] = v[i];
        } else {
          bf16* vt = static_cast<bf16*>(p.vt);
#pragma unroll
          for (int i = 0; i < CNT; ++i) vt[(row0 + i) * p.ld_vt + l] = __float2bfloat16_rn(v[i]);
        }
      }
      break;
    }
    case EPI_HEAD: {
      const int Hp = p.H >> 1, Wp = p.W >> 1;
      const int f = l / (Hp * Wp);
      const int i = (l / Wp) % Hp;
      const int j = l % Wp;
#pragma unroll
      for (int k = 0; k < CNT; ++k) {
        const int n = n0 + k;
        const int c = n >> 2, di = (n >> 1) & 1, dj = n & 1;
        p.vout[(((long long)b * p.C + c) * p.F + f) * p.H * p.W + (long long)(2 * i + di) * p.W +
               (2 * j + dj)] = v[k];
      }
      break;
    }
    default:
      break;
  }
}

}  // namespace wan

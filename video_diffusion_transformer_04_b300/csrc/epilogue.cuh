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
  EPI_QKV = 3,    // out[m, n] = acc + bias, RoPE on cols [0, n_rot), fp16 on cols [0, n_f16)
  EPI_HEAD = 4,   // depatchify: vout[b, c, f, 2i+di, 2j+dj] = acc + bias, n = c*4 + di*2 + dj
  EPI_GELU_TANH = 5,  // out[m, n] = GELU_tanh(acc + bias)
};

struct RopeGeom {
  const float* omega;  // [nf | nh | nw] angular frequency of each rotation pair of a head
  int Fg, Hg, Wg;      // token grid
  int nf, nh, nw;      // rotation pairs per axis
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
  // EPI_QKV (also uses out / ldo / out_type for the columns past n_f16)
  int n_rot, n_f16;
  int head_dim;
  RopeGeom rope;
  // EPI_HEAD
  float* vout;
  int C, F, H, W;
  // FP8 GEMM: acc[m, n] * a_scale[m] * b_scale[n] before everything above
  const float* a_scale;
  const float* b_scale;
  // EPI_STORE / EPI_GELU / EPI_GELU_TANH / EPI_QKV: the tile goes out through shared
  // memory and TMA stores (set by the host when the output allows it) instead of one
  // row per thread.
  int tma_store;
};

// v[i] += bias[n0 + i] with 16-byte vector loads (bias rows are 16-byte aligned and n0
// is a multiple of CNT).
template <int CNT>
__device__ __forceinline__ void epi_add_bias(const EpiParams& p, int n0, float* v) {
  if (!p.bias) return;
  if (p.bias_f32) {
    const float4* b = reinterpret_cast<const float4*>(static_cast<const float*>(p.bias) + n0);
#pragma unroll
    for (int i = 0; i < CNT / 4; ++i) {
      const float4 q = b[i];
      v[4 * i] += q.x;
      v[4 * i + 1] += q.y;
      v[4 * i + 2] += q.z;
      v[4 * i + 3] += q.w;
    }
  } else if constexpr (CNT % 8 == 0) {
    const uint4* b = reinterpret_cast<const uint4*>(static_cast<const bf16*>(p.bias) + n0);
#pragma unroll
    for (int i = 0; i < CNT / 8; ++i) {
      const uint4 q = b[i];
      const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const float2 f = unpack_bf16x2(w[u]);
        v[8 * i + 2 * u] += f.x;
        v[8 * i + 2 * u + 1] += f.y;
      }
    }
  } else {
    const uint2* b = reinterpret_cast<const uint2*>(static_cast<const bf16*>(p.bias) + n0);
#pragma unroll
    for (int i = 0; i < CNT / 4; ++i) {
      const uint2 q = b[i];
      const float2 lo = unpack_bf16x2(q.x), hi = unpack_bf16x2(q.y);
      v[4 * i] += lo.x;
      v[4 * i + 1] += lo.y;
      v[4 * i + 2] += hi.x;
      v[4 * i + 3] += hi.y;
    }
  }
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
// the 3D-RoPE angles of token l: pair j of the head turns by pos_a(j) * omega[j], pos_a
// the token's frame, height or width index for the axis that owns pair j.  The sine and
// cosine come from the SFU (__sincosf, absolute error about 1e-6 at the grid's angles).
template <int CNT>
__device__ __forceinline__ void epi_rope(const RopeGeom& g, int head_dim, int dd0, int l, float* v) {
  const int hw = g.Hg * g.Wg;
  const int pf = l / hw;
  const int rem = l - pf * hw;
  const int ph = rem / g.Wg;
  const int pw = rem - ph * g.Wg;
#pragma unroll
  for (int i = 0; i < CNT / 2; ++i) {
    const int pair = (dd0 >> 1) + i;  // pair index within the head
    const int pos = pair < g.nf ? pf : (pair < g.nf + g.nh ? ph : pw);
    float sn, cs;
    __sincosf((float)pos * g.omega[pair], &sn, &cs);
    const float x0 = v[2 * i], x1 = v[2 * i + 1];
    v[2 * i] = x0 * cs - x1 * sn;
    v[2 * i + 1] = x0 * sn + x1 * cs;
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
  epi_add_bias<CNT>(p, n0, v);
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

// The values the store-type epilogues write for row m, columns n0..n0+CNT-1: bias, then
// GELU, or 3D RoPE on the q / k columns of EPI_QKV.
template <int CNT>
__device__ __forceinline__ void epilogue_values(const EpiParams& p, int m, int n0, float* v) {
  epi_add_bias<CNT>(p, n0, v);
  if (p.kind == EPI_GELU) {
#pragma unroll
    for (int i = 0; i < CNT; i += 2) gelu_erf2(v[i], v[i + 1]);
  } else if (p.kind == EPI_GELU_TANH) {
#pragma unroll
    for (int i = 0; i < CNT; ++i) v[i] = gelu_tanh_form(v[i]);
  } else if (p.kind == EPI_QKV && n0 < p.n_rot) {
    const int b = m / p.rows_per_batch;
    epi_rope<CNT>(p.rope, p.head_dim, n0 % p.head_dim, m - b * p.rows_per_batch, v);
  }
}
// Storage type of the store-type epilogues' column n0.
__device__ __forceinline__ int epilogue_out_type(const EpiParams& p, int n0) {
  return (p.kind == EPI_QKV && n0 < p.n_f16) ? OUT_F16 : p.out_type;
}

// Apply the epilogue to values v[0..CNT) of row m, columns n0..n0+CNT-1 (all valid;
// n0 % CNT == 0 and the chunk never straddles a section or head boundary).
template <int CNT>
__device__ __forceinline__ void epilogue_chunk(const EpiParams& p, int m, int n0, float* v) {
  epi_add_bias<CNT>(p, n0, v);
  const int b = m / p.rows_per_batch;
  const int l = m - b * p.rows_per_batch;
  switch (p.kind) {
    case EPI_GELU_TANH:
#pragma unroll
      for (int i = 0; i < CNT; ++i) v[i] = gelu_tanh_form(v[i]);
      epi_store_row<CNT>(p.out, p.out_type, (long long)m * p.ldo + n0, v);
      break;
    case EPI_GELU:
#pragma unroll
      for (int i = 0; i < CNT; i += 2) gelu_erf2(v[i], v[i + 1]);
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
      // q | k | v row of the projection: RoPE on q and k, q and k in fp16 for the QK^T
      // product, v in the call's storage type, all stored in place in one row buffer.
      if (n0 < p.n_rot) epi_rope<CNT>(p.rope, p.head_dim, n0 % p.head_dim, l, v);
      epi_store_row<CNT>(p.out, n0 < p.n_f16 ? OUT_F16 : p.out_type, (long long)m * p.ldo + n0, v);
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

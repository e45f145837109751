// Bandwidth-bound passes of the DiT step: LayerNorm + AdaLN modulation, fused CFG +
// Euler update, the patch gather feeding the patchify GEMM, and the small kernels of
// the time embedding, RoPE table and layout changes.
#include <type_traits>

#include "kernels.h"

namespace wan {

// ------------------------------------------------------------------ LayerNorm + modulation
// One 128-thread CTA per token row; the row stays in registers between the mean, the
// (centred) variance and the normalisation.  y = (x - mu) * rstd * (1 + scale) + shift.
template <int NV, typename OutT>
__global__ void __launch_bounds__(128) ln_mod_kernel(const float* __restrict__ x, const float* __restrict__ shift,
                                                     const float* __restrict__ scale, long long mod_bstride,
                                                     OutT* __restrict__ y, float* __restrict__ sy, int L, int D,
                                                     float eps) {
  __shared__ float red[4];
  const int row = blockIdx.x;
  const int b = row / L;
  const int t = threadIdx.x;
  const int nv4 = D >> 2;
  const float4* xr = reinterpret_cast<const float4*>(x + (long long)row * D);
  float4 v[NV];
  float s = 0.f;
#pragma unroll
  for (int i = 0; i < NV; ++i) {
    const int c = t + i * 128;
    v[i] = c < nv4 ? xr[c] : make_float4(0.f, 0.f, 0.f, 0.f);
    s += (v[i].x + v[i].y) + (v[i].z + v[i].w);
  }
  auto block_sum = [&](float a) {
    for (int o = 16; o > 0; o >>= 1) a += __shfl_xor_sync(0xffffffffu, a, o);
    __syncthreads();
    if ((t & 31) == 0) red[t >> 5] = a;
    __syncthreads();
    return (red[0] + red[1]) + (red[2] + red[3]);
  };
  const float mean = block_sum(s) / (float)D;
  float q = 0.f;
#pragma unroll
  for (int i = 0; i < NV; ++i) {
    const int c = t + i * 128;
    if (c < nv4) {
      const float a0 = v[i].x - mean, a1 = v[i].y - mean, a2 = v[i].z - mean, a3 = v[i].w - mean;
      q += (a0 * a0 + a1 * a1) + (a2 * a2 + a3 * a3);
    }
  }
  const float var = block_sum(q) / (float)D;
  const float rstd = rsqrtf(var + eps);
  const float* sh = shift ? shift + (long long)b * mod_bstride : nullptr;
  const float* sc = scale ? scale + (long long)b * mod_bstride : nullptr;
  float o[NV][4];
#pragma unroll
  for (int i = 0; i < NV; ++i) {
    const int c = t + i * 128;
    o[i][0] = (v[i].x - mean) * rstd; o[i][1] = (v[i].y - mean) * rstd;
    o[i][2] = (v[i].z - mean) * rstd; o[i][3] = (v[i].w - mean) * rstd;
    if (c >= nv4) continue;
    if (sc) {
      const float4 s4 = reinterpret_cast<const float4*>(sc)[c];
      o[i][0] *= 1.f + s4.x; o[i][1] *= 1.f + s4.y; o[i][2] *= 1.f + s4.z; o[i][3] *= 1.f + s4.w;
    }
    if (sh) {
      const float4 h4 = reinterpret_cast<const float4*>(sh)[c];
      o[i][0] += h4.x; o[i][1] += h4.y; o[i][2] += h4.z; o[i][3] += h4.w;
    }
  }
  // E4M3 output: per-row scale from the row's |max| (decided in fp32).
  float inv = 0.f;
  if constexpr (sizeof(OutT) == 1) {
    float a = 0.f;
#pragma unroll
    for (int i = 0; i < NV; ++i)
      if (t + i * 128 < nv4)
        a = fmaxf(a, fmaxf(fmaxf(fabsf(o[i][0]), fabsf(o[i][1])), fmaxf(fabsf(o[i][2]), fabsf(o[i][3]))));
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, off));
    __syncthreads();
    if ((t & 31) == 0) red[t >> 5] = a;
    __syncthreads();
    a = fmaxf(fmaxf(red[0], red[1]), fmaxf(red[2], red[3]));
    inv = e4m3_inv(a);
    if (t == 0) sy[row] = e4m3_deq(a);
  }
#pragma unroll
  for (int i = 0; i < NV; ++i) {
    const int c = t + i * 128;
    if (c >= nv4) continue;
    if constexpr (sizeof(OutT) == 4) {
      reinterpret_cast<float4*>(y + (long long)row * D)[c] = make_float4(o[i][0], o[i][1], o[i][2], o[i][3]);
    } else if constexpr (std::is_same<OutT, __half>::value) {
      uint2 u;
      u.x = pack_half2(o[i][0], o[i][1]);
      u.y = pack_half2(o[i][2], o[i][3]);
      reinterpret_cast<uint2*>(y + (long long)row * D)[c] = u;
    } else if constexpr (sizeof(OutT) == 2) {
      uint2 u;
      u.x = pack_bf16x2(o[i][0], o[i][1]);
      u.y = pack_bf16x2(o[i][2], o[i][3]);
      reinterpret_cast<uint2*>(y + (long long)row * D)[c] = u;
    } else {
      reinterpret_cast<uint32_t*>(y + (long long)row * D)[c] =
          e4m3x4(__fmul_rn(o[i][0], inv), __fmul_rn(o[i][1], inv), __fmul_rn(o[i][2], inv), __fmul_rn(o[i][3], inv));
    }
  }
}

// The same pass with one warp per token row (rows up to 2048 wide): the row stays in
// registers (NV float4 per lane), mean and centred variance reduce by warp shuffles
// alone, and a 256-thread CTA carries eight rows, so no block barrier sits between a
// row's loads and its stores.
template <int NV, typename OutT>
__global__ void __launch_bounds__(256) ln_mod_warp_kernel(const float* __restrict__ x,
                                                          const float* __restrict__ shift,
                                                          const float* __restrict__ scale, long long mod_bstride,
                                                          OutT* __restrict__ y, int rows, int L, int D, float eps) {
  const int lane = threadIdx.x & 31;
  const int row = blockIdx.x * 8 + (threadIdx.x >> 5);
  if (row >= rows) return;
  const int b = row / L;
  const int nv4 = D >> 2;
  const float4* xr = reinterpret_cast<const float4*>(x + (long long)row * D);
  float4 v[NV];
  float s = 0.f;
#pragma unroll
  for (int i = 0; i < NV; ++i) {
    const int c = lane + i * 32;
    v[i] = c < nv4 ? xr[c] : make_float4(0.f, 0.f, 0.f, 0.f);
    s += (v[i].x + v[i].y) + (v[i].z + v[i].w);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  const float mean = s / (float)D;
  float q = 0.f;
#pragma unroll
  for (int i = 0; i < NV; ++i) {
    if (lane + i * 32 < nv4) {
      const float a0 = v[i].x - mean, a1 = v[i].y - mean, a2 = v[i].z - mean, a3 = v[i].w - mean;
      q += (a0 * a0 + a1 * a1) + (a2 * a2 + a3 * a3);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) q += __shfl_xor_sync(0xffffffffu, q, o);
  const float rstd = rsqrtf(q / (float)D + eps);
  const float4* sh = shift ? reinterpret_cast<const float4*>(shift + (long long)b * mod_bstride) : nullptr;
  const float4* sc = scale ? reinterpret_cast<const float4*>(scale + (long long)b * mod_bstride) : nullptr;
#pragma unroll
  for (int i = 0; i < NV; ++i) {
    const int c = lane + i * 32;
    if (c >= nv4) continue;
    float o0 = (v[i].x - mean) * rstd, o1 = (v[i].y - mean) * rstd;
    float o2 = (v[i].z - mean) * rstd, o3 = (v[i].w - mean) * rstd;
    if (sc) {
      const float4 s4 = sc[c];
      o0 *= 1.f + s4.x; o1 *= 1.f + s4.y; o2 *= 1.f + s4.z; o3 *= 1.f + s4.w;
    }
    if (sh) {
      const float4 h4 = sh[c];
      o0 += h4.x; o1 += h4.y; o2 += h4.z; o3 += h4.w;
    }
    if constexpr (sizeof(OutT) == 4) {
      reinterpret_cast<float4*>(y + (long long)row * D)[c] = make_float4(o0, o1, o2, o3);
    } else if constexpr (std::is_same<OutT, __half>::value) {
      reinterpret_cast<uint2*>(y + (long long)row * D)[c] = make_uint2(pack_half2(o0, o1), pack_half2(o2, o3));
    } else {
      reinterpret_cast<uint2*>(y + (long long)row * D)[c] = make_uint2(pack_bf16x2(o0, o1), pack_bf16x2(o2, o3));
    }
  }
}

template <typename OutT>
static void ln_dispatch(const LaunchCtx& c, const float* x, const float* sh, const float* sc, long long bs, OutT* y,
                        float* sy, int rows, int L, int D, float eps) {
  if constexpr (sizeof(OutT) != 1) {  // E4M3 output keeps the block kernel (row |max| decision)
    if (D <= 2048) {
      const int nw = (D / 4 + 31) / 32;  // float4 per lane
      const unsigned grid = (unsigned)((rows + 7) / 8);
      if (nw <= 4) ln_mod_warp_kernel<4, OutT><<<grid, 256, 0, c.stream>>>(x, sh, sc, bs, y, rows, L, D, eps);
      else if (nw <= 8) ln_mod_warp_kernel<8, OutT><<<grid, 256, 0, c.stream>>>(x, sh, sc, bs, y, rows, L, D, eps);
      else if (nw <= 12) ln_mod_warp_kernel<12, OutT><<<grid, 256, 0, c.stream>>>(x, sh, sc, bs, y, rows, L, D, eps);
      else ln_mod_warp_kernel<16, OutT><<<grid, 256, 0, c.stream>>>(x, sh, sc, bs, y, rows, L, D, eps);
      return;
    }
  }
  const int nv = (D / 4 + 127) / 128;
  if (nv <= 1) ln_mod_kernel<1, OutT><<<rows, 128, 0, c.stream>>>(x, sh, sc, bs, y, sy, L, D, eps);
  else if (nv <= 3) ln_mod_kernel<3, OutT><<<rows, 128, 0, c.stream>>>(x, sh, sc, bs, y, sy, L, D, eps);
  else if (nv <= 10) ln_mod_kernel<10, OutT><<<rows, 128, 0, c.stream>>>(x, sh, sc, bs, y, sy, L, D, eps);
  else ln_mod_kernel<16, OutT><<<rows, 128, 0, c.stream>>>(x, sh, sc, bs, y, sy, L, D, eps);
}

int launch_ln_mod(const LaunchCtx& c, const float* x, const float* shift, const float* scale, long long mod_bstride,
                  void* y, int out_type, int rows, int L, int D, float eps) {
  if (rows <= 0) return WAN_OK;
  if (D % 4 != 0 || D > 8192) return WAN_ERR_UNSUPPORTED;
  count_launch("ln_modulate", c.stream, true);
  if (out_type == OUT_F32)
    ln_dispatch<float>(c, x, shift, scale, mod_bstride, static_cast<float*>(y), nullptr, rows, L, D, eps);
  else if (out_type == OUT_F16)
    ln_dispatch<__half>(c, x, shift, scale, mod_bstride, static_cast<__half*>(y), nullptr, rows, L, D, eps);
  else
    ln_dispatch<bf16>(c, x, shift, scale, mod_bstride, static_cast<bf16*>(y), nullptr, rows, L, D, eps);
  count_launch("ln_modulate", c.stream, false);
  return cudaGetLastError() == cudaSuccess ? WAN_OK : WAN_ERR_CUDA;
}

int launch_ln_mod_e4m3(const LaunchCtx& c, const float* x, const float* shift, const float* scale,
                       long long mod_bstride, uint8_t* y8, float* sy, int rows, int L, int D, float eps) {
  if (rows <= 0) return WAN_OK;
  if (D % 4 != 0 || D > 8192) return WAN_ERR_UNSUPPORTED;
  count_launch("ln_modulate_e4m3", c.stream, true);
  ln_dispatch<uint8_t>(c, x, shift, scale, mod_bstride, y8, sy, rows, L, D, eps);
  count_launch("ln_modulate_e4m3", c.stream, false);
  return cudaGetLastError() == cudaSuccess ? WAN_OK : WAN_ERR_CUDA;
}

// ------------------------------------------------------------------ CFG + Euler
// x <- x + dt * (vu + s * (vc - vu)) on float4 groups (16-byte accesses); a scalar loop
// takes the n % 4 tail.
template <typename VT>
__device__ __forceinline__ void load4(const VT* p, long long i, float* o);
template <>
__device__ __forceinline__ void load4<float>(const float* p, long long i, float* o) {
  const float4 a = *reinterpret_cast<const float4*>(p + i);
  o[0] = a.x; o[1] = a.y; o[2] = a.z; o[3] = a.w;
}
template <>
__device__ __forceinline__ void load4<bf16>(const bf16* p, long long i, float* o) {
  const uint2 a = *reinterpret_cast<const uint2*>(p + i);
  const float2 lo = unpack_bf16x2(a.x), hi = unpack_bf16x2(a.y);
  o[0] = lo.x; o[1] = lo.y; o[2] = hi.x; o[3] = hi.y;
}
template <typename VT>
__device__ __forceinline__ float load1(const VT* p, long long i) {
  if constexpr (sizeof(VT) == 4) return p[i];
  else return bf2f(p[i]);
}

// Each thread takes U float4 groups per pass (g, g + T, ..., g + (U-1) T for T threads in
// the grid) and issues all their loads before any arithmetic, so every thread keeps 3U
// 16-byte loads in flight; the grid covers the tensor in one or two passes.
template <typename VT, int U>
__global__ void __launch_bounds__(128) cfg_euler_kernel(float* __restrict__ x, const VT* __restrict__ vc,
                                                        const VT* __restrict__ vu, long long n, float s, float dt,
                                                        const float* __restrict__ t_pair) {
  if (t_pair) dt = t_pair[1] - t_pair[0];
  const long long n4 = n >> 2;
  const long long T = (long long)gridDim.x * blockDim.x;
  for (long long g = (long long)blockIdx.x * blockDim.x + threadIdx.x; g < n4; g += T * U) {
    float a[U][4], c[U][4], u[U][4];
#pragma unroll
    for (int k = 0; k < U; ++k) {
      const long long gi = g + k * T;
      if (gi < n4) {
        load4<float>(x, gi << 2, a[k]);
        load4<VT>(vc, gi << 2, c[k]);
        load4<VT>(vu, gi << 2, u[k]);
      }
    }
#pragma unroll
    for (int k = 0; k < U; ++k) {
      const long long gi = g + k * T;
      if (gi < n4) {
#pragma unroll
        for (int e = 0; e < 4; ++e) a[k][e] = a[k][e] + dt * (u[k][e] + s * (c[k][e] - u[k][e]));
        *reinterpret_cast<float4*>(x + (gi << 2)) = make_float4(a[k][0], a[k][1], a[k][2], a[k][3]);
      }
    }
  }
  if (blockIdx.x == 0)
    for (long long i = (n4 << 2) + threadIdx.x; i < n; i += blockDim.x) {
      const float c1 = load1<VT>(vc, i), u1 = load1<VT>(vu, i);
      x[i] = x[i] + dt * (u1 + s * (c1 - u1));
    }
}

int launch_cfg_euler(const LaunchCtx& c, float* x, const void* vc, const void* vu, long long n, float s, float dt,
                     const float* t_pair, int v_f32) {
  if (n <= 0) return WAN_OK;
  constexpr int U = 4, TPB = 128;  // the fastest of a sweep of U x threads per block on this part
  long long blocks = ((n >> 2) + (long long)TPB * U - 1) / ((long long)TPB * U);
  const long long cap = (long long)c.num_sms * 32;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  count_launch("cfg_euler", c.stream, true);
  if (v_f32)
    cfg_euler_kernel<float, U><<<(unsigned)blocks, TPB, 0, c.stream>>>(x, static_cast<const float*>(vc),
                                                                      static_cast<const float*>(vu), n, s, dt, t_pair);
  else
    cfg_euler_kernel<bf16, U><<<(unsigned)blocks, TPB, 0, c.stream>>>(x, static_cast<const bf16*>(vc),
                                                                     static_cast<const bf16*>(vu), n, s, dt, t_pair);
  count_launch("cfg_euler", c.stream, false);
  return cudaGetLastError() == cudaSuccess ? WAN_OK : WAN_ERR_CUDA;
}

// ------------------------------------------------------------------ patch gather
// A row of token m = (b, f, i, j) holds latent[b, c, f, 2i+di, 2j+dj] at column
// c*4 + di*2 + dj.  bf16 output keeps the value exactly as a two-term split:
// columns [0, kpad) hold hi = bf16(v), columns [kpad, 2 kpad) hold lo = bf16(v - hi),
// padding columns are zero.  fp32 output has kpad = C*4 columns.
__global__ void patch_gather_kernel(const float* __restrict__ lat, long long lat_bstride, void* __restrict__ A,
                                    int out_f32, int B, int C, int F, int H, int W, int kpad) {
  const int Hp = H >> 1, Wp = W >> 1;
  const long long L = (long long)F * Hp * Wp;
  const long long total = (long long)B * L * C;
  for (long long g = (long long)blockIdx.x * blockDim.x + threadIdx.x; g < total; g += (long long)gridDim.x * blockDim.x) {
    const int c = (int)(g % C);
    const long long m = g / C;
    const int b = (int)(m / L);
    const long long l = m - (long long)b * L;
    const int f = (int)(l / ((long long)Hp * Wp));
    const int i = (int)((l / Wp) % Hp);
    const int j = (int)(l % Wp);
    const float* src = lat + (long long)b * lat_bstride + (((long long)c * F + f) * H + 2 * i) * W + 2 * j;
    const float v[4] = {src[0], src[1], src[W], src[W + 1]};
    if (out_f32) {
      float* row = static_cast<float*>(A) + m * kpad;
#pragma unroll
      for (int k = 0; k < 4; ++k) row[c * 4 + k] = v[k];
    } else {
      bf16* row = static_cast<bf16*>(A) + m * (2LL * kpad);
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const bf16 hi = __float2bfloat16_rn(v[k]);
        row[c * 4 + k] = hi;
        row[kpad + c * 4 + k] = __float2bfloat16_rn(v[k] - bf2f(hi));
      }
      if (c == 0)
        for (int k = C * 4; k < kpad; ++k) {
          row[k] = __float2bfloat16_rn(0.f);
          row[kpad + k] = __float2bfloat16_rn(0.f);
        }
    }
  }
}

int launch_patch_gather(const LaunchCtx& c, const float* latent, long long latent_bstride, void* A, int out_f32,
                        int B, int C, int F, int H, int W, int kpad) {
  const long long total = (long long)B * F * (H / 2) * (W / 2) * C;
  if (total <= 0) return WAN_OK;
  long long blocks = (total + 255) / 256;
  if (blocks > (long long)c.num_sms * 16) blocks = (long long)c.num_sms * 16;
  count_launch("patch_gather", c.stream, true);
  patch_gather_kernel<<<(unsigned)blocks, 256, 0, c.stream>>>(latent, latent_bstride, A, out_f32, B, C, F, H, W,
                                                              kpad);
  count_launch("patch_gather", c.stream, false);
  return cudaGetLastError() == cudaSuccess ? WAN_OK : WAN_ERR_CUDA;
}

// ------------------------------------------------------------------ RoPE frequencies
// omega of pair j of axis a (n_a = d_a / 2 pairs): theta^(-2j/d_a), in double precision.
__global__ void rope_table_kernel(float* omega, RopeGeom g, float theta) {
  const int total = g.nf + g.nh + g.nw;
  for (int e = threadIdx.x; e < total; e += blockDim.x) {
    int j = e, pairs = g.nf;
    if (j >= g.nf) {
      j -= g.nf;
      pairs = g.nh;
      if (j >= g.nh) {
        j -= g.nh;
        pairs = g.nw;
      }
    }
    omega[e] = (float)pow((double)theta, -2.0 * j / (2.0 * pairs));
  }
}

int launch_rope_table(const LaunchCtx& c, float* omega, int head_dim, float theta) {
  RopeGeom g = rope_geom(omega, 1, 1, 1, head_dim);
  count_launch("rope_table", c.stream, true);
  rope_table_kernel<<<1, 128, 0, c.stream>>>(omega, g, theta);
  count_launch("rope_table", c.stream, false);
  return cudaGetLastError() == cudaSuccess ? WAN_OK : WAN_ERR_CUDA;
}

// ------------------------------------------------------------------ time embedding
// s[b] = [cos(tau w_k), sin(tau w_k)], tau = 1000 t[b], w_k = 10000^(-k/half), in double.
__global__ void sinusoid_kernel(const float* t, int t_stride, float* s, int dim) {
  const int b = blockIdx.x;
  const int half = dim / 2;
  const double tau = 1000.0 * (double)t[b * t_stride];
  for (int k = threadIdx.x; k < half; k += blockDim.x) {
    const double a = tau * pow(10000.0, -(double)k / half);
    s[(long long)b * dim + k] = (float)cos(a);
    s[(long long)b * dim + half + k] = (float)sin(a);
  }
}

int launch_sinusoid(const LaunchCtx& c, const float* t, int t_stride, float* s, int B, int dim) {
  count_launch("sinusoid", c.stream, true);
  sinusoid_kernel<<<B, 128, 0, c.stream>>>(t, t_stride, s, dim);
  count_launch("sinusoid", c.stream, false);
  return cudaGetLastError() == cudaSuccess ? WAN_OK : WAN_ERR_CUDA;
}

__device__ __forceinline__ float silu_f(float x) { return x / (1.0f + expf(-x)); }

// One warp per output feature n; lanes stride over K.
__global__ void __launch_bounds__(256) small_linear_kernel(const float* __restrict__ x, const void* __restrict__ W,
                                                           const void* __restrict__ bias, int w_f32,
                                                           float* __restrict__ out, int B, int N, int K,
                                                           int act_in, int act_out) {
  const int n = blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (n >= N) return;
  for (int b = 0; b < B; ++b) {
    float acc = 0.f;
    for (int k = lane; k < K; k += 32) {
      float xv = x[(long long)b * K + k];
      if (act_in) xv = silu_f(xv);
      const float wv = w_f32 ? static_cast<const float*>(W)[(long long)n * K + k]
                             : bf2f(static_cast<const bf16*>(W)[(long long)n * K + k]);
      acc = fmaf(wv, xv, acc);
    }
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if (lane == 0) {
      if (bias) acc += w_f32 ? static_cast<const float*>(bias)[n] : bf2f(static_cast<const bf16*>(bias)[n]);
      if (act_out) acc = silu_f(acc);
      out[(long long)b * N + n] = acc;
    }
  }
}

int launch_small_linear(const LaunchCtx& c, const float* x, const void* W, const void* bias, int w_f32, float* out,
                        int B, int N, int K, int act_in, int act_out) {
  count_launch("time_mlp", c.stream, true);
  small_linear_kernel<<<(N + 7) / 8, 256, 0, c.stream>>>(x, W, bias, w_f32, out, B, N, K, act_in, act_out);
  count_launch("time_mlp", c.stream, false);
  return cudaGetLastError() == cudaSuccess ? WAN_OK : WAN_ERR_CUDA;
}

struct ModPtrs {
  const void* p[64];
};

__global__ void block_mods_kernel(const float* __restrict__ e0, ModPtrs mp, int nblk, int w_f32,
                                  float* __restrict__ mods, int B, int D) {
  const long long per = (long long)B * 6 * D;
  const long long total = per * nblk;
  for (long long g = (long long)blockIdx.x * blockDim.x + threadIdx.x; g < total; g += (long long)gridDim.x * blockDim.x) {
    const int blk = (int)(g / per);
    const long long r = g - blk * per;
    const int b = (int)(r / (6LL * D));
    const int kn = (int)(r - (long long)b * 6 * D);
    const float m = w_f32 ? static_cast<const float*>(mp.p[blk])[kn] : bf2f(static_cast<const bf16*>(mp.p[blk])[kn]);
    mods[g] = e0[(long long)b * 6 * D + kn] + m;
  }
}

int launch_block_mods(const LaunchCtx& c, const float* e0, const void* const* mod_ptrs, int nblk, int w_f32,
                      float* mods, int B, int D) {
  for (int s = 0; s < nblk; s += 64) {
    ModPtrs mp;
    const int n = nblk - s < 64 ? nblk - s : 64;
    for (int i = 0; i < n; ++i) mp.p[i] = mod_ptrs[s + i];
    const long long total = (long long)n * B * 6 * D;
    long long blocks = (total + 255) / 256;
    if (blocks > 4096) blocks = 4096;
    count_launch("block_mods", c.stream, true);
    block_mods_kernel<<<(unsigned)blocks, 256, 0, c.stream>>>(e0, mp, n, w_f32, mods + (long long)s * B * 6 * D, B, D);
    count_launch("block_mods", c.stream, false);
    if (cudaGetLastError() != cudaSuccess) return WAN_ERR_CUDA;
  }
  return WAN_OK;
}

// ------------------------------------------------------------------ layout helpers
template <typename Tin, typename Tout>
__global__ void rope_apply_kernel(const Tin* __restrict__ in, Tout* __restrict__ out, RopeGeom g, long long rows,
                                  int L, int H, int d) {
  const long long pairs_per_row = (long long)H * d / 2;
  const long long total = rows * pairs_per_row;
  for (long long e = (long long)blockIdx.x * blockDim.x + threadIdx.x; e < total; e += (long long)gridDim.x * blockDim.x) {
    const long long m = e / pairs_per_row;
    const int pr = (int)(e - m * pairs_per_row);
    const int l = (int)(m % L);
    const int dd0 = (pr * 2) % d;
    const long long i0 = m * H * d + 2 * pr;
    float v[2];
    if constexpr (sizeof(Tin) == 4) {
      v[0] = in[i0];
      v[1] = in[i0 + 1];
    } else if constexpr (std::is_same<Tin, __half>::value) {
      v[0] = __half2float(in[i0]);
      v[1] = __half2float(in[i0 + 1]);
    } else {
      v[0] = bf2f(in[i0]);
      v[1] = bf2f(in[i0 + 1]);
    }
    epi_rope<2>(g, d, dd0, l, v);
    if constexpr (sizeof(Tout) == 4) {
      out[i0] = v[0];
      out[i0 + 1] = v[1];
    } else {
      out[i0] = __float2half_rn(v[0]);
      out[i0 + 1] = __float2half_rn(v[1]);
    }
  }
}

int launch_rope_apply(const LaunchCtx& c, const void* in, void* out, const RopeGeom& g, int B, int L, int H, int d,
                      int in_type) {
  const long long total = (long long)B * L * H * d / 2;
  if (total <= 0) return WAN_OK;
  long long blocks = (total + 255) / 256;
  if (blocks > (long long)c.num_sms * 16) blocks = (long long)c.num_sms * 16;
  count_launch("rope_apply", c.stream, true);
  if (in_type == OUT_F32)
    rope_apply_kernel<float, float><<<(unsigned)blocks, 256, 0, c.stream>>>(
        static_cast<const float*>(in), static_cast<float*>(out), g, (long long)B * L, L, H, d);
  else if (in_type == OUT_F16)
    rope_apply_kernel<__half, __half><<<(unsigned)blocks, 256, 0, c.stream>>>(
        static_cast<const __half*>(in), static_cast<__half*>(out), g, (long long)B * L, L, H, d);
  else
    rope_apply_kernel<bf16, __half><<<(unsigned)blocks, 256, 0, c.stream>>>(
        static_cast<const bf16*>(in), static_cast<__half*>(out), g, (long long)B * L, L, H, d);
  count_launch("rope_apply", c.stream, false);
  return cudaGetLastError() == cudaSuccess ? WAN_OK : WAN_ERR_CUDA;
}

__global__ void schedule_kernel(float* ts, int steps) {
  for (int k = threadIdx.x; k <= steps; k += blockDim.x) ts[k] = 1.0f - (float)k / (float)steps;
}

int launch_schedule(const LaunchCtx& c, float* ts, int steps) {
  count_launch("schedule", c.stream, true);
  schedule_kernel<<<1, 256, 0, c.stream>>>(ts, steps);
  count_launch("schedule", c.stream, false);
  return cudaGetLastError() == cudaSuccess ? WAN_OK : WAN_ERR_CUDA;
}

// ------------------------------------------------------------------ watchdog self-test
// One thread waits, through the same bounded wait every pipeline uses, on an mbarrier
// that nothing ever arrives on; after limit_ns it records a timeout in the device status
// word and returns.  Exercises the failure path without faulting or hanging the GPU.
__global__ void watchdog_selftest_kernel(unsigned long long limit_ns, int* status) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_barrier_init();
    mbar_wait_for(&bar, 0, status, kDevTimeoutSelftest, limit_ns);
  }
}

int launch_watchdog_selftest(const LaunchCtx& c, unsigned long long limit_ns) {
  count_launch("watchdog_selftest", c.stream, true);
  watchdog_selftest_kernel<<<1, 32, 0, c.stream>>>(limit_ns, c.dev_status);
  count_launch("watchdog_selftest", c.stream, false);
  return cudaGetLastError() == cudaSuccess ? WAN_OK : WAN_ERR_CUDA;
}

// ------------------------------------------------------------------ q/k RMSNorm + RoPE (variant)
// One 128-thread CTA per token row of the q | k | v buffer: for q (columns [0, D)) and k
// ([D, 2D)): x <- RoPE(x * rsqrt(mean(x^2) + eps) * w), in place, fp32 statistics.
template <typename T>
__device__ __forceinline__ float2 ld2(const T* p) {
  if constexpr (sizeof(T) == 4) return make_float2(p[0], p[1]);
  else return __half22float2(*reinterpret_cast<const __half2*>(p));
}
template <typename T>
__device__ __forceinline__ void st2(T* p, float2 v) {
  if constexpr (sizeof(T) == 4) { p[0] = v.x; p[1] = v.y; }
  else *reinterpret_cast<__half2*>(p) = __floats2half2_rn(v.x, v.y);
}

template <typename T, typename WT>
__global__ void __launch_bounds__(128) qk_rmsnorm_rope_kernel(T* __restrict__ qkv, long long ld, const WT* __restrict__ wq,
                                                              const WT* __restrict__ wk, RopeGeom g, int L, int D,
                                                              int hd, float eps) {
  __shared__ float red[2][4];
  const long long row = blockIdx.x;
  const int l = (int)(row % L);
  const int t = threadIdx.x;
  T* base = qkv + row * ld;
  float s[2] = {0.f, 0.f};
  for (int part = 0; part < 2; ++part)
    for (int c = 2 * t; c < D; c += 256) {
      const float2 v = ld2(base + part * D + c);
      s[part] += v.x * v.x + v.y * v.y;
    }
#pragma unroll
  for (int part = 0; part < 2; ++part) {
    float a = s[part];
    for (int o = 16; o > 0; o >>= 1) a += __shfl_xor_sync(0xffffffffu, a, o);
    if ((t & 31) == 0) red[part][t >> 5] = a;
  }
  __syncthreads();
  float r[2];
#pragma unroll
  for (int part = 0; part < 2; ++part)
    r[part] = rsqrtf(((red[part][0] + red[part][1]) + (red[part][2] + red[part][3])) / (float)D + eps);
  for (int part = 0; part < 2; ++part) {
    const WT* w = part ? wk : wq;
    for (int c = 2 * t; c < D; c += 256) {
      float2 v = ld2(base + part * D + c);
      float x[2];
      if constexpr (sizeof(WT) == 4) {
        x[0] = v.x * r[part] * w[c];
        x[1] = v.y * r[part] * w[c + 1];
      } else {
        x[0] = v.x * r[part] * bf2f(w[c]);
        x[1] = v.y * r[part] * bf2f(w[c + 1]);
      }
      epi_rope<2>(g, hd, c % hd, l, x);
      st2(base + part * D + c, make_float2(x[0], x[1]));
    }
  }
}

int launch_qk_rmsnorm_rope(const LaunchCtx& c, void* qkv, long long ld, const void* wq, const void* wk, const RopeGeom& g,
                           int rows, int L, int D, int hd, float eps, int f32) {
  if (rows <= 0) return WAN_OK;
  count_launch("qk_rmsnorm_rope", c.stream, true);
  if (f32)
    qk_rmsnorm_rope_kernel<float, float><<<rows, 128, 0, c.stream>>>(
        static_cast<float*>(qkv), ld, static_cast<const float*>(wq), static_cast<const float*>(wk), g, L, D, hd, eps);
  else
    qk_rmsnorm_rope_kernel<__half, bf16><<<rows, 128, 0, c.stream>>>(
        static_cast<__half*>(qkv), ld, static_cast<const bf16*>(wq), static_cast<const bf16*>(wk), g, L, D, hd, eps);
  count_launch("qk_rmsnorm_rope", c.stream, false);
  return cudaGetLastError() == cudaSuccess ? WAN_OK : WAN_ERR_CUDA;
}

}  // namespace wan

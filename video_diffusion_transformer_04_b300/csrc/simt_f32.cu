// fp32 parity path: the same projections and attention in plain fp32 SIMT arithmetic
// (no tensor cores; tf32 would not meet a 1e-4 relative bound).  Used when a call asks
// for WAN_F32; shapes of any size are handled, speed is not a goal.
#include "kernels.h"

namespace wan {

// C[M, N] = A[M, K] * B[N, K]^T, 64x64 tiles, 4x4 outputs per thread.
__global__ void __launch_bounds__(256) gemm_f32_kernel(const float* __restrict__ A, long long lda,
                                                       const float* __restrict__ B, long long ldb, int M, int N,
                                                       int K, const EpiParams ep) {
  __shared__ float As[16][64 + 4];
  __shared__ float Bs[16][64 + 4];
  const int row0 = blockIdx.y * 64, col0 = blockIdx.x * 64;
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  float acc[4][4] = {};
  for (int k0 = 0; k0 < K; k0 += 16) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int idx = threadIdx.x + i * 256;
      const int r = idx >> 4, kk = idx & 15;
      As[kk][r] = (row0 + r < M && k0 + kk < K) ? A[(long long)(row0 + r) * lda + k0 + kk] : 0.f;
      Bs[kk][r] = (col0 + r < N && k0 + kk < K) ? B[(long long)(col0 + r) * ldb + k0 + kk] : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < 16; ++kk) {
      float a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        a[i] = As[kk][ty * 4 + i];
        b[i] = Bs[kk][tx * 4 + i];
      }
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    __syncthreads();
  }
  const int n0 = col0 + tx * 4;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int m = row0 + ty * 4 + i;
    if (m < M && n0 < N) epilogue_chunk<4>(ep, m, n0, acc[i]);
  }
}

int gemm_f32(const LaunchCtx& c, const float* A, long long lda, const float* B, long long ldb, int M, int N, int K,
             const EpiParams& ep, const char* tag) {
  if (M <= 0 || N <= 0) return WAN_OK;
  dim3 grid((N + 63) / 64, (M + 63) / 64);
  count_launch(tag, c.stream, true);
  gemm_f32_kernel<<<grid, 256, 0, c.stream>>>(A, lda, B, ldb, M, N, K, ep);
  count_launch(tag, c.stream, false);
  return cudaGetLastError() == cudaSuccess ? WAN_OK : WAN_ERR_CUDA;
}

// One warp per query row; each lane runs an online softmax over keys lane, lane+32, ...
// and the lanes' partial results are merged at the end.
__global__ void __launch_bounds__(256) attn_f32_kernel(const AttnArgs a, float scale) {
  __shared__ float sq[8][128];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int row = blockIdx.x * 8 + warp;
  const int bh = blockIdx.y;
  const int b = bh / a.H, h = bh - (bh / a.H) * a.H;
  const int hd = a.head_dim;
  const float* q = static_cast<const float*>(a.q);
  const float* k = static_cast<const float*>(a.k);
  const float* vv = static_cast<const float*>(a.v);
  if (row < a.Lq)
    for (int d = lane; d < hd; d += 32) sq[warp][d] = q[((long long)b * a.Lq + row) * a.ldq + a.q_col + h * hd + d];
  __syncwarp();
  if (row >= a.Lq) return;
  const int lkv = a.kv_lens ? min(max(a.kv_lens[b], 1), a.Lkv) : a.Lkv;
  float m = -INFINITY, l = 0.f;
  float acc[128];
  for (int d = 0; d < hd; ++d) acc[d] = 0.f;
  for (int j = lane; j < lkv; j += 32) {
    const float* kr = k + ((long long)b * a.Lkv + j) * a.ldk + a.k_col + h * hd;
    float s = 0.f;
    for (int d = 0; d < hd; ++d) s = fmaf(sq[warp][d], kr[d], s);
    s *= scale;
    const float mn = fmaxf(m, s);
    const float corr = expf(m - mn);
    const float pj = expf(s - mn);
    l = l * corr + pj;
    const float* vr = vv + ((long long)b * a.Lkv + j) * a.ldv + a.v_col + h * hd;
    for (int d = 0; d < hd; ++d) acc[d] = fmaf(pj, vr[d], acc[d] * corr);
    m = mn;
  }
  float M = m;
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  const float f = (m == -INFINITY) ? 0.f : expf(m - M);
  float lt = l * f;
  for (int o = 16; o > 0; o >>= 1) lt += __shfl_xor_sync(0xffffffffu, lt, o);
  float* out = static_cast<float*>(a.o) + ((long long)b * a.Lq + row) * a.ldo + a.o_col + h * hd;
  for (int d = 0; d < hd; ++d) {
    float v = acc[d] * f;
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if (lane == (d & 31)) out[d] = (a.accumulate ? out[d] : 0.f) + v / lt;
  }
}

int attention_f32(const LaunchCtx& c, const AttnArgs& a) {
  if (a.head_dim > 128 || (a.head_dim & 1)) return WAN_ERR_UNSUPPORTED;
  if (a.Lq <= 0 || a.Lkv <= 0) return WAN_OK;
  dim3 grid((a.Lq + 7) / 8, a.B * a.H);
  count_launch(a.tag ? a.tag : "attn", c.stream, true);
  attn_f32_kernel<<<grid, 256, 0, c.stream>>>(a, 1.0f / sqrtf((float)a.head_dim));
  count_launch(a.tag ? a.tag : "attn", c.stream, false);
  return cudaGetLastError() == cudaSuccess ? WAN_OK : WAN_ERR_CUDA;
}

}  // namespace wan

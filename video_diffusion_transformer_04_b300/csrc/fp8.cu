// 8-bit (OCP FP8 E4M3) operands and the 8-bit self-attention of the DiT's FP8 variant
// ("FP8 GEMM and 8-bit FlashAttention" of the Method section's inference paragraph).
//
// Quantisation, decided in fp32 like its CPU definition: per group
//   amax = max |x|, inv = 448 / amax (IEEE division), code = e4m3_rn_satfinite(x * inv),
//   dequantisation scale s = amax / 448; an all-zero group has inv = s = 0.
// Groups: GEMM activations per row (token), GEMM weights per row (output channel);
// attention q per (token, head), k per (head, block of 128 keys), v per (head, channel)
// over all keys.  v is stored transposed, [B, H, d, Lp] with Lp = L rounded up to 16,
// keys contiguous, so that the PV product reads it as a K-major operand like every
// other tile.
//
// Attention (attn_e4m3_tc_kernel): the bf16 kernel's structure (two 128-row query
// tiles per CTA, TMA / MMA / two softmax warpgroups, S and O of each tile in TMEM) on
// 8-bit operands: S = Q8 K8^T and O += P8 V8 by tcgen05.mma kind::f8f6f4, K = 32 per
// instruction, so each 128-key step takes half the MMA instructions of the bf16 kernel.
// Issue order per key tile j: PV_0(j), S_0(j+1) | wait P_1(j) | PV_1(j), S_1(j+1): each
// tile's cycle is its own MMAs plus its softmax, the two tiles half a cycle apart.
// Softmax per row, fp32: the logit of key j is S_j * c with c = log2(e)/sqrt(d) * sq_row *
// sk_block; P' = 2^(S_j c - m + 8) is rounded to E4M3 into TMEM (four keys per 32-bit
// column) and the row sum accumulates the unrounded P'; O = (sum_j P'_j V8_j) * sv / l.
// The reference max m is lazy: it moves (rescaling O and l) only when a tile's row max
// exceeds it by more than 0.75 (log2), which keeps every P' <= 2^8.75 < 448.
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "kernels.h"

namespace wan {

// ------------------------------------------------------------------ E4M3 helpers
template <typename T>
__device__ __forceinline__ float2 ld2(const T* p);
template <>
__device__ __forceinline__ float2 ld2<bf16>(const bf16* p) {
  return unpack_bf16x2(*reinterpret_cast<const uint32_t*>(p));
}
template <>
__device__ __forceinline__ float2 ld2<__half>(const __half* p) {
  return __half22float2(*reinterpret_cast<const __half2*>(p));
}
template <>
__device__ __forceinline__ float2 ld2<float>(const float* p) {
  return *reinterpret_cast<const float2*>(p);
}

template <typename T, int E>
__device__ __forceinline__ void ld_vec(const T* p, float (&v)[E]) {
#pragma unroll
  for (int e = 0; e < E; e += 2) {
    const float2 f = ld2<T>(p + e);
    v[e] = f.x;
    v[e + 1] = f.y;
  }
}
template <int E>
__device__ __forceinline__ void st_codes(uint8_t* dst, const float (&v)[E], float inv) {
  if constexpr (E == 4) {
    *reinterpret_cast<uint32_t*>(dst) =
        e4m3x4(__fmul_rn(v[0], inv), __fmul_rn(v[1], inv), __fmul_rn(v[2], inv), __fmul_rn(v[3], inv));
  } else {
    *reinterpret_cast<uint16_t*>(dst) = (uint16_t)e4m3x2(__fmul_rn(v[0], inv), __fmul_rn(v[1], inv));
  }
}
__device__ __forceinline__ float warp_max(float a) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
  return a;
}

// ------------------------------------------------------------------ quantisers
// Rows of K elements (K % 4 == 0): one 128-thread CTA per row, two passes over the row.
template <typename T>
__global__ void __launch_bounds__(128) quant_rows_kernel(const T* __restrict__ x, long long ldx, int K,
                                                         uint8_t* __restrict__ x8, long long ld8,
                                                         float* __restrict__ s) {
  __shared__ float red[4];
  const long long row = blockIdx.x;
  const T* src = x + row * ldx;
  float a = 0.f;
  for (int k = threadIdx.x * 4; k < K; k += 128 * 4) {
    float v[4];
    ld_vec<T, 4>(src + k, v);
    a = fmaxf(fmaxf(a, fmaxf(fabsf(v[0]), fabsf(v[1]))), fmaxf(fabsf(v[2]), fabsf(v[3])));
  }
  a = warp_max(a);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = a;
  __syncthreads();
  a = fmaxf(fmaxf(red[0], red[1]), fmaxf(red[2], red[3]));
  const float inv = e4m3_inv(a);
  for (int k = threadIdx.x * 4; k < K; k += 128 * 4) {
    float v[4];
    ld_vec<T, 4>(src + k, v);
    st_codes<4>(x8 + row * ld8 + k, v, inv);
  }
  if (threadIdx.x == 0) s[row] = e4m3_deq(a);
}

// q: one warp per (token row, head); lane holds HD/32 consecutive elements.
template <typename T, int HD>
__global__ void __launch_bounds__(256) quant_q_kernel(const T* __restrict__ x, long long ldx, int col0,
                                                      uint8_t* __restrict__ q8, long long ld8,
                                                      float* __restrict__ s, long long rows, int H) {
  constexpr int E = HD / 32;
  const long long g = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (g >= rows * H) return;
  const long long row = g / H;
  const int h = (int)(g - row * H);
  float v[E];
  ld_vec<T, E>(x + row * ldx + col0 + h * HD + lane * E, v);
  float a = 0.f;
#pragma unroll
  for (int e = 0; e < E; ++e) a = fmaxf(a, fabsf(v[e]));
  a = warp_max(a);
  st_codes<E>(q8 + row * ld8 + h * HD + lane * E, v, e4m3_inv(a));
  if (lane == 0) s[row * H + h] = e4m3_deq(a);
}

// k: one 256-thread CTA per (128-key block, head, batch entry); warp w takes keys
// 16w .. 16w+15 of the block, lane E consecutive elements of each.
template <typename T, int HD>
__global__ void __launch_bounds__(256) quant_k_kernel(const T* __restrict__ x, long long ldx, int col0,
                                                      uint8_t* __restrict__ k8, long long ld8,
                                                      float* __restrict__ s, int L, int H, int nkb) {
  constexpr int E = HD / 32;
  __shared__ float red[8];
  const int kb = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float v[16][E];
  float a = 0.f;
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const int key = kb * 128 + warp * 16 + i;
    if (key < L) {
      ld_vec<T, E>(x + ((long long)b * L + key) * ldx + col0 + h * HD + lane * E, v[i]);
    } else {
#pragma unroll
      for (int e = 0; e < E; ++e) v[i][e] = 0.f;
    }
#pragma unroll
    for (int e = 0; e < E; ++e) a = fmaxf(a, fabsf(v[i][e]));
  }
  a = warp_max(a);
  if (lane == 0) red[warp] = a;
  __syncthreads();
  a = red[0];
#pragma unroll
  for (int w = 1; w < 8; ++w) a = fmaxf(a, red[w]);
  const float inv = e4m3_inv(a);
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const int key = kb * 128 + warp * 16 + i;
    if (key < L) st_codes<E>(k8 + ((long long)b * L + key) * ld8 + h * HD + lane * E, v[i], inv);
  }
  if (threadIdx.x == 0) s[((long long)b * H + h) * nkb + kb] = e4m3_deq(a);
}

// v, pass 1: per-channel |max| of each 128-key block, merged over blocks by an atomic
// max on the float bits (non-negative floats order like their bit patterns) into
// amax[b, h, c], which the caller zeroes first.
template <typename T, int HD>
__global__ void __launch_bounds__(256) v_amax_kernel(const T* __restrict__ x, long long ldx, int col0,
                                                     unsigned int* __restrict__ amax, int L, int H) {
  constexpr int E = HD / 32;
  __shared__ float red[8][HD];
  const int kb = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float m[E];
#pragma unroll
  for (int e = 0; e < E; ++e) m[e] = 0.f;
#pragma unroll 4
  for (int i = 0; i < 16; ++i) {
    const int key = kb * 128 + warp * 16 + i;
    if (key < L) {
      float v[E];
      ld_vec<T, E>(x + ((long long)b * L + key) * ldx + col0 + h * HD + lane * E, v);
#pragma unroll
      for (int e = 0; e < E; ++e) m[e] = fmaxf(m[e], fabsf(v[e]));
    }
  }
#pragma unroll
  for (int e = 0; e < E; ++e) red[warp][lane * E + e] = m[e];
  __syncthreads();
  for (int c = threadIdx.x; c < HD; c += 256) {
    float a = red[0][c];
#pragma unroll
    for (int w = 1; w < 8; ++w) a = fmaxf(a, red[w][c]);
    atomicMax(amax + ((long long)b * H + h) * HD + c, __float_as_uint(a));
  }
}

// v, pass 2: quantise a 128-key block with its channel scales and store it transposed,
// v8t[b, h, c, key] (row length Lp); block 0 of each (b, h) also writes sv[b, h, c].
// Codes go to shared memory in the natural [key][channel] order (one 32-bit store per
// lane), then each 16-byte chunk of a channel row is gathered byte by byte and stored,
// eight lanes per 128-byte row.
template <typename T, int HD>
__global__ void __launch_bounds__(256) quant_vt_kernel(const T* __restrict__ x, long long ldx, int col0,
                                                       const unsigned int* __restrict__ amax,
                                                       uint8_t* __restrict__ v8t, float* __restrict__ sv, int L,
                                                       int Lp, int H) {
  constexpr int E = HD / 32;
  __shared__ __align__(16) uint8_t tile[128][HD];
  __shared__ float inv_c[HD];
  const int kb = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long bh = (long long)b * H + h;
  for (int c = threadIdx.x; c < HD; c += 256) {
    const float a = __uint_as_float(amax[bh * HD + c]);
    inv_c[c] = e4m3_inv(a);
    if (kb == 0) sv[bh * HD + c] = e4m3_deq(a);
  }
  __syncthreads();
#pragma unroll 4
  for (int i = 0; i < 16; ++i) {
    const int kl = warp * 16 + i;
    const int key = kb * 128 + kl;
    float v[E];
    if (key < L) {
      ld_vec<T, E>(x + ((long long)b * L + key) * ldx + col0 + h * HD + lane * E, v);
    } else {
#pragma unroll
      for (int e = 0; e < E; ++e) v[e] = 0.f;
    }
    float q[E];
#pragma unroll
    for (int e = 0; e < E; ++e) q[e] = __fmul_rn(v[e], inv_c[lane * E + e]);
    if constexpr (E == 4) {
      *reinterpret_cast<uint32_t*>(&tile[kl][lane * 4]) = e4m3x4(q[0], q[1], q[2], q[3]);
    } else {
      *reinterpret_cast<uint16_t*>(&tile[kl][lane * 2]) = (uint16_t)e4m3x2(q[0], q[1]);
    }
  }
  __syncthreads();
  for (int task = threadIdx.x; task < HD * 8; task += 256) {
    const int r = task >> 3, ch = task & 7;
    const int k0 = kb * 128 + ch * 16;
    if (k0 >= Lp) continue;
    uint32_t w[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int kl = ch * 16 + q * 4;
      w[q] = (uint32_t)tile[kl][r] | ((uint32_t)tile[kl + 1][r] << 8) | ((uint32_t)tile[kl + 2][r] << 16) |
             ((uint32_t)tile[kl + 3][r] << 24);
    }
    *reinterpret_cast<uint4*>(v8t + (bh * HD + r) * Lp + k0) = make_uint4(w[0], w[1], w[2], w[3]);
  }
}

// ------------------------------------------------------------------ 8-bit attention
template <int HD>
struct Attn8Cfg {
  static constexpr int BQ = 128;
  static constexpr int BKV = 128;
  static constexpr int TILE = 128 * HD;  // bytes of a 128-row E4M3 tile: one 128-byte swizzle box
  static constexpr int STAGES = 3;       // K and V ring depth
  static constexpr int SMEM_TILES = 2 * TILE + STAGES * 2 * TILE;
  static constexpr int SMEM = SMEM_TILES + 256 + 1024;
  static constexpr int TMEM_COLS = 512;
  static constexpr int THREADS = 384;
  static constexpr int PRODUCER_REGS = 56;
  static constexpr int SOFTMAX_REGS = 224;
  static_assert(128 * PRODUCER_REGS + 256 * SOFTMAX_REGS <= 384 * 168, "register split");
  static_assert(HD == 128, "one 128-byte swizzle row per tile row");
};

struct Attn8Params {
  int Lq, Lkv, H, nkb;
  int nq_pairs;
  float scale_log2;       // log2(e) / sqrt(d)
  const float* sq;        // [B, Lq, H]
  const float* sk;        // [B, H, nkb]
  const float* sv;        // [B, H, d]
  bf16* o;                // [B, Lq, ldo], head h at columns o_col + h*d
  long long ldo;
  int o_col;
  const int* kv_lens;     // [B] or NULL
};

// A tile's row max exceeding the reference by more than this (log2 units) moves the
// reference: P' = 2^(x - m + 8) then stays <= 2^8.75 = 430.5 < 448.
constexpr float kLazyMaxStep = 0.75f;

template <int HD>
__global__ void __launch_bounds__(384, 1)
    attn_e4m3_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                        const __grid_constant__ CUtensorMap tmV, const Attn8Params p, int* status) {
  using Cfg = Attn8Cfg<HD>;
  constexpr int ST = Cfg::STAGES;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem;                    // [2][TILE]
  uint8_t* sK = sQ + 2 * Cfg::TILE;      // [ST][TILE]
  uint8_t* sV = sK + ST * Cfg::TILE;     // [ST][TILE] (V^T: d rows of 128 keys)
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Cfg::SMEM_TILES);
  uint64_t* q_full = bars;
  uint64_t* k_full = bars + 1;
  uint64_t* k_empty = k_full + ST;
  uint64_t* v_full = k_empty + ST;
  uint64_t* v_empty = v_full + ST;
  uint64_t* s_full = v_empty + ST;  // [2]
  uint64_t* p_ready = s_full + 2;   // [2]
  uint64_t* drain = p_ready + 2;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(drain + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int bh = blockIdx.x / p.nq_pairs;
  const int qp = blockIdx.x - bh * p.nq_pairs;
  const int b = bh / p.H;
  const int h = bh - b * p.H;
  const int q0 = qp * 256;
  const int ntile = (q0 + 128 < p.Lq) ? 2 : 1;
  const int lkv = p.kv_lens ? min(max(p.kv_lens[b], 1), p.Lkv) : p.Lkv;
  const int nkv = (lkv + Cfg::BKV - 1) / Cfg::BKV;

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < ST; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&k_empty[s], 1);
      mbar_init(&v_full[s], 1);
      mbar_init(&v_empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&p_ready[i], 4);  // one arrival per softmax warp
    }
    mbar_init(drain, 1);
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_holder, Cfg::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;

  if (warp < 4) {
  regs_dec<Cfg::PRODUCER_REGS>();
  if (warp == 0 && lane == 0) {
    // ---------------------------------------------------------------- TMA producer
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
    mbar_arrive_expect_tx(q_full, ntile * Cfg::TILE);
    for (int i = 0; i < ntile; ++i) tma_load_3d(sQ + i * Cfg::TILE, &tmQ, q_full, h * HD, q0 + i * 128, b);
    uint32_t kissued = 0, vissued = 0;
    bool ok = true;
    for (int j = 0; j < nkv && ok; ++j) {
      const int s = j % ST;
      const uint32_t ph = (j / ST) & 1;
      if (!mbar_wait(&k_empty[s], ph ^ 1, status, kDevTimeoutAttn8)) { ok = false; break; }
      mbar_arrive_expect_tx(&k_full[s], Cfg::TILE);
      tma_load_3d(sK + s * Cfg::TILE, &tmK, &k_full[s], h * HD, j * Cfg::BKV, b);
      kissued = j + 1;
      if (!mbar_wait(&v_empty[s], ph ^ 1, status, kDevTimeoutAttn8)) { ok = false; break; }
      mbar_arrive_expect_tx(&v_full[s], Cfg::TILE);
      tma_load_2d(sV + s * Cfg::TILE, &tmV, &v_full[s], j * Cfg::BKV, bh * HD);
      vissued = j + 1;
    }
    if (!ok) {  // error path: let issued copies land
      const unsigned long long t0 = globaltimer_ns();
      for (uint32_t j = (kissued > ST ? kissued - ST : 0); j < kissued; ++j)
        while (!mbar_test(&k_full[j % ST], (j / ST) & 1) && globaltimer_ns() - t0 < kWaitLimitNs) {}
      for (uint32_t j = (vissued > ST ? vissued - ST : 0); j < vissued; ++j)
        while (!mbar_test(&v_full[j % ST], (j / ST) & 1) && globaltimer_ns() - t0 < kWaitLimitNs) {}
      while (!mbar_test(q_full, 0) && globaltimer_ns() - t0 < kWaitLimitNs) {}
    }
  } else if (warp == 1 && lane == 0) {
    // ---------------------------------------------------------------- MMA issuer
    constexpr uint32_t idS = make_idesc_e4m3(128, Cfg::BKV);
    constexpr uint32_t idO = make_idesc_e4m3(128, HD);
    constexpr uint32_t kTileLo = Cfg::TILE >> 4;  // descriptor start-address step of one tile
    bool ok = mbar_wait(q_full, 0, status, kDevTimeoutAttn8) && mbar_wait(&k_full[0], 0, status, kDevTimeoutAttn8);
    const uint32_t q_lo0 = sdesc_sw128_lo(smem_u32(sQ));
    const uint32_t k_lo0 = sdesc_sw128_lo(smem_u32(sK));
    const uint32_t v_lo0 = sdesc_sw128_lo(smem_u32(sV));
    // 32 bytes (one K = 32 step of 8-bit operands) = 2 in descriptor units.
    auto issue_S = [&](int i, int ks) {
      const uint32_t qa = q_lo0 + i * kTileLo, ka = k_lo0 + ks * kTileLo;
      const uint32_t d = tmem_base + i * 256;
#pragma unroll
      for (int kk = 0; kk < HD / 32; ++kk) tc_mma_ss_f8_lo(d, qa + kk * 2, ka + kk * 2, idS, kk > 0 ? 1u : 0u);
    };
    // P: 128 keys as E4M3, four per TMEM column -> 8 columns per K = 32 step.
    auto issue_PV = [&](int i, int vs, uint32_t acc) {
      const uint32_t va = v_lo0 + vs * kTileLo;
      const uint32_t d = tmem_base + i * 256 + 128;
      const uint32_t pa = tmem_base + i * 256;
#pragma unroll
      for (int kk = 0; kk < Cfg::BKV / 32; ++kk)
        tc_mma_ts_f8_lo(d, pa + kk * 8, va + kk * 2, idO, (acc | (uint32_t)kk) != 0 ? 1u : 0u);
    };
    if (ok) {
      tc_fence_after();
      for (int i = 0; i < ntile; ++i) {
        issue_S(i, 0);
        tc_commit(&s_full[i]);
      }
      tc_commit(&k_empty[0]);
    }
    for (int j = 0; j < nkv && ok; ++j) {
      const int vs = j % ST;
      const int ks = (j + 1) % ST;
      const bool more = j + 1 < nkv;
      if (!mbar_wait(&v_full[vs], (j / ST) & 1, status, kDevTimeoutAttn8)) { ok = false; break; }
      if (more && !mbar_wait(&k_full[ks], ((j + 1) / ST) & 1, status, kDevTimeoutAttn8)) { ok = false; break; }
      if (!mbar_wait(&p_ready[0], j & 1, status, kDevTimeoutAttn8)) { ok = false; break; }
      tc_fence_after();
      // Tile 0's next scores right behind its PV product: its softmax can start as soon
      // as these finish, independently of tile 1 (the tensor pipe runs them in order, so
      // S_0(j+1) overwrites P_0 only after PV_0(j) has read it).
      issue_PV(0, vs, j > 0 ? 1u : 0u);
      if (more) issue_S(0, ks);
      tc_commit(&s_full[0]);
      if (ntile == 2) {
        if (!mbar_wait(&p_ready[1], j & 1, status, kDevTimeoutAttn8)) { ok = false; break; }
        tc_fence_after();
        issue_PV(1, vs, j > 0 ? 1u : 0u);
        tc_commit(&v_empty[vs]);
        if (more) {
          issue_S(1, ks);
          tc_commit(&k_empty[ks]);
        }
        tc_commit(&s_full[1]);
      } else {
        tc_commit(&v_empty[vs]);
        if (more) tc_commit(&k_empty[ks]);
      }
    }
    if (!ok) {
      tc_commit(drain);
      const unsigned long long t0 = globaltimer_ns();
      while (!mbar_test(drain, 0) && globaltimer_ns() - t0 < kWaitLimitNs) {}
    }
  }
  } else {
    // ---------------------------------------------------------------- softmax
    regs_inc<Cfg::SOFTMAX_REGS>();
    const int i = (warp - 4) >> 2;
    const int quad = warp & 3;
    if (i < ntile) {
      const uint32_t tS = tmem_base + ((uint32_t)(quad * 32) << 16) + i * 256;
      const uint32_t tO = tS + 128;
      const int qrow = q0 + i * 128 + quad * 32 + lane;
      const float sq = qrow < p.Lq ? p.sq[((long long)b * p.Lq + qrow) * p.H + h] : 0.f;
      const float c_row = p.scale_log2 * sq;
      const float* skp = p.sk + (long long)bh * p.nkb;
      float m_used = -INFINITY;  // reference max of the scaled logits (log2 units)
      float l_sum = 0.f;         // sum of P' (unrounded)
      bool ok = true;
      uint32_t sr[Cfg::BKV];
      auto load_scores = [&](int valid) {
#pragma unroll
        for (int c = 0; c < 4; ++c) tmem_ld32_nowait(tS + c * 32, sr + c * 32);
        tmem_wait_ld();
        if (valid < Cfg::BKV) {
#pragma unroll
          for (int e = 0; e < Cfg::BKV; ++e)
            if (e >= valid) sr[e] = __float_as_uint(-INFINITY);
        }
      };
      auto row_max = [&]() -> float {
        float mx0 = __uint_as_float(sr[0]), mx1 = __uint_as_float(sr[1]);
        float mx2 = __uint_as_float(sr[2]), mx3 = __uint_as_float(sr[3]);
#pragma unroll
        for (int e = 4; e < Cfg::BKV - 4; e += 8) {
          mx0 = fmax3(mx0, __uint_as_float(sr[e]), __uint_as_float(sr[e + 1]));
          mx1 = fmax3(mx1, __uint_as_float(sr[e + 2]), __uint_as_float(sr[e + 3]));
          mx2 = fmax3(mx2, __uint_as_float(sr[e + 4]), __uint_as_float(sr[e + 5]));
          mx3 = fmax3(mx3, __uint_as_float(sr[e + 6]), __uint_as_float(sr[e + 7]));
        }
        mx0 = fmax3(mx0, __uint_as_float(sr[Cfg::BKV - 4]), __uint_as_float(sr[Cfg::BKV - 3]));
        mx1 = fmax3(mx1, __uint_as_float(sr[Cfg::BKV - 2]), __uint_as_float(sr[Cfg::BKV - 1]));
        return fmax3(mx0, mx1, fmaxf(mx2, mx3));
      };
      float sk_next = skp[0];
      for (int j = 0; j < nkv; ++j) {
        const float skj = sk_next;
        if (j + 1 < nkv) sk_next = skp[j + 1];
        if (!mbar_wait_warp(&s_full[i], j & 1, status, kDevTimeoutAttn8)) { ok = false; break; }
        tc_fence_after();
        const int valid = lkv - j * Cfg::BKV;  // >= 1
        load_scores(valid);
        // c > 0 always, so that a masked -inf logit stays -inf (never -inf * 0).
        const float c = fmaxf(c_row * skj, 1e-30f);
        const float mt = row_max() * c;
        if (j == 0) {
          m_used = mt;
        } else {
          const bool need = mt > m_used + kLazyMaxStep;
          if (__any_sync(0xffffffffu, need)) {
            const float alpha = need ? ex2_approx(m_used - mt) : 1.0f;
            l_sum *= alpha;
            if (need) m_used = mt;
#pragma unroll 1
            for (int cc = 0; cc < HD / 32; ++cc) {
              uint32_t orr[32];
              tmem_ld32(tO + cc * 32, orr);
#pragma unroll
              for (int e = 0; e < 32; ++e) orr[e] = __float_as_uint(__uint_as_float(orr[e]) * alpha);
              tmem_st32(tO + cc * 32, orr);
            }
          }
        }
        // P' = 2^(s c - (m - 8)) on packed pairs; four E4M3 codes per 32-bit word written
        // over the already-consumed front of sr (word w <= element 4w).
        const uint64_t c2 = f2_pack(c, c);
        const float nm = 8.0f - m_used;
        const uint64_t nm2 = f2_pack(nm, nm);
        uint64_t acc0 = 0, acc1 = 0;
#pragma unroll
        for (int w = 0; w < Cfg::BKV / 4; ++w) {
          const float2 t01 = f2_unpack(f2_fma(f2_pack(__uint_as_float(sr[4 * w]), __uint_as_float(sr[4 * w + 1])), c2, nm2));
          const float2 t23 = f2_unpack(f2_fma(f2_pack(__uint_as_float(sr[4 * w + 2]), __uint_as_float(sr[4 * w + 3])), c2, nm2));
          const float p0 = ex2_approx(t01.x), p1 = ex2_approx(t01.y);
          const float p2 = ex2_approx(t23.x), p3 = ex2_approx(t23.y);
          sr[w] = e4m3x4(p0, p1, p2, p3);
          acc0 = f2_add(acc0, f2_pack(p0, p1));
          acc1 = f2_add(acc1, f2_pack(p2, p3));
        }
        const float2 rs = f2_unpack(f2_add(acc0, acc1));
        tmem_st32_nowait(tS, sr);
        tmem_wait_st();
        l_sum += rs.x + rs.y;
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&p_ready[i]);
      }
      if (ok && mbar_wait_warp(&s_full[i], nkv & 1, status, kDevTimeoutAttn8)) {
        tc_fence_after();
        const float inv = 1.0f / l_sum;
        const float* svp = p.sv + (long long)bh * HD;
        bf16* orow = p.o + ((long long)b * p.Lq + qrow) * p.ldo + p.o_col + h * HD;
#pragma unroll 1
        for (int cc = 0; cc < HD / 32; ++cc) {
          uint32_t orr[32];
          tmem_ld32(tO + cc * 32, orr);
          if (qrow < p.Lq) {
            uint4* dst = reinterpret_cast<uint4*>(orow + cc * 32);
            const float4* s4 = reinterpret_cast<const float4*>(svp + cc * 32);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float4 sa = s4[2 * e], sb = s4[2 * e + 1];
              const float sc[8] = {sa.x, sa.y, sa.z, sa.w, sb.x, sb.y, sb.z, sb.w};
              float v[8];
#pragma unroll
              for (int u = 0; u < 8; ++u) v[u] = __uint_as_float(orr[e * 8 + u]) * (sc[u] * inv);
              uint4 o4;
              o4.x = pack_bf16x2(v[0], v[1]);
              o4.y = pack_bf16x2(v[2], v[3]);
              o4.z = pack_bf16x2(v[4], v[5]);
              o4.w = pack_bf16x2(v[6], v[7]);
              dst[e] = o4;
            }
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem_base, Cfg::TMEM_COLS);
}

// ------------------------------------------------------------------ launchers
template <typename T>
static int quant_rows_t(const LaunchCtx& c, const void* x, long long ldx, int rows, int K, uint8_t* x8,
                        long long ld8, float* s) {
  quant_rows_kernel<T><<<rows, 128, 0, c.stream>>>(static_cast<const T*>(x), ldx, K, x8, ld8, s);
  return WAN_OK;
}

int launch_quant_rows_e4m3(const LaunchCtx& c, const void* x, int in_type, long long ldx, int rows, int K,
                           uint8_t* x8, long long ld8, float* s) {
  if (rows <= 0) return WAN_OK;
  if (K % 4 != 0 || ldx % 4 != 0 || ld8 % 4 != 0) return WAN_ERR_UNSUPPORTED;
  count_launch("quant_rows_e4m3", c.stream, true);
  if (in_type == OUT_F32) quant_rows_t<float>(c, x, ldx, rows, K, x8, ld8, s);
  else if (in_type == OUT_F16) quant_rows_t<__half>(c, x, ldx, rows, K, x8, ld8, s);
  else quant_rows_t<bf16>(c, x, ldx, rows, K, x8, ld8, s);
  count_launch("quant_rows_e4m3", c.stream, false);
  return cudaGetLastError() == cudaSuccess ? WAN_OK : WAN_ERR_CUDA;
}

template <typename TQK, typename TV>
static void quant_attn_t(const LaunchCtx& c, const Attn8Operands& a) {
  const long long rows = (long long)a.B * a.L;
  const unsigned qgrid = (unsigned)((rows * a.H + 7) / 8);
  const dim3 bgrid(a.nkb, a.H, a.B);
  count_launch("quant_q_e4m3", c.stream, true);
  quant_q_kernel<TQK, 128><<<qgrid, 256, 0, c.stream>>>(static_cast<const TQK*>(a.q), a.ldq, a.q_col, a.q8,
                                                        (long long)a.H * 128, a.sq, rows, a.H);
  count_launch("quant_q_e4m3", c.stream, false);
  count_launch("quant_k_e4m3", c.stream, true);
  quant_k_kernel<TQK, 128><<<bgrid, 256, 0, c.stream>>>(static_cast<const TQK*>(a.k), a.ldk, a.k_col, a.k8,
                                                        (long long)a.H * 128, a.sk, a.L, a.H, a.nkb);
  count_launch("quant_k_e4m3", c.stream, false);
  count_launch("quant_v_amax", c.stream, true);
  v_amax_kernel<TV, 128><<<bgrid, 256, 0, c.stream>>>(static_cast<const TV*>(a.v), a.ldv, a.v_col, a.v_amax, a.L,
                                                      a.H);
  count_launch("quant_v_amax", c.stream, false);
  count_launch("quant_vt_e4m3", c.stream, true);
  quant_vt_kernel<TV, 128><<<bgrid, 256, 0, c.stream>>>(static_cast<const TV*>(a.v), a.ldv, a.v_col, a.v_amax,
                                                        a.v8t, a.sv, a.L, a.Lp, a.H);
  count_launch("quant_vt_e4m3", c.stream, false);
}

int quant_attn_e4m3(const LaunchCtx& c, const Attn8Operands& a) {
  if (a.B <= 0 || a.L <= 0) return WAN_OK;
  if (a.head_dim != 128) return WAN_ERR_UNSUPPORTED;
  if (a.ldq % 4 || a.ldk % 4 || a.ldv % 4 || a.q_col % 4 || a.k_col % 4 || a.v_col % 4) return WAN_ERR_UNSUPPORTED;
  if (a.nkb != (a.L + 127) / 128 || a.Lp != ((a.L + 15) & ~15)) return WAN_ERR_INVALID_ARG;
  if (cudaMemsetAsync(a.v_amax, 0, sizeof(unsigned int) * (size_t)a.B * a.H * 128, c.stream) != cudaSuccess)
    return WAN_ERR_CUDA;
  if (a.qk_type == OUT_F16) {
    if (a.v_type == OUT_F16) quant_attn_t<__half, __half>(c, a);
    else quant_attn_t<__half, bf16>(c, a);
  } else {
    if (a.v_type == OUT_F16) quant_attn_t<bf16, __half>(c, a);
    else quant_attn_t<bf16, bf16>(c, a);
  }
  return cudaGetLastError() == cudaSuccess ? WAN_OK : WAN_ERR_CUDA;
}

int attention_e4m3(const LaunchCtx& c, const Attn8Args& a) {
  using Cfg = Attn8Cfg<128>;
  if (a.head_dim != 128) return WAN_ERR_UNSUPPORTED;
  if (a.B <= 0 || a.L <= 0) return WAN_OK;
  const int D = a.H * 128;
  CUtensorMap tq, tk, tv;
  int st = make_tmap_3d(&tq, a.q8, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, (uint64_t)D, (uint64_t)a.L, (uint64_t)a.B,
                        (uint64_t)D, (uint64_t)D * a.L, 128, 128);
  if (st != WAN_OK) return st;
  st = make_tmap_3d(&tk, a.k8, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, (uint64_t)D, (uint64_t)a.L, (uint64_t)a.B,
                    (uint64_t)D, (uint64_t)D * a.L, 128, 128);
  if (st != WAN_OK) return st;
  st = make_tmap_2d(&tv, a.v8t, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, (uint64_t)a.L, (uint64_t)a.B * a.H * 128,
                    (uint64_t)a.Lp, 128, 128);
  if (st != WAN_OK) return st;
  Attn8Params p;
  p.Lq = a.L;
  p.Lkv = a.L;
  p.H = a.H;
  p.nkb = (a.L + 127) / 128;
  p.nq_pairs = ((a.L + 127) / 128 + 1) / 2;
  p.scale_log2 = 1.4426950408889634f / sqrtf(128.0f);
  p.sq = a.sq;
  p.sk = a.sk;
  p.sv = a.sv;
  p.o = static_cast<bf16*>(a.o);
  p.ldo = a.ldo;
  p.o_col = a.o_col;
  p.kv_lens = a.kv_lens;
  static std::atomic<unsigned long long> smem_set{0};
  {
    const int st = set_smem_limit_once(reinterpret_cast<const void*>(attn_e4m3_tc_kernel<128>), Cfg::SMEM, &smem_set);
    if (st != WAN_OK) return st;
  }
  const long long grid = (long long)a.B * a.H * p.nq_pairs;
  const char* tag = a.tag ? a.tag : "attn_e4m3";
  count_launch(tag, c.stream, true);
  attn_e4m3_tc_kernel<128><<<(unsigned)grid, Cfg::THREADS, Cfg::SMEM, c.stream>>>(tq, tk, tv, p, c.dev_status);
  count_launch(tag, c.stream, false);
  return cudaGetLastError() == cudaSuccess ? WAN_OK : WAN_ERR_CUDA;
}

}  // namespace wan

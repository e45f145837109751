// bf16 GEMM on the 5th-generation tensor cores: C[M, N] = A[M, K] * B[N, K]^T with a
// fused epilogue (epilogue.cuh).  Every projection of the DiT block (QKV, output,
// cross-attention, FFN, patchify, head, text projection) runs through this kernel.
// The operand type is a template parameter: bf16 or fp16 A and B (kind::f16; the
// cross-attention projections run in fp16), or E4M3 (kind::f8f6f4, 128 elements per
// 128-byte stage row), whose instantiation multiplies the fp32 accumulator by the row
// scale of A and the column scale of B before the same epilogue.
//
// Design (one CTA per SM, persistent over output tiles of 128 x BN):
//   warp 0      TMA producer: A and B tiles (128-byte swizzle) into a STAGES-deep ring
//   warp 1      allocates TMEM, issues tcgen05.mma (M=128, N=BN, K=16) from one thread,
//               commits each consumed stage back to the producer
//   warps 2..9  epilogue: tcgen05.ld of the fp32 accumulator (one TMEM lane = one output
//               row per thread; two warps per TMEM lane quadrant, each taking half of the
//               tile's columns), bias/GELU/RoPE/gated residual/layout, global stores
// The accumulator is double-buffered in TMEM (2 x BN columns), so the epilogue of tile
// i overlaps the main loop of tile i+1.
// The gated residual x += gate * (acc + bias) never reads x into the SM: each warp
// stages its 32 x 32 fp32 chunk in shared memory (128-byte swizzle, conflict-free for
// one-row-per-thread writes) and a TMA reduce-add applies it to x in L2, so the
// read-modify-write of the fp32 residual stream moves whole lines and leaves no load
// latency in the epilogue.  The store-type epilogues go out the same way: each warp
// stages 32 rows x 128 bytes (32 fp32 or 64 16-bit columns) and issues a TMA store.  With
// one output row per thread, direct stores would send 32 scattered 16-byte pieces per
// instruction through the SM's memory pipe and hold up the next tile.
#include <cstdio>
#include <cstring>

#include "epilogue.cuh"
#include "kernels.h"

namespace wan {

// PAIR: the CTA holds half of a 256-row tile pair's A rows and half of its BN B rows
// (cta_group::2 MMA), so a stage is 16 + 16 KB and six stages fit.
template <int BN, bool PAIR = false>
struct GemmCfg {
  static constexpr int BM = 128;        // rows of A (and of the accumulator) in this CTA
  static constexpr int BK_BYTES = 128;  // one 128-byte swizzle row: 64 bf16 or 128 E4M3
  static constexpr int B_ROWS = PAIR ? BN / 2 : BN;
  static constexpr int A_BYTES = BM * BK_BYTES;
  static constexpr int B_BYTES = B_ROWS * BK_BYTES;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int STAGES = PAIR ? 6 : ((BN == 256) ? 4 : (BN == 128 ? 6 : 8));
  static constexpr int TMEM_COLS = 2 * BN;
  static constexpr int EPI_WARPS = 8;
  static constexpr int THREADS = 64 + 32 * EPI_WARPS;
  static constexpr int EPI_STAGE_BYTES = EPI_WARPS * 32 * 32 * 4;  // one [32][32] fp32 tile per epilogue warp
  static constexpr int BAR_BYTES = 256;
  static constexpr int SMEM = STAGES * STAGE_BYTES + EPI_STAGE_BYTES + BAR_BYTES + 1024;
  static_assert(TMEM_COLS == 128 || TMEM_COLS == 256 || TMEM_COLS == 512, "TMEM columns");
  static_assert(SMEM <= 232448, "dynamic shared memory above the 227 KB per-CTA limit");
};

// Operand types of one GEMM instantiation (A and B always share one type).
enum GemmAB : int { AB_BF16 = 0, AB_F16 = 1, AB_E4M3 = 2 };

// The kernel body.  PAIR: one 256 x BN tile per cluster of two CTAs (cta_group::2).  Each
// CTA loads its own halves of the A and B rows with its own TMA unit (one unit does not
// keep up with both halves), completing on the leader CTA's (rank 0) stage barrier; the
// leader issues every MMA and frees each stage in both CTAs; both CTAs' epilogue warps
// drain their own accumulator rows and free the accumulator on the leader's barrier.
template <int BN, int AB, bool PAIR>
__device__ __forceinline__ void gemm_body(const CUtensorMap& tmA, const CUtensorMap& tmB, const CUtensorMap& tmR,
                                          const EpiParams& ep, int M, int N, int K, int kb_period, int* status) {
  using Cfg = GemmCfg<BN, PAIR>;
  constexpr bool FP8 = AB == AB_E4M3;
  constexpr int TILE_M = PAIR ? 256 : 128;  // accumulator rows per tile (over the pair)
  constexpr int BK = FP8 ? 128 : 64;  // K elements per stage
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* epi_stage = smem + Cfg::STAGES * Cfg::STAGE_BYTES;
  uint64_t* full = reinterpret_cast<uint64_t*>(epi_stage + Cfg::EPI_STAGE_BYTES);
  uint64_t* empty = full + Cfg::STAGES;
  uint64_t* tfull = empty + Cfg::STAGES;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(drain + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int num_m = (M + TILE_M - 1) / TILE_M;
  const int num_n = (N + BN - 1) / BN;
  const int num_k = (K + BK - 1) / BK;
  const int num_tiles = num_m * num_n;
  const uint32_t rank = PAIR ? cluster_ctarank() : 0u;
  const bool leader = rank == 0;
  const int tile0 = PAIR ? (int)cluster_id_x() : (int)blockIdx.x;
  const int tile_step = PAIR ? (int)cluster_count_x() : (int)gridDim.x;

  if (threadIdx.x == 0) {
    for (int s = 0; s < Cfg::STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], (PAIR ? 2 : 1) * Cfg::EPI_WARPS);  // one arrival per epilogue warp (of both CTAs)
    }
    mbar_init(drain, 1);
    fence_barrier_init();
  }
  if (warp == 1) {
    if constexpr (PAIR) {
      tmem_alloc_pair(tmem_holder, Cfg::TMEM_COLS);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(tmem_holder, Cfg::TMEM_COLS);
      tmem_relinquish();
    }
  }
  tc_fence_before();
  __syncthreads();
  if constexpr (PAIR) cluster_sync();  // both CTAs' barriers exist before either is signalled
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;

  if (warp == 0 && lane == 0) {
    // ---------------------------------------------------------------- TMA producer
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    int stage = 0;
    uint32_t phase = 0;
    uint32_t issued = 0, issued_phase = 0;  // bit s: stage s holds a load; its phase
    bool ok = true;
    for (int tile = tile0; tile < num_tiles && ok; tile += tile_step) {
      const int mb = tile / num_n, nb = tile - (tile / num_n) * num_n;
      for (int kb = 0; kb < num_k; ++kb) {
        if (!mbar_wait(&empty[stage], phase ^ 1, status, kDevTimeoutGemm)) { ok = false; break; }
        uint8_t* sa = smem + stage * Cfg::STAGE_BYTES;
        const int kb_b = kb_period ? (kb % kb_period) : kb;
        if constexpr (PAIR) {
          // this CTA's rows mb*256 + rank*128 + [0, 128) of A and nb*BN + rank*BN/2 +
          // [0, BN/2) of B; the leader's barrier expects both CTAs' bytes (the peer's may
          // land before the leader's expect_tx: the phase cannot complete before the
          // leader's arrival)
          if (leader) mbar_arrive_expect_tx(&full[stage], 2 * Cfg::STAGE_BYTES);
          const uint32_t bar = cluster_addr(smem_u32(&full[stage]), 0);
          const uint32_t dst = smem_u32(sa);
          tma_load_2d_pair(dst, &tmA, bar, kb * BK, mb * TILE_M + (int)rank * Cfg::BM);
          tma_load_2d_pair(dst + Cfg::A_BYTES, &tmB, bar, kb_b * BK, nb * BN + (int)rank * Cfg::B_ROWS);
        } else {
          mbar_arrive_expect_tx(&full[stage], Cfg::STAGE_BYTES);
          tma_load_2d(sa, &tmA, &full[stage], kb * BK, mb * Cfg::BM);
          tma_load_2d(sa + Cfg::A_BYTES, &tmB, &full[stage], kb_b * BK, nb * BN);
        }
        issued |= 1u << stage;
        issued_phase = (issued_phase & ~(1u << stage)) | (phase << stage);
        if (++stage == Cfg::STAGES) { stage = 0; phase ^= 1; }
      }
    }
    if (!ok) {  // error path: let the copies in flight land before the CTA exits
      if (PAIR && !leader) {
        // the peer's copies complete on the leader's barriers, which it cannot test:
        // give them a fixed 50 us (a copy lands in a few)
        const unsigned long long t0 = globaltimer_ns();
        while (globaltimer_ns() - t0 < 50000ull) {}
      } else {
        for (int s = 0; s < Cfg::STAGES; ++s)
          if (issued & (1u << s)) {
            const unsigned long long t0 = globaltimer_ns();
            while (!mbar_test(&full[s], (issued_phase >> s) & 1u) && globaltimer_ns() - t0 < kWaitLimitNs) {}
          }
      }
    }
  } else if (warp == 1 && lane == 0 && leader) {
    // ---------------------------------------------------------------- MMA issuer
    constexpr uint32_t idesc = FP8 ? make_idesc_e4m3(TILE_M, BN)
                                   : (AB == AB_F16 ? make_idesc_f16(TILE_M, BN) : make_idesc_bf16(TILE_M, BN));
    // The commits of a pair signal the leader's stage barriers and both CTAs' accumulator
    // barriers.
    auto commit = [&](uint64_t* bar) {
      if constexpr (PAIR) tc_commit_pair(smem_u32(bar));
      else tc_commit(bar);
    };
    const uint32_t smem_lo0 = sdesc_sw128_lo(smem_u32(smem));
    int stage = 0;
    uint32_t phase = 0;
    int acc = 0;
    uint32_t acc_phase = 0;
    bool ok = true;
    for (int tile = tile0; tile < num_tiles && ok; tile += tile_step) {
      if (!mbar_wait(&tempty[acc], acc_phase ^ 1, status, kDevTimeoutGemm)) { ok = false; break; }
      tc_fence_after();
      const uint32_t d_tmem = tmem_base + acc * BN;
      for (int kb = 0; kb < num_k; ++kb) {
        if (!mbar_wait(&full[stage], phase, status, kDevTimeoutGemm)) { ok = false; break; }
        tc_fence_after();
        // Descriptor low words only (the issuing thread shares its SM sub-partition with
        // an epilogue warp): stage base + 32 bytes (>> 4 = 2) per MMA K step (16 bf16 or
        // 32 E4M3 elements).
        const uint32_t a_lo = smem_lo0 + (uint32_t)stage * (Cfg::STAGE_BYTES >> 4);
        const uint32_t b_lo = a_lo + (Cfg::A_BYTES >> 4);
#pragma unroll
        for (int kk = 0; kk < Cfg::BK_BYTES / 32; ++kk) {
          const uint32_t accum = (kb | kk) != 0 ? 1u : 0u;
          if constexpr (PAIR) {
            if constexpr (FP8) tc_mma_ss_f8_lo_pair(d_tmem, a_lo + kk * 2, b_lo + kk * 2, idesc, accum);
            else tc_mma_ss_lo_pair(d_tmem, a_lo + kk * 2, b_lo + kk * 2, idesc, accum);
          } else {
            if constexpr (FP8) tc_mma_ss_f8_lo(d_tmem, a_lo + kk * 2, b_lo + kk * 2, idesc, accum);
            else tc_mma_ss_lo(d_tmem, a_lo + kk * 2, b_lo + kk * 2, idesc, accum);
          }
        }
        commit(&empty[stage]);
        if constexpr (PAIR) tc_commit_pair(cluster_addr(smem_u32(&empty[stage]), 1));  // the peer's stage
        if (++stage == Cfg::STAGES) { stage = 0; phase ^= 1; }
      }
      if (!ok) break;
      commit(&tfull[acc]);
      if constexpr (PAIR) tc_commit_pair(cluster_addr(smem_u32(&tfull[acc]), 1));  // the peer's accumulator barrier
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1;
    }
    if (!ok) {  // error path: wait for the MMAs in flight before TMEM is released
      commit(drain);
      const unsigned long long t0 = globaltimer_ns();
      while (!mbar_test(drain, 0) && globaltimer_ns() - t0 < kWaitLimitNs) {}
    }
  } else if (warp >= 2) {
    // ---------------------------------------------------------------- epilogue
    const int quad = warp & 3;  // TMEM lanes [32*quad, 32*quad + 32) belong to this warp
    const int ehalf = (warp - 2) >> 2;  // which half of the tile's 32-column chunks
    constexpr int CH = BN / 32 / 2;     // chunks per epilogue warp
    const bool tma_resid = ep.kind == EPI_RESID;
    const bool tma_out = ep.tma_store != 0;  // tmR then maps the output [M, N]
    float* stage = reinterpret_cast<float*>(epi_stage + (warp - 2) * (32 * 32 * 4));  // [32][32], 1 KB aligned
    int acc = 0;
    uint32_t acc_phase = 0;
    const uint32_t tempty_leader0 = PAIR ? cluster_addr(smem_u32(&tempty[0]), 0) : 0u;
    for (int tile = tile0; tile < num_tiles; tile += tile_step) {
      const int mb = tile / num_n, nb = tile - (tile / num_n) * num_n;
      if (!mbar_wait_warp(&tfull[acc], acc_phase, status, kDevTimeoutGemm)) break;
      tc_fence_after();
      const int row0 = mb * TILE_M + (int)rank * Cfg::BM + quad * 32;
      const int row = row0 + lane;
      const uint32_t taddr = tmem_base + ((uint32_t)(quad * 32) << 16) + acc * BN;
      float sa_row = 1.f;
      if constexpr (FP8) sa_row = row < M ? ep.a_scale[row] : 0.f;
      // fp32 accumulator chunk -> v (times the A row and B column scales of the FP8 GEMM)
      auto acc_values = [&](const uint32_t (&r)[32], int n0, float (&v)[32]) {
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
        if constexpr (FP8) {
          const float4* sb4 = reinterpret_cast<const float4*>(ep.b_scale + n0);
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const float4 q = sb4[i];
            v[4 * i] *= sa_row * q.x;
            v[4 * i + 1] *= sa_row * q.y;
            v[4 * i + 2] *= sa_row * q.z;
            v[4 * i + 3] *= sa_row * q.w;
          }
        }
      };
#pragma unroll 1
      for (int c = ehalf * CH; c < (ehalf + 1) * CH; ++c) {
        uint32_t r[32];
        tmem_ld32(taddr + c * 32, r);
        const int n0 = nb * BN + c * 32;
        if (tma_resid) {
          if (row0 < M && n0 < N) {  // warp-uniform; rows past M are clipped by the TMA
            float v[32];
            acc_values(r, n0, v);
            epi_resid_values<32>(ep, row, n0, v);
            float* buf = stage;
            if (lane == 0) bulk_wait_group_read<0>();  // the reduce that last read `buf` is done
            __syncwarp();
            float4* dst = reinterpret_cast<float4*>(buf + lane * 32);
#pragma unroll
            for (int j = 0; j < 8; ++j)
              dst[j ^ (lane & 7)] = make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              tma_reduce_add_2d(&tmR, buf, n0, row0);
              bulk_commit_group();
            }
          }
        } else if (tma_out) {
          // 16-bit output: two 32-column chunks fill one 128-byte box row (64 columns;
          // the host enables this path only when BN >= 128, so a box never spans two
          // warps' columns); fp32 output: one chunk per box.  Rows past M and columns
          // past N are clipped by the TMA store.
          const bool wide = ep.out_type == OUT_F32;
          const int nbox = wide ? n0 : (n0 & ~63);  // first column of this chunk's box
          if (row0 < M && nbox < N) {  // warp-uniform
            const int ot = epilogue_out_type(ep, nbox);
            uint8_t* buf = reinterpret_cast<uint8_t*>(stage);
            if (wide || !(c & 1)) {  // the box is about to be refilled
              if (lane == 0) bulk_wait_group_read<0>();
              __syncwarp();
            }
            const uint32_t row_addr = smem_u32(buf) + lane * 128;
            if (n0 < N) {
              float v[32];
              acc_values(r, n0, v);
              epilogue_values<32>(ep, row, n0, v);
              if (wide) {
#pragma unroll
                for (int j = 0; j < 8; ++j)
                  st_shared_v4(row_addr + ((uint32_t)(j ^ (lane & 7)) << 4),
                               make_uint4(__float_as_uint(v[4 * j]), __float_as_uint(v[4 * j + 1]),
                                          __float_as_uint(v[4 * j + 2]), __float_as_uint(v[4 * j + 3])));
              } else {
                const bool h = ot == OUT_F16;
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                  uint4 u;
                  const float* w = v + 8 * e;
                  u.x = h ? pack_half2(w[0], w[1]) : pack_bf16x2(w[0], w[1]);
                  u.y = h ? pack_half2(w[2], w[3]) : pack_bf16x2(w[2], w[3]);
                  u.z = h ? pack_half2(w[4], w[5]) : pack_bf16x2(w[4], w[5]);
                  u.w = h ? pack_half2(w[6], w[7]) : pack_bf16x2(w[6], w[7]);
                  st_shared_v4(row_addr + ((uint32_t)(((c & 1) * 4 + e) ^ (lane & 7)) << 4), u);
                }
              }
            }
            if (wide || (c & 1)) {  // the box is complete
              fence_proxy_async_smem();
              __syncwarp();
              if (lane == 0) {
                tma_store_2d(&tmR, buf, nbox, row0);
                bulk_commit_group();
              }
            }
          }
        } else if (row < M && n0 < N) {
          float v[32];
          acc_values(r, n0, v);
          epilogue_chunk<32>(ep, row, n0, v);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (PAIR && !leader) mbar_arrive_cluster(tempty_leader0 + acc * sizeof(uint64_t));
        else mbar_arrive(&tempty[acc]);
      }
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1;
    }
    if ((tma_resid || tma_out) && lane == 0) bulk_wait_group_all();  // bulk writes finished before the CTA exits
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  if constexpr (PAIR) cluster_sync();  // the peer's shared and tensor memory are no longer in use
  tc_fence_after();
  if (warp == 1) {
    if constexpr (PAIR) tmem_dealloc_pair(tmem_base, Cfg::TMEM_COLS);
    else tmem_dealloc(tmem_base, Cfg::TMEM_COLS);
  }
}

template <int BN, int AB>
__global__ void __launch_bounds__(64 + 32 * GemmCfg<BN>::EPI_WARPS, 1)
    gemm_bf16_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                        const __grid_constant__ CUtensorMap tmR, const EpiParams ep, int M, int N, int K,
                        int kb_period, int* status) {
  gemm_body<BN, AB, false>(tmA, tmB, tmR, ep, M, N, K, kb_period, status);
}

// 256 x 256 tiles over a cluster of two CTAs (cta_group::2): per CTA and K step, 16 KB of
// A and 16 KB of B, so the L2 -> SM operand stream per FLOP is a third lower than with a
// 128 x 256 tile per CTA, and six stages are in flight.
template <int AB>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(64 + 32 * GemmCfg<256, true>::EPI_WARPS, 1)
    gemm_pair_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                        const __grid_constant__ CUtensorMap tmR, const EpiParams ep, int M, int N, int K,
                        int kb_period, int* status) {
  gemm_body<256, AB, true>(tmA, tmB, tmR, ep, M, N, K, kb_period, status);
}

template <int BN, int AB>
static int launch_gemm(const LaunchCtx& c, const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& tr,
                       const EpiParams& ep, int M, int N, int K, int kb_period, const char* tag) {
  using Cfg = GemmCfg<BN>;
  static std::atomic<unsigned long long> smem_set{0};
  {
    const int st = set_smem_limit_once(reinterpret_cast<const void*>(gemm_bf16_tc_kernel<BN, AB>), Cfg::SMEM, &smem_set);
    if (st != WAN_OK) return st;
  }
  const int tiles = ((M + 127) / 128) * ((N + BN - 1) / BN);
  const int grid = tiles < c.num_sms ? tiles : c.num_sms;
  count_launch(tag, c.stream, true);
  gemm_bf16_tc_kernel<BN, AB><<<grid, Cfg::THREADS, Cfg::SMEM, c.stream>>>(ta, tb, tr, ep, M, N, K, kb_period,
                                                                           c.dev_status);
  count_launch(tag, c.stream, false);
  return cudaGetLastError() == cudaSuccess ? WAN_OK : WAN_ERR_CUDA;
}

template <int AB>
static int launch_gemm_pair(const LaunchCtx& c, const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& tr,
                            const EpiParams& ep, int M, int N, int K, int kb_period, const char* tag) {
  using Cfg = GemmCfg<256, true>;
  static std::atomic<unsigned long long> smem_set{0};
  {
    const int st = set_smem_limit_once(reinterpret_cast<const void*>(gemm_pair_tc_kernel<AB>), Cfg::SMEM, &smem_set);
    if (st != WAN_OK) return st;
  }
  // Clusters that fit on the GPU at once (a pair needs two free SMs of one GPC, so this can
  // be below half the SM count); tiles are strided over the resident clusters only.
  static std::atomic<int> resident[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return WAN_ERR_CUDA;
  int pairs = resident[dev].load(std::memory_order_acquire);
  if (pairs <= 0) {
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = 2;
    attr.val.clusterDim.y = 1;
    attr.val.clusterDim.z = 1;
    cfg.gridDim = dim3(c.num_sms, 1, 1);
    cfg.blockDim = dim3(Cfg::THREADS, 1, 1);
    cfg.dynamicSmemBytes = Cfg::SMEM;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, reinterpret_cast<const void*>(gemm_pair_tc_kernel<AB>), &cfg) !=
            cudaSuccess ||
        n <= 0) {
      // No answer: half the SMs is still a correct grid (clusters that do not fit at
      // once run later); clear the error so the launch check below does not see it.
      (void)cudaGetLastError();
      n = c.num_sms / 2;
    }
    pairs = n < c.num_sms / 2 ? n : c.num_sms / 2;
    if (pairs < 1) pairs = 1;
    resident[dev].store(pairs, std::memory_order_release);
  }
  const int tiles = ((M + 255) / 256) * (N / 256);
  const int clusters = tiles < pairs ? tiles : pairs;
  count_launch(tag, c.stream, true);
  gemm_pair_tc_kernel<AB><<<2 * clusters, Cfg::THREADS, Cfg::SMEM, c.stream>>>(ta, tb, tr, ep, M, N, K, kb_period,
                                                                               c.dev_status);
  count_launch(tag, c.stream, false);
  return cudaGetLastError() == cudaSuccess ? WAN_OK : WAN_ERR_CUDA;
}

// The CTA-pair GEMM takes the projections whose N is a multiple of 256 and whose M spans
// at least a few pairs of tiles; the others (the head, small test shapes) stay on one SM
// per tile.  GELU epilogues stay on one SM too: timed inside the 1.3B step on one B300,
// the pair takes FFN-down, the output projections and the cross-attention query 3-11 %
// below the one-SM kernel but the FFN up-projection with its GELU epilogue 2.5 % above it.
static bool use_pair(int M, int N, const EpiParams& ep) {
  return N % 256 == 0 && M >= 4 * 256 && ep.kind != EPI_GELU && ep.kind != EPI_GELU_TANH;
}

// Tensor map of the epilogue's bulk writes: the fp32 residual x [M, N] (row stride ldr,
// 32 x 32 boxes) for EPI_RESID; for the store-type epilogues the output [M, N] (32 x 32
// fp32 boxes, or 64 x 32 16-bit boxes when the tile is at least 128 columns wide), which
// turns on ep.tma_store.  Other epilogues write directly.
static int output_map(CUtensorMap* m, EpiParams& ep, int M, int N, int bn) {
  memset(m, 0, sizeof(*m));
  ep.tma_store = 0;
  if (ep.kind == EPI_RESID) {
    if (ep.ldr % 4 != 0) return WAN_ERR_UNSUPPORTED;
    return make_tmap_2d(m, ep.resid, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, (uint64_t)N, (uint64_t)M,
                        (uint64_t)ep.ldr * 4, 32, 32);
  }
  const bool store_kind = ep.kind == EPI_STORE || ep.kind == EPI_GELU || ep.kind == EPI_GELU_TANH || ep.kind == EPI_QKV;
  if (!store_kind || !ep.out || (reinterpret_cast<uintptr_t>(ep.out) & 15)) return WAN_OK;
  if (ep.out_type == OUT_F32) {
    if (ep.ldo % 4 != 0) return WAN_OK;
    if (make_tmap_2d(m, ep.out, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, (uint64_t)N, (uint64_t)M, (uint64_t)ep.ldo * 4,
                     32, 32) != WAN_OK)
      return WAN_OK;  // direct stores
  } else {
    if (bn < 128 || ep.ldo % 8 != 0) return WAN_OK;
    if (make_tmap_2d(m, ep.out, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, (uint64_t)N, (uint64_t)M, (uint64_t)ep.ldo * 2,
                     64, 32) != WAN_OK)
      return WAN_OK;
  }
  ep.tma_store = 1;
  return WAN_OK;
}

int gemm_bf16(const LaunchCtx& c, const void* A, long long lda, int a_cols, const void* B, long long ldb, int b_cols,
              int M, int N, int K, int kb_period, const EpiParams& ep_in, const char* tag, bool ab_f16) {
  if (M <= 0 || N <= 0 || K <= 0) return WAN_OK;
  int bn = (N % 256 == 0) ? 256 : (N % 128 == 0 ? 128 : 64);
  const CUtensorMapDataType dt = ab_f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const bool pair = use_pair(M, N, ep_in);
  CUtensorMap ta, tb;
  int st = make_tmap_2d(&ta, A, dt, 2, (uint64_t)a_cols, (uint64_t)M, (uint64_t)lda * 2, 64, 128);
  if (st != WAN_OK) return st;
  st = make_tmap_2d(&tb, B, dt, 2, (uint64_t)b_cols, (uint64_t)N, (uint64_t)ldb * 2, 64, (uint32_t)(pair ? 128 : bn));
  if (st != WAN_OK) return st;
  CUtensorMap tr;
  EpiParams ep = ep_in;
  st = output_map(&tr, ep, M, N, bn);
  if (st != WAN_OK) return st;
  if (pair)
    return ab_f16 ? launch_gemm_pair<AB_F16>(c, ta, tb, tr, ep, M, N, K, kb_period, tag)
                  : launch_gemm_pair<AB_BF16>(c, ta, tb, tr, ep, M, N, K, kb_period, tag);
  if (ab_f16) {
    switch (bn) {
      case 256: return launch_gemm<256, AB_F16>(c, ta, tb, tr, ep, M, N, K, kb_period, tag);
      case 128: return launch_gemm<128, AB_F16>(c, ta, tb, tr, ep, M, N, K, kb_period, tag);
      default: return launch_gemm<64, AB_F16>(c, ta, tb, tr, ep, M, N, K, kb_period, tag);
    }
  }
  switch (bn) {
    case 256: return launch_gemm<256, AB_BF16>(c, ta, tb, tr, ep, M, N, K, kb_period, tag);
    case 128: return launch_gemm<128, AB_BF16>(c, ta, tb, tr, ep, M, N, K, kb_period, tag);
    default: return launch_gemm<64, AB_BF16>(c, ta, tb, tr, ep, M, N, K, kb_period, tag);
  }
}

int gemm_e4m3(const LaunchCtx& c, const uint8_t* A, long long lda, int a_cols, const float* sa, const uint8_t* B,
              long long ldb, int b_cols, const float* sb, int M, int N, int K, const EpiParams& ep_in, const char* tag) {
  if (M <= 0 || N <= 0 || K <= 0) return WAN_OK;
  if (!sa || !sb || (reinterpret_cast<uintptr_t>(sb) & 15) || N % 32) return WAN_ERR_UNSUPPORTED;
  const int bn = (N % 256 == 0) ? 256 : (N % 128 == 0 ? 128 : 64);
  CUtensorMap ta, tb;
  int st = make_tmap_2d(&ta, A, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, (uint64_t)a_cols, (uint64_t)M, (uint64_t)lda, 128,
                        128);
  if (st != WAN_OK) return st;
  const bool pair = use_pair(M, N, ep_in);
  st = make_tmap_2d(&tb, B, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, (uint64_t)b_cols, (uint64_t)N, (uint64_t)ldb, 128,
                    (uint32_t)(pair ? 128 : bn));
  if (st != WAN_OK) return st;
  EpiParams ep = ep_in;
  ep.a_scale = sa;
  ep.b_scale = sb;
  CUtensorMap tr;
  st = output_map(&tr, ep, M, N, bn);
  if (st != WAN_OK) return st;
  if (pair) return launch_gemm_pair<AB_E4M3>(c, ta, tb, tr, ep, M, N, K, 0, tag);
  switch (bn) {
    case 256: return launch_gemm<256, AB_E4M3>(c, ta, tb, tr, ep, M, N, K, 0, tag);
    case 128: return launch_gemm<128, AB_E4M3>(c, ta, tb, tr, ep, M, N, K, 0, tag);
    default: return launch_gemm<64, AB_E4M3>(c, ta, tb, tr, ep, M, N, K, 0, tag);
  }
}

}  // namespace wan

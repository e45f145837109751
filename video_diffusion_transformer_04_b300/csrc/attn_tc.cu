// Flash-style attention on the 5th-generation tensor cores for the DiT's full
// bidirectional self-attention and its short-context cross-attention:
//   o = softmax(q k^T / sqrt(d)) v  per (batch, head), no mask.
//
// One CTA owns two 128-row query tiles of one (batch, head) and streams the whole key
// sequence in 128-key tiles.  Tensor memory holds, per query tile, the score tile S
// (128 fp32 columns; the bf16 probabilities P overwrite its first 64 columns) and the
// output accumulator O (d fp32 columns): 2 x 256 = 512 columns.
//   warp 0      TMA: Q once, then K and V tiles into 2-deep rings
//   warp 1      tcgen05.mma from one thread: S_i = Q_i K^T (both operands in smem),
//               O_i += P_i V (P from TMEM, V tile from smem), ping-ponging the tiles.
//               Per key tile j: PV_0(j), S_0(j+1) | wait for P_1(j) | PV_1(j), S_1(j+1):
//               each tile's cycle is its own MMAs plus its softmax, the two tiles half
//               a cycle apart.  S_i(j+1) always follows PV_i(j), because P_i overwrites
//               S_i in TMEM.
//   warps 4..11 softmax, one warpgroup per query tile, one thread per query row: fp32
//               running max and sum, exp2 on the MUFU unit, lazy rescale of O in TMEM
//               only when the running max grows by more than 2^8, final 1/l and store.
// The first warpgroup (TMA, MMA, two idle warps) gives registers to the softmax
// warpgroups (setmaxnreg), which keep a whole 128-column score row in registers.
// Per score element the softmax issues half an FFMA2 (scale and max subtraction on
// packed pairs), one MUFU ex2, half a bf16x2 pack and half an FADD2 (row sum); the row
// max is only computed for the first key tile and when a row sum signals that the
// reference max must move; the ragged-tile mask runs only on the last key tile.
// V is read in its natural [token, H*d] layout: in the PV product it is the B operand
// with N = d contiguous, i.e. MN-major (descriptor LBO = the 64-column box stride,
// SBO = 1024 bytes per 8 keys), so no transposed copy of V is ever written.
// Ragged tails: keys past the entry's key count (Lkv, or its k_lens value) are masked to
// -inf (past Lkv TMA also zero-fills them); query rows past Lq are computed on zero rows
// and not stored.
#include "kernels.h"
#include "wan_common.cuh"

namespace wan {

template <int HD>
struct AttnCfg {
  static constexpr int BQ = 128;
  static constexpr int BKV = 128;
  static constexpr int Q_BYTES = BQ * HD * 2;    // HD/64 boxes of 128 rows x 128 B
  static constexpr int K_BYTES = BKV * HD * 2;   // HD/64 boxes of 128 rows x 128 B
  static constexpr int V_BYTES = BKV * HD * 2;   // HD/64 boxes of 128 keys x 128 B
  static constexpr int Q_BOX = BQ * 128;         // bytes per 64-column box of a Q/K tile
  static constexpr int V_BOX = BKV * 128;        // bytes per 64-column box of a V tile
  static constexpr int SMEM_TILES = 2 * Q_BYTES + 2 * K_BYTES + 2 * V_BYTES;
  static constexpr int SMEM = SMEM_TILES + 256 + 1024;
  static constexpr int TMEM_COLS = 512;
  static constexpr int THREADS = 384;
  // setmaxnreg split of the 384 x 168 registers the CTA launches with:
  // 128 x PRODUCER_REGS + 256 x SOFTMAX_REGS <= 384 x 168.
  // (64 for the producer warpgroup: at 56 the MMA issuer's loop spills.)
  static constexpr int PRODUCER_REGS = 64;
  static constexpr int SOFTMAX_REGS = 216;
  static_assert(128 * PRODUCER_REGS + 256 * SOFTMAX_REGS <= 384 * 168, "register split");
  static_assert(HD % 64 == 0, "Q/K/V tiles are whole 64-column (128-byte) boxes");
};

struct AttnParams {
  int Lq, Lkv, H;
  int q_col, k_col, v_col;  // column offset of head 0 inside the q / k / v rows
  int nq_pairs;           // ceil(ceil(Lq/128)/2)
  float scale_log2;       // log2(e) / sqrt(d)
  bf16* o;                // [B, Lq, ldo]
  long long ldo;
  int o_col;
  int accumulate;         // o += result (decoupled cross-attention)
  const int* kv_lens;     // [B] valid keys per batch entry, or NULL (all Lkv)
};

template <int HD, bool QK_F16>
__global__ void __launch_bounds__(384, 1)
    attn_bf16_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                        const __grid_constant__ CUtensorMap tmV, const AttnParams p, int* status) {
  using Cfg = AttnCfg<HD>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem;                                  // [2][Q_BYTES]
  uint8_t* sK = sQ + 2 * Cfg::Q_BYTES;                 // [2][K_BYTES]
  uint8_t* sV = sK + 2 * Cfg::K_BYTES;                 // [2][V_BYTES]
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Cfg::SMEM_TILES);
  uint64_t* q_full = bars + 0;
  uint64_t* k_full = bars + 1;   // [2]
  uint64_t* k_empty = bars + 3;  // [2]
  uint64_t* v_full = bars + 5;   // [2]
  uint64_t* v_empty = bars + 7;  // [2]
  uint64_t* s_full = bars + 9;   // [2] per query tile
  uint64_t* p_ready = bars + 11; // [2] per query tile
  uint64_t* drain = bars + 13;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + 14);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int bh = blockIdx.x / p.nq_pairs;
  const int qp = blockIdx.x - bh * p.nq_pairs;
  const int b = bh / p.H;
  const int h = bh - b * p.H;
  const int q0 = qp * 256;
  const int ntile = (q0 + 128 < p.Lq) ? 2 : 1;
  // Keys of this batch entry: all Lkv, or its own length (k_lens), clamped to [1, Lkv].
  const int lkv = p.kv_lens ? min(max(p.kv_lens[b], 1), p.Lkv) : p.Lkv;
  const int nkv = (lkv + Cfg::BKV - 1) / Cfg::BKV;

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&k_empty[s], 1);
      mbar_init(&v_full[s], 1);
      mbar_init(&v_empty[s], 1);
      mbar_init(&s_full[s], 1);
      mbar_init(&p_ready[s], 4);  // one arrival per softmax warp
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
    mbar_arrive_expect_tx(q_full, ntile * Cfg::Q_BYTES);
    for (int i = 0; i < ntile; ++i)
      for (int c = 0; c < HD / 64; ++c)
        tma_load_3d(sQ + i * Cfg::Q_BYTES + c * Cfg::Q_BOX, &tmQ, q_full, p.q_col + h * HD + c * 64,
                    q0 + i * 128, b);
    uint32_t kissued = 0, vissued = 0;
    bool ok = true;
    for (int j = 0; j < nkv && ok; ++j) {
      const int s = j & 1;
      const uint32_t ph = (j >> 1) & 1;
      if (!mbar_wait(&k_empty[s], ph ^ 1, status, kDevTimeoutAttn)) { ok = false; break; }
      mbar_arrive_expect_tx(&k_full[s], Cfg::K_BYTES);
      for (int c = 0; c < HD / 64; ++c)
        tma_load_3d(sK + s * Cfg::K_BYTES + c * Cfg::Q_BOX, &tmK, &k_full[s], p.k_col + h * HD + c * 64,
                    j * Cfg::BKV, b);
      kissued = j + 1;
      if (!mbar_wait(&v_empty[s], ph ^ 1, status, kDevTimeoutAttn)) { ok = false; break; }
      mbar_arrive_expect_tx(&v_full[s], Cfg::V_BYTES);
      for (int c = 0; c < HD / 64; ++c)
        tma_load_3d(sV + s * Cfg::V_BYTES + c * Cfg::V_BOX, &tmV, &v_full[s], p.v_col + h * HD + c * 64,
                    j * Cfg::BKV, b);
      vissued = j + 1;
    }
    if (!ok) {  // error path: let issued copies land
      const unsigned long long t0 = globaltimer_ns();
      for (uint32_t j = (kissued > 2 ? kissued - 2 : 0); j < kissued; ++j)
        while (!mbar_test(&k_full[j & 1], (j >> 1) & 1) && globaltimer_ns() - t0 < kWaitLimitNs) {}
      for (uint32_t j = (vissued > 2 ? vissued - 2 : 0); j < vissued; ++j)
        while (!mbar_test(&v_full[j & 1], (j >> 1) & 1) && globaltimer_ns() - t0 < kWaitLimitNs) {}
      while (!mbar_test(q_full, 0) && globaltimer_ns() - t0 < kWaitLimitNs) {}
    }
  } else if (warp == 1 && lane == 0) {
    // ---------------------------------------------------------------- MMA issuer
    constexpr uint32_t idS = QK_F16 ? make_idesc_f16(128, Cfg::BKV) : make_idesc_bf16(128, Cfg::BKV);
    constexpr uint32_t idO = make_idesc_bf16(128, HD) | kIdescBMnMajor;
    bool ok = mbar_wait(q_full, 0, status, kDevTimeoutAttn) && mbar_wait(&k_full[0], 0, status, kDevTimeoutAttn);
    // Descriptor low words of every operand buffer, computed once: the issuing thread
    // shares its SM sub-partition with two softmax warps, so each MMA costs only an add.
    const uint32_t q_lo0 = sdesc_sw128_lo(smem_u32(sQ)), q_lo1 = sdesc_sw128_lo(smem_u32(sQ + Cfg::Q_BYTES));
    const uint32_t k_lo0 = sdesc_sw128_lo(smem_u32(sK)), k_lo1 = sdesc_sw128_lo(smem_u32(sK + Cfg::K_BYTES));
    const uint32_t v_lo0 = sdesc_sw128_mn_lo(smem_u32(sV), Cfg::V_BOX);
    const uint32_t v_lo1 = sdesc_sw128_mn_lo(smem_u32(sV + Cfg::V_BYTES), Cfg::V_BOX);
    auto issue_S = [&](int i, int ks) {
      const uint32_t qa = i ? q_lo1 : q_lo0;
      const uint32_t ka = ks ? k_lo1 : k_lo0;
      const uint32_t d = tmem_base + i * 256;
#pragma unroll
      for (int kk = 0; kk < HD / 16; ++kk) {
        const uint32_t off = ((kk >> 2) * Cfg::Q_BOX + (kk & 3) * 32) >> 4;
        tc_mma_ss_lo(d, qa + off, ka + off, idS, kk > 0 ? 1u : 0u);
      }
    };
    auto issue_PV = [&](int i, int vs, uint32_t acc) {
      const uint32_t va = vs ? v_lo1 : v_lo0;
      const uint32_t d = tmem_base + i * 256 + 128;
      const uint32_t pa = tmem_base + i * 256;
#pragma unroll
      for (int kk = 0; kk < Cfg::BKV / 16; ++kk) {
        const uint32_t off = (kk * 16 * 128) >> 4;  // 16 keys = 16 rows of 128 bytes
        tc_mma_ts_lo(d, pa + kk * 8, va + off, idO, (acc | (uint32_t)kk) != 0 ? 1u : 0u);
      }
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
      const int vs = j & 1;
      const int ks = (j + 1) & 1;
      const bool more = j + 1 < nkv;
      if (!mbar_wait(&v_full[vs], (j >> 1) & 1, status, kDevTimeoutAttn)) { ok = false; break; }
      if (more && !mbar_wait(&k_full[ks], ((j + 1) >> 1) & 1, status, kDevTimeoutAttn)) { ok = false; break; }
      if (!mbar_wait(&p_ready[0], j & 1, status, kDevTimeoutAttn)) { ok = false; break; }
      tc_fence_after();
      // Tile 0's next scores right behind its PV product: its softmax starts as soon as
      // they finish, independently of tile 1 (the tensor pipe runs them in order, so
      // S_0(j+1) overwrites P_0 only after PV_0(j) has read it).
      issue_PV(0, vs, j > 0 ? 1u : 0u);
      if (more) issue_S(0, ks);
      tc_commit(&s_full[0]);
      if (ntile == 2) {
        if (!mbar_wait(&p_ready[1], j & 1, status, kDevTimeoutAttn)) { ok = false; break; }
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
    const int i = (warp - 4) >> 2;   // query tile of this warpgroup
    const int quad = warp & 3;       // TMEM lane quadrant of this warp
    if (i < ntile) {
      const uint32_t tS = tmem_base + ((uint32_t)(quad * 32) << 16) + i * 256;
      const uint32_t tO = tS + 128;
      const float sl2 = p.scale_log2;
      const uint64_t sl2x2 = f2_pack(sl2, sl2);
      float m_used = -INFINITY;  // running max of the scaled logits (log2 units)
      float l_sum = 0.f;
      bool ok = true;
      uint32_t sr[Cfg::BKV];
      // S row of this thread -> sr (keys >= Lkv of a ragged last tile set to -inf).
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
      // p = 2^(s * scale - m): packed pairs through FFMA2, exp2 on MUFU, bf16x2 into the
      // first half of each 32-column chunk's registers (dead once read), row sum in
      // four FADD2 accumulators on the fp32 values.
      auto exp_pass = [&](float m, float& rowsum) {
        const uint64_t negm = f2_pack(-m, -m);
        uint64_t acc0 = 0, acc1 = 0, acc2 = 0, acc3 = 0;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const float s0 = __uint_as_float(sr[c * 32 + 2 * e]), s1 = __uint_as_float(sr[c * 32 + 2 * e + 1]);
            const float2 t = f2_unpack(f2_fma(f2_pack(s0, s1), sl2x2, negm));
            const float p0 = ex2_approx(t.x), p1 = ex2_approx(t.y);
            sr[c * 32 + e] = pack_bf16x2(p0, p1);
            const uint64_t pp = f2_pack(p0, p1);
            switch (e & 3) {
              case 0: acc0 = f2_add(acc0, pp); break;
              case 1: acc1 = f2_add(acc1, pp); break;
              case 2: acc2 = f2_add(acc2, pp); break;
              default: acc3 = f2_add(acc3, pp); break;
            }
          }
        }
        const float2 rs = f2_unpack(f2_add(f2_add(acc0, acc1), f2_add(acc2, acc3)));
        rowsum = rs.x + rs.y;
      };
      // Row max of the scores in sr (four chains of 3-input max).
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
      for (int j = 0; j < nkv; ++j) {
        if (!mbar_wait_warp(&s_full[i], j & 1, status, kDevTimeoutAttn)) { ok = false; break; }
        tc_fence_after();
        const int valid = lkv - j * Cfg::BKV;  // >= 1
        load_scores(valid);
        float rowsum;
        if (j == 0) {
          // First key tile: the reference max is this tile's row max.
          m_used = row_max() * sl2;
          exp_pass(m_used, rowsum);
        } else {
          // Lazy rescale: exponentiate against the current reference max.  A tile row sum
          // above 2^16 means some exponential exceeded 2^9 (128 keys), i.e. the row's max
          // rose by more than 9 (log2) since its reference was set: only then does the warp
          // find those rows' new max, rescale their O and sum (alpha = 1 for the other rows:
          // the tcgen05.ld/st are warp-collective), reload S and redo the exponentials.
          // Otherwise every p <= 2^16, which bf16 P and the fp32 O and sum hold as well as
          // p <= 1.  (An overflow to inf or a NaN also takes the slow path.)
          exp_pass(m_used, rowsum);
          const bool need = !(rowsum <= 65536.0f);
          if (__any_sync(0xffffffffu, need)) {
            load_scores(valid);
            const float mt = row_max() * sl2;
            const float alpha = need ? ex2_approx(m_used - mt) : 1.0f;
            l_sum *= alpha;
            if (need) m_used = mt;
#pragma unroll 1
            for (int c = 0; c < HD / 32; ++c) {
              uint32_t orr[32];
              tmem_ld32(tO + c * 32, orr);
#pragma unroll
              for (int e = 0; e < 32; ++e) orr[e] = __float_as_uint(__uint_as_float(orr[e]) * alpha);
              tmem_st32(tO + c * 32, orr);
            }
            exp_pass(m_used, rowsum);
          }
        }
#pragma unroll
        for (int c = 0; c < 4; ++c) tmem_st16_nowait(tS + c * 16, sr + c * 32);
        tmem_wait_st();
        l_sum += rowsum;
        // One arrival per warp: the warp's TMEM stores are complete and ordered before it.
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&p_ready[i]);
      }
      if (ok && mbar_wait_warp(&s_full[i], nkv & 1, status, kDevTimeoutAttn)) {
        tc_fence_after();
        const float inv = 1.0f / l_sum;
        const int qrow = q0 + i * 128 + quad * 32 + lane;
        bf16* orow = p.o + ((long long)b * p.Lq + qrow) * p.ldo + p.o_col + h * HD;
#pragma unroll 1
        for (int c = 0; c < HD / 32; ++c) {
          uint32_t orr[32];
          tmem_ld32(tO + c * 32, orr);
          if (qrow < p.Lq) {
            uint4* dst = reinterpret_cast<uint4*>(orow + c * 32);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              float v[8];
#pragma unroll
              for (int u = 0; u < 8; ++u) v[u] = __uint_as_float(orr[e * 8 + u]) * inv;
              if (p.accumulate) {
                const uint4 prev = dst[e];
                const uint32_t pw[4] = {prev.x, prev.y, prev.z, prev.w};
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                  const float2 f = unpack_bf16x2(pw[u]);
                  v[2 * u] += f.x;
                  v[2 * u + 1] += f.y;
                }
              }
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

template <int HD, bool QK_F16>
static int launch_attn(const LaunchCtx& c, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                       const AttnParams& p, int B, const char* tag) {
  using Cfg = AttnCfg<HD>;
  static std::atomic<unsigned long long> smem_set{0};
  {
    const int st = set_smem_limit_once(reinterpret_cast<const void*>(attn_bf16_tc_kernel<HD, QK_F16>), Cfg::SMEM, &smem_set);
    if (st != WAN_OK) return st;
  }
  const long long grid = (long long)B * p.H * p.nq_pairs;
  count_launch(tag, c.stream, true);
  attn_bf16_tc_kernel<HD, QK_F16><<<(unsigned)grid, Cfg::THREADS, Cfg::SMEM, c.stream>>>(tq, tk, tv, p, c.dev_status);
  count_launch(tag, c.stream, false);
  return cudaGetLastError() == cudaSuccess ? WAN_OK : WAN_ERR_CUDA;
}

int attention_bf16(const LaunchCtx& c, const AttnArgs& a) {
  if (a.head_dim != 64 && a.head_dim != 128) return WAN_ERR_UNSUPPORTED;
  if (a.Lq <= 0 || a.Lkv <= 0) return WAN_OK;
  const int HD = a.head_dim;
  CUtensorMap tq, tk, tv;
  const CUtensorMapDataType qkt = a.qk_f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  int st = make_tmap_3d(&tq, a.q, qkt, 2, (uint64_t)a.q_row_len, (uint64_t)a.Lq,
                        (uint64_t)a.B, (uint64_t)a.ldq * 2, (uint64_t)a.ldq * 2 * a.Lq, 64, 128);
  if (st != WAN_OK) return st;
  st = make_tmap_3d(&tk, a.k, qkt, 2, (uint64_t)a.k_row_len, (uint64_t)a.Lkv,
                    (uint64_t)a.B, (uint64_t)a.ldk * 2, (uint64_t)a.ldk * 2 * a.Lkv, 64, 128);
  if (st != WAN_OK) return st;
  st = make_tmap_3d(&tv, a.v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, (uint64_t)a.v_row_len, (uint64_t)a.Lkv,
                    (uint64_t)a.B, (uint64_t)a.ldv * 2, (uint64_t)a.ldv * 2 * a.Lkv, 64, 128);
  if (st != WAN_OK) return st;
  AttnParams p;
  p.Lq = a.Lq;
  p.Lkv = a.Lkv;
  p.H = a.H;
  p.q_col = a.q_col;
  p.k_col = a.k_col;
  p.v_col = a.v_col;
  p.nq_pairs = ((a.Lq + 127) / 128 + 1) / 2;
  p.scale_log2 = 1.4426950408889634f / sqrtf((float)HD);
  p.o = static_cast<bf16*>(a.o);
  p.ldo = a.ldo;
  p.o_col = a.o_col;
  p.accumulate = a.accumulate;
  p.kv_lens = a.kv_lens;
  const char* tag = a.tag ? a.tag : "attn";
  if (HD == 128)
    return a.qk_f16 ? launch_attn<128, true>(c, tq, tk, tv, p, a.B, tag) : launch_attn<128, false>(c, tq, tk, tv, p, a.B, tag);
  return a.qk_f16 ? launch_attn<64, true>(c, tq, tk, tv, p, a.B, tag) : launch_attn<64, false>(c, tq, tk, tv, p, a.B, tag);
}

}  // namespace wan

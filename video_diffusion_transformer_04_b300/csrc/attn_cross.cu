// Cross-attention of the DiT block on the 5th-generation tensor cores.  Every query row
// attends to the short text context and, for image-to-video, separately to the image
// context; the two softmax results are summed (decoupled cross-attention):
//   o = softmax(q kt^T / sqrt(d)) vt + softmax(q ki^T / sqrt(d)) vi   per (batch, head).
//
// The contexts are short (512 text and 257 image tokens: 4 and 3 key tiles), so a CTA
// per pair of query tiles would spend much of its life filling and draining its
// pipeline.  This kernel is persistent instead: one CTA per SM walks a list of work
// items (batch, head, pair of 128-row query tiles), numbered so that the CTAs running at
// any moment hold neighbouring items of the same head (the context's keys and values
// stay hot in L2), and its pipeline runs straight across item boundaries.
//   warp 0      TMA producer of the key and value tiles (2-deep rings), text tiles then
//               image tiles of each item, across items
//   warp 2      TMA producer of the query tiles (2-slot ring); it also prefetches the
//               next item's query tiles into L2, so a slot refills from L2 as soon as
//               its tile's last score product is done
//   warp 1      tcgen05.mma from one thread.  Per item: S_0(0), S_1(0); per key tile j:
//               PV_0(j), S_0(j+1) | PV_1(j), S_1(j+1).  The first PV of a segment
//               overwrites O and waits until the softmax warps have read the previous
//               segment's O out of tensor memory, so the next item's first scores are
//               computed while the current item's output is being written.
//   warps 4..11 softmax, one warpgroup per query tile of the item, one thread per query
//               row: fp32 running max and sum per segment with the same lazy rescale as
//               the self-attention kernel; at a segment's end the row sum l goes to
//               shared memory and the warpgroup moves straight on to the next segment.
//   warps 12-15 output: for each segment end of either tile, O out of tensor memory (then
//               O is free for the next segment's first PV product), times 1/l, to 16-bit,
//               through two 4 KB shared-memory boxes per warp (128-byte swizzle) and TMA
//               stores, 64 columns at a time.  One-row-per-thread global stores would
//               send 32 scattered 16-byte pieces per instruction through the SM's memory
//               pipe, whose queue then also holds up the MMA issuer's barrier operations.
//               At the end of the text segment of an image-to-video item the normalised
//               text term is parked in the output rows themselves; at the end of the
//               image segment TMA loads bring it back into the warp's boxes, it is added
//               to the normalised image term in fp32, and the sum is rounded once.
// Tensor memory per query tile: S (128 fp32 columns; P overwrites the first 64) and O
// (d columns): 2 x 256 = 512 columns.  A ragged last key tile (k_lens, or the 257th
// image token) is masked in the softmax, and its products are trimmed: the score MMA
// runs with N = the valid keys rounded up to 16, the PV product over as many 16-key
// slices.
// Number formats: q and k bf16 or fp16 (QK_F16); P, v and o both bf16 or both fp16
// (PV_F16).  With fp16 P the lazy rescale keeps every probability below 2^15.
#include "kernels.h"
#include "wan_common.cuh"

namespace wan {

template <int HD>
struct CrossCfg {
  static constexpr int TILE_BYTES = 128 * HD * 2;  // a 128-row Q, K or V tile: HD/64 boxes of 16 KB
  static constexpr int BOX = 128 * 128;            // bytes per 64-column box
  static constexpr int QSLOTS = 2;
  static constexpr int STAGE_BYTES = 32 * 128;     // one box: 32 rows x 64 columns (16-bit)
  static constexpr int SMEM_TILES = (QSLOTS + 4) * TILE_BYTES + 4 * 2 * STAGE_BYTES;  // 2 boxes per output warp
  static constexpr int LBUF_BYTES = 2 * 128 * 4;   // row sums l of both query tiles
  static constexpr int SMEM = SMEM_TILES + 256 + LBUF_BYTES + 1024;
  static constexpr int TMEM_COLS = 512;
  static constexpr int THREADS = 512;
  // setmaxnreg split of the 512 x 128 registers the CTA launches with.
  static constexpr int PRODUCER_REGS = 80;  // at 72 the issuer's code spills
  static constexpr int SOFTMAX_REGS = 176;
  static constexpr int OUTPUT_REGS = 80;
  static_assert(128 * PRODUCER_REGS + 256 * SOFTMAX_REGS + 128 * OUTPUT_REGS <= 512 * 128, "register split");
  static_assert(SMEM <= 232448, "dynamic shared memory above the per-CTA limit");
};

struct CrossParams {
  int L, H, Lt, Li;    // query rows, heads, text keys, image keys (0: text only)
  int npairs;          // ceil(ceil(L / 128) / 2)
  int n_items;         // B * H * npairs
  int q_col, kt_col, vt_col, ki_col, vi_col;  // column of head 0 in the q / k / v rows
  float scale_log2;    // log2(e) / sqrt(d)
  int o_col;           // column of head 0 in the output rows (written through tmO)
  const int* kt_lens;  // [B] valid text keys per batch entry (clamped to [1, Lt]), or NULL
};

struct CrossItem {
  int b, h, q0, ntile;  // batch entry, head, first query row, query tiles (1 or 2)
  int lt, nkt, nk;      // valid text keys, text key tiles, text + image key tiles
};

__device__ __forceinline__ CrossItem cross_item(const CrossParams& p, int it) {
  CrossItem r;
  const int bh = it / p.npairs;
  const int qp = it - bh * p.npairs;
  r.b = bh / p.H;
  r.h = bh - r.b * p.H;
  r.q0 = qp * 256;
  r.ntile = (r.q0 + 128 < p.L) ? 2 : 1;
  r.lt = p.kt_lens ? min(max(p.kt_lens[r.b], 1), p.Lt) : p.Lt;
  r.nkt = (r.lt + 127) >> 7;
  r.nk = r.nkt + ((p.Li + 127) >> 7);
  return r;
}

// Valid keys of key tile j of an item (1..128).
__device__ __forceinline__ int cross_valid(const CrossParams& p, const CrossItem& I, int j) {
  return j < I.nkt ? min(128, I.lt - j * 128) : min(128, p.Li - (j - I.nkt) * 128);
}

template <bool F16>
__device__ __forceinline__ uint32_t pack16x2(float lo, float hi) {
  if constexpr (F16) return pack_half2(lo, hi);
  else return pack_bf16x2(lo, hi);
}
template <bool F16>
__device__ __forceinline__ float2 unpack16x2(uint32_t u) {
  if constexpr (F16) {
    __half2 h = *reinterpret_cast<__half2*>(&u);
    return __half22float2(h);
  } else {
    return unpack_bf16x2(u);
  }
}

template <int HD, bool QK_F16, bool PV_F16>
__global__ void __launch_bounds__(512, 1)
    attn_cross_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmKt,
                         const __grid_constant__ CUtensorMap tmVt, const __grid_constant__ CUtensorMap tmKi,
                         const __grid_constant__ CUtensorMap tmVi, const __grid_constant__ CUtensorMap tmO,
                         const CrossParams p, int* status) {
  using Cfg = CrossCfg<HD>;
  constexpr int TB = Cfg::TILE_BYTES;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem;                      // [2][TB]
  uint8_t* sK = sQ + Cfg::QSLOTS * TB;     // [2][TB]
  uint8_t* sV = sK + 2 * TB;               // [2][TB]
  uint8_t* sStage = sV + 2 * TB;           // [4 output warps][2 boxes][STAGE_BYTES], 1024-byte aligned
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Cfg::SMEM_TILES);
  uint64_t* q_full = bars + 0;    // [2]
  uint64_t* q_empty = bars + 2;   // [2]
  uint64_t* k_full = bars + 4;    // [2]
  uint64_t* k_empty = bars + 6;   // [2]
  uint64_t* v_full = bars + 8;    // [2]
  uint64_t* v_empty = bars + 10;  // [2]
  uint64_t* s_full = bars + 12;   // [2] per query tile: scores ready
  uint64_t* o_full = bars + 14;   // [2] per query tile: a segment's last PV done
  uint64_t* p_ready = bars + 16;  // [2] per query tile: probabilities in TMEM (4 warps)
  uint64_t* o_free = bars + 18;   // [2] per query tile: O read out of TMEM (4 warps)
  uint64_t* drain = bars + 20;
  uint64_t* parked_full = bars + 21;  // [4] per output warp: parked text term back in its boxes
  uint64_t* l_ready = bars + 25;      // [2] per query tile: a segment's row sums in l_buf (4 warps)
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + 27);
  float* l_buf = reinterpret_cast<float*>(smem + Cfg::SMEM_TILES + 256);  // [2][128]

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < Cfg::QSLOTS; ++s) {
      mbar_init(&q_full[s], 1);
      mbar_init(&q_empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&k_empty[s], 1);
      mbar_init(&v_full[s], 1);
      mbar_init(&v_empty[s], 1);
      mbar_init(&s_full[s], 1);
      mbar_init(&o_full[s], 1);
      mbar_init(&p_ready[s], 4);
      mbar_init(&o_free[s], 4);
      mbar_init(&l_ready[s], 4);
    }
    mbar_init(drain, 1);
    for (int w = 0; w < 4; ++w) mbar_init(&parked_full[w], 1);
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
      // ------------------------------------------------------------ key/value producer
      tma_prefetch_desc(&tmKt);
      tma_prefetch_desc(&tmVt);
      if (p.Li) {
        tma_prefetch_desc(&tmKi);
        tma_prefetch_desc(&tmVi);
      }
      uint32_t kissued = 0, vissued = 0;
      bool ok = true;
      for (int it = blockIdx.x; it < p.n_items && ok; it += gridDim.x) {
        const CrossItem I = cross_item(p, it);
        for (int j = 0; j < I.nk; ++j) {
          const bool img = j >= I.nkt;
          const int row = (img ? j - I.nkt : j) * 128;
          const CUtensorMap* tk = img ? &tmKi : &tmKt;
          const CUtensorMap* tv = img ? &tmVi : &tmVt;
          const int kc = (img ? p.ki_col : p.kt_col) + I.h * HD;
          const int vc = (img ? p.vi_col : p.vt_col) + I.h * HD;
          const uint32_t s = kissued & 1, ph = (kissued >> 1) & 1;
          if (!mbar_wait(&k_empty[s], ph ^ 1, status, kDevTimeoutAttn)) { ok = false; break; }
          mbar_arrive_expect_tx(&k_full[s], TB);
          for (int c = 0; c < HD / 64; ++c)
            tma_load_3d(sK + s * TB + c * Cfg::BOX, tk, &k_full[s], kc + c * 64, row, I.b);
          ++kissued;
          if (!mbar_wait(&v_empty[s], ph ^ 1, status, kDevTimeoutAttn)) { ok = false; break; }
          mbar_arrive_expect_tx(&v_full[s], TB);
          for (int c = 0; c < HD / 64; ++c)
            tma_load_3d(sV + s * TB + c * Cfg::BOX, tv, &v_full[s], vc + c * 64, row, I.b);
          ++vissued;
        }
      }
      if (!ok) {  // error path: let the copies in flight land before the CTA exits
        const unsigned long long t0 = globaltimer_ns();
        for (uint32_t n = (kissued > 2 ? kissued - 2 : 0); n < kissued; ++n)
          while (!mbar_test(&k_full[n & 1], (n >> 1) & 1) && globaltimer_ns() - t0 < kWaitLimitNs) {}
        for (uint32_t n = (vissued > 2 ? vissued - 2 : 0); n < vissued; ++n)
          while (!mbar_test(&v_full[n & 1], (n >> 1) & 1) && globaltimer_ns() - t0 < kWaitLimitNs) {}
      }
    } else if (warp == 2 && lane == 0) {
      // ------------------------------------------------------------ query producer
      tma_prefetch_desc(&tmQ);
      uint32_t g = 0;
      bool ok = true;
      for (int it = blockIdx.x; it < p.n_items && ok; it += gridDim.x) {
        const CrossItem I = cross_item(p, it);
        if (it + (int)gridDim.x < p.n_items) {  // the next item's query tiles into L2
          const CrossItem N = cross_item(p, it + gridDim.x);
          for (int i = 0; i < N.ntile; ++i)
            for (int c = 0; c < HD / 64; ++c) tma_prefetch_l2_3d(&tmQ, p.q_col + N.h * HD + c * 64, N.q0 + i * 128, N.b);
        }
        for (int i = 0; i < I.ntile; ++i) {
          const uint32_t s = g & 1, ph = (g >> 1) & 1;
          if (!mbar_wait(&q_empty[s], ph ^ 1, status, kDevTimeoutAttn)) { ok = false; break; }
          mbar_arrive_expect_tx(&q_full[s], TB);
          for (int c = 0; c < HD / 64; ++c)
            tma_load_3d(sQ + s * TB + c * Cfg::BOX, &tmQ, &q_full[s], p.q_col + I.h * HD + c * 64, I.q0 + i * 128,
                        I.b);
          ++g;
        }
      }
      if (!ok) {
        const unsigned long long t0 = globaltimer_ns();
        for (uint32_t n = (g > 2 ? g - 2 : 0); n < g; ++n)
          while (!mbar_test(&q_full[n & 1], (n >> 1) & 1) && globaltimer_ns() - t0 < kWaitLimitNs) {}
      }
    } else if (warp == 1 && lane == 0) {
      // ------------------------------------------------------------ MMA issuer
      constexpr uint32_t idO = (PV_F16 ? make_idesc_f16(128, HD) : make_idesc_bf16(128, HD)) | kIdescBMnMajor;
      const uint32_t q_lo = sdesc_sw128_lo(smem_u32(sQ));
      const uint32_t k_lo = sdesc_sw128_lo(smem_u32(sK));
      const uint32_t v_lo = sdesc_sw128_mn_lo(smem_u32(sV), Cfg::BOX);
      // S_i = Q_i K^T over the first n keys of the tile in K slot ks (n a multiple of 16).
      auto issue_S = [&](int i, uint32_t qa, int ks, int n) {
        const uint32_t ka = k_lo + (uint32_t)ks * (TB >> 4);
        const uint32_t id = QK_F16 ? make_idesc_f16(128, n) : make_idesc_bf16(128, n);
        const uint32_t d = tmem_base + i * 256;
#pragma unroll
        for (int kk = 0; kk < HD / 16; ++kk) {
          const uint32_t off = ((kk >> 2) * Cfg::BOX + (kk & 3) * 32) >> 4;
          tc_mma_ss_lo(d, qa + off, ka + off, id, kk > 0 ? 1u : 0u);
        }
      };
      // O_i (+)= P_i V over the first nsub 16-key slices of the tile in V slot vs.
      auto issue_PV = [&](int i, int vs, int nsub, uint32_t acc) {
        const uint32_t va = v_lo + (uint32_t)vs * (TB >> 4);
        const uint32_t d = tmem_base + i * 256 + 128;
        const uint32_t pa = tmem_base + i * 256;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          if (kk < nsub) tc_mma_ts_lo(d, pa + kk * 8, va + ((kk * 16 * 128) >> 4), idO, (acc | (uint32_t)kk) != 0 ? 1u : 0u);
      };
      // Compact per-item state (the issuer runs within the producers' register budget):
      // query tiles, text key tiles, all key tiles, valid text keys.
      struct Shape {
        int ntile, nkt, nk, lt;
      };
      auto shape_of = [&](int it) -> Shape {
        const CrossItem I = cross_item(p, it);
        return Shape{I.ntile, I.nkt, I.nk, I.lt};
      };
      auto valid_of = [&](const Shape& S, int j) -> int {
        return j < S.nkt ? min(128, S.lt - j * 128) : min(128, p.Li - (j - S.nkt) * 128);
      };
      uint32_t g = 0, c = 0;            // first query tile / key tile of the current item
      uint32_t pr0 = 0, pr1 = 0;        // p_ready phases waited, per query tile slot
      uint32_t sg0 = 0, sg1 = 0;        // segments started, per query tile slot
      bool ok = true;
      // S_i(0) of an item with shape S whose first query tile is gq and first key tile ck.
      auto first_scores = [&](const Shape& S, int i, uint32_t gq, uint32_t ck) -> bool {
        const uint32_t t = gq + i;
        if (!mbar_wait(&q_full[t & 1], (t >> 1) & 1, status, kDevTimeoutAttn)) return false;
        tc_fence_after();
        issue_S(i, q_lo + (t & 1) * (TB >> 4), ck & 1, (valid_of(S, 0) + 15) & ~15);
        if (S.nk == 1) tc_commit(&q_empty[t & 1]);
        tc_commit(&s_full[i]);
        return true;
      };
      int it = blockIdx.x;
      Shape I = shape_of(it < p.n_items ? it : 0);
      if (it < p.n_items) {
        ok = mbar_wait(&k_full[0], 0, status, kDevTimeoutAttn);
        for (int i = 0; i < I.ntile && ok; ++i) ok = first_scores(I, i, 0, 0);
        if (ok) tc_commit(&k_empty[0]);
      }
      // Each tile's next scores follow its PV product, across item boundaries too: at an
      // item's last key tile, S_i of the next item's first key tile comes right behind
      // PV_i, exactly like S_i(j+1) within an item.
#pragma unroll 1
      while (it < p.n_items && ok) {
        const int nit = it + (int)gridDim.x;
        const bool has_next = nit < p.n_items;
        const Shape N = shape_of(has_next ? nit : it);
        const uint32_t gn = g + I.ntile, cn = c + I.nk;
#pragma unroll 1
        for (int j = 0; j < I.nk && ok; ++j) {
          const uint32_t cj = c + j;
          const int vs = cj & 1;
          const bool more = j + 1 < I.nk;
          const bool seg_first = (j == 0 || j == I.nkt);
          const bool seg_last = (j == I.nkt - 1 || j == I.nk - 1);
          if (!mbar_wait(&v_full[vs], (cj >> 1) & 1, status, kDevTimeoutAttn)) { ok = false; break; }
          const uint32_t kn = more ? cj + 1 : cn;  // the key tile of the next score product
          if ((more || has_next) && !mbar_wait(&k_full[kn & 1], (kn >> 1) & 1, status, kDevTimeoutAttn)) {
            ok = false;
            break;
          }
          uint32_t deferred = 0;  // next-item first score products waiting for their query tile
#pragma unroll 1
          for (int i = 0; i < I.ntile; ++i) {
            uint32_t& pr = i ? pr1 : pr0;
            uint32_t& sg = i ? sg1 : sg0;
            if (!mbar_wait(&p_ready[i], pr & 1, status, kDevTimeoutAttn)) { ok = false; break; }
            ++pr;
            if (seg_first) {
              if (sg > 0 && !mbar_wait(&o_free[i], (sg - 1) & 1, status, kDevTimeoutAttn)) { ok = false; break; }
              ++sg;
            }
            tc_fence_after();
            issue_PV(i, vs, (valid_of(I, j) + 15) >> 4, seg_first ? 0u : 1u);
            if (seg_last) tc_commit(&o_full[i]);
            if (more) {
              issue_S(i, q_lo + ((g + i) & 1) * (TB >> 4), kn & 1, (valid_of(I, j + 1) + 15) & ~15);
              if (j + 2 == I.nk) tc_commit(&q_empty[(g + i) & 1]);
              tc_commit(&s_full[i]);
            } else if (has_next && i < N.ntile) {
              // Only if its query tile has landed: otherwise it would hold up the other
              // tile's PV product; it is then issued after the loop.
              const uint32_t t = gn + i;
              if (mbar_test(&q_full[t & 1], (t >> 1) & 1)) {
                if (!first_scores(N, i, gn, cn)) { ok = false; break; }
              } else {
                deferred |= 1u << i;
              }
            }
          }
          if (!ok) break;
          if (!more && has_next)
            for (int i = 0; i < N.ntile && ok; ++i)
              if (i >= I.ntile || ((deferred >> i) & 1)) ok = first_scores(N, i, gn, cn);
          tc_commit(&v_empty[vs]);
          if (more || has_next) tc_commit(&k_empty[kn & 1]);
        }
        g = gn;
        c = cn;
        it = nit;
        I = N;
      }
      if (!ok) {  // error path: wait for the MMAs in flight before TMEM is released
        tc_commit(drain);
        const unsigned long long t0 = globaltimer_ns();
        while (!mbar_test(drain, 0) && globaltimer_ns() - t0 < kWaitLimitNs) {}
      }
    }
  } else if (warp < 12) {
    // -------------------------------------------------------------- softmax
    regs_inc<Cfg::SOFTMAX_REGS>();
    const int i = (warp - 4) >> 2;  // query tile of the item that this warpgroup owns
    const int quad = warp & 3;      // TMEM lane quadrant of this warp
    const uint32_t tS = tmem_base + ((uint32_t)(quad * 32) << 16) + i * 256;
    const uint32_t tO = tS + 128;
    const uint64_t sl2x2 = f2_pack(p.scale_log2, p.scale_log2);
    // A tile row sum above this bound takes the slow path (new max, rescale): it keeps
    // every probability representable in P's format.
    const float sum_bound = PV_F16 ? 32768.0f : 65536.0f;
    uint32_t sph = 0;
    bool ok = true;
    uint32_t sr[128];
    auto load_scores = [&](int valid) {
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_ld32_nowait(tS + c * 32, sr + c * 32);
      tmem_wait_ld();
      if (valid < 128) {
#pragma unroll
        for (int e = 0; e < 128; ++e)
          if (e >= valid) sr[e] = __float_as_uint(-INFINITY);
      }
    };
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
          sr[c * 32 + e] = pack16x2<PV_F16>(p0, p1);
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
    auto row_max = [&]() -> float {
      float mx0 = __uint_as_float(sr[0]), mx1 = __uint_as_float(sr[1]);
      float mx2 = __uint_as_float(sr[2]), mx3 = __uint_as_float(sr[3]);
#pragma unroll
      for (int e = 4; e < 124; e += 8) {
        mx0 = fmax3(mx0, __uint_as_float(sr[e]), __uint_as_float(sr[e + 1]));
        mx1 = fmax3(mx1, __uint_as_float(sr[e + 2]), __uint_as_float(sr[e + 3]));
        mx2 = fmax3(mx2, __uint_as_float(sr[e + 4]), __uint_as_float(sr[e + 5]));
        mx3 = fmax3(mx3, __uint_as_float(sr[e + 6]), __uint_as_float(sr[e + 7]));
      }
      mx0 = fmax3(mx0, __uint_as_float(sr[124]), __uint_as_float(sr[125]));
      mx1 = fmax3(mx1, __uint_as_float(sr[126]), __uint_as_float(sr[127]));
      return fmax3(mx0, mx1, fmaxf(mx2, mx3));
    };
    const int nki = (p.Li + 127) >> 7;
    for (int it = blockIdx.x; it < p.n_items && ok; it += gridDim.x) {
      const CrossItem I = cross_item(p, it);
      if (i >= I.ntile) continue;
      for (int seg = 0; seg < (p.Li ? 2 : 1) && ok; ++seg) {
        const int ntiles = seg ? nki : I.nkt;
        const int seglen = seg ? p.Li : I.lt;
        float m_used = -INFINITY, l_sum = 0.f;
        for (int jj = 0; jj < ntiles; ++jj) {
          if (!mbar_wait_warp(&s_full[i], sph & 1, status, kDevTimeoutAttn)) { ok = false; break; }
          ++sph;
          tc_fence_after();
          const int valid = min(128, seglen - jj * 128);
          load_scores(valid);
          float rowsum;
          if (jj == 0) {
            m_used = row_max() * p.scale_log2;
            exp_pass(m_used, rowsum);
          } else {
            exp_pass(m_used, rowsum);
            const bool need = !(rowsum <= sum_bound);
            if (__any_sync(0xffffffffu, need)) {
              load_scores(valid);
              const float mt = row_max() * p.scale_log2;
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
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&p_ready[i]);
        }
        if (!ok) break;
        // The segment's row sums for the output warps (the arrival releases the store).
        l_buf[i * 128 + quad * 32 + lane] = l_sum;
        __syncwarp();
        if (lane == 0) mbar_arrive(&l_ready[i]);
      }
    }
  } else {
    // -------------------------------------------------------------- output
    regs_dec<Cfg::OUTPUT_REGS>();
    const int quad = warp & 3;  // TMEM lane quadrant = this warp's 32 rows of a query tile
    uint8_t* box0 = sStage + quad * 2 * Cfg::STAGE_BYTES;
    const uint32_t row_off = lane * 128;  // this thread's 128-byte row within a box
    uint32_t ph0 = 0, ph1 = 0;  // segment ends handled so far, per query tile (l_ready / o_full phases)
    uint32_t pkph = 0;
    bool parked_pending = false;  // a TMA load into this warp's boxes not yet waited for
    bool ok = true;
    for (int it = blockIdx.x; it < p.n_items && ok; it += gridDim.x) {
      const CrossItem I = cross_item(p, it);
      for (int seg = 0; seg < (p.Li ? 2 : 1) && ok; ++seg) {
        // Output of the segment: O / l (+ the parked text term at the end of the image
        // segment) -> 16-bit -> boxes -> TMA stores.  At the end of a text segment followed
        // by an image segment the same path parks the normalised text term in the output.
        const bool combine = seg == 1;
        for (int i = 0; i < I.ntile && ok; ++i) {
          const int row0 = I.q0 + i * 128 + quad * 32;
          const int ocol = p.o_col + I.h * HD;
          if (lane == 0) {
            if (combine) {
              bulk_wait_group_all();  // the parked text term is written, the boxes are free
              mbar_arrive_expect_tx(&parked_full[quad], (HD / 64) * Cfg::STAGE_BYTES);
              for (int half = 0; half < HD / 64; ++half)
                tma_load_3d(box0 + half * Cfg::STAGE_BYTES, &tmO, &parked_full[quad], ocol + half * 64, row0, I.b);
            } else {
              bulk_wait_group_read<0>();  // earlier stores out of the boxes have read them
            }
          }
          parked_pending = combine;
          __syncwarp();
          uint32_t& ph = i ? ph1 : ph0;
          if (!mbar_wait_warp(&l_ready[i], ph & 1, status, kDevTimeoutAttn) ||
              !mbar_wait_warp(&o_full[i], ph & 1, status, kDevTimeoutAttn)) {
            ok = false;
            break;
          }
          ++ph;
          tc_fence_after();
          const float inv = 1.0f / l_buf[i * 128 + quad * 32 + lane];
          if (combine) {
            if (!mbar_wait_warp(&parked_full[quad], pkph & 1, status, kDevTimeoutAttn)) { ok = false; break; }
            ++pkph;
            parked_pending = false;
          }
          const uint32_t tO = tmem_base + ((uint32_t)(quad * 32) << 16) + i * 256 + 128;
#pragma unroll 1
          for (int c = 0; c < HD / 32; ++c) {
            uint32_t orr[32];
            tmem_ld32(tO + c * 32, orr);
            if (c == HD / 32 - 1) {  // O is read: the next segment's first PV may overwrite it
              tc_fence_before();
              __syncwarp();
              if (lane == 0) mbar_arrive(&o_free[i]);
            }
            const uint32_t box_row = smem_u32(box0 + (c >> 1) * Cfg::STAGE_BYTES) + row_off;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const uint32_t addr = box_row + ((uint32_t)(((c & 1) * 4 + e) ^ (lane & 7)) << 4);
              float v[8];
#pragma unroll
              for (int u = 0; u < 8; ++u) v[u] = __uint_as_float(orr[e * 8 + u]) * inv;
              if (combine) {
                const uint4 pw4 = ld_shared_v4(addr);
                const uint32_t pw[4] = {pw4.x, pw4.y, pw4.z, pw4.w};
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                  const float2 f = unpack16x2<PV_F16>(pw[u]);
                  v[2 * u] += f.x;
                  v[2 * u + 1] += f.y;
                }
              }
              uint4 o4;
              o4.x = pack16x2<PV_F16>(v[0], v[1]);
              o4.y = pack16x2<PV_F16>(v[2], v[3]);
              o4.z = pack16x2<PV_F16>(v[4], v[5]);
              o4.w = pack16x2<PV_F16>(v[6], v[7]);
              st_shared_v4(addr, o4);
            }
            if (c & 1) {  // a 64-column box is complete: store it
              fence_proxy_async_smem();
              __syncwarp();
              if (lane == 0) {
                tma_store_3d(&tmO, box0 + (c >> 1) * Cfg::STAGE_BYTES, ocol + (c >> 1) * 64, row0, I.b);
                bulk_commit_group();
              }
            }
          }
        }
      }
    }
    if (lane == 0) {
      bulk_wait_group_all();  // this warp's stores are complete before the CTA exits
      if (parked_pending) {   // error path: let the loads into the boxes land first
        const unsigned long long t0 = globaltimer_ns();
        while (!mbar_test(&parked_full[quad], pkph & 1) && globaltimer_ns() - t0 < kWaitLimitNs) {}
      }
    }
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem_base, Cfg::TMEM_COLS);
}

template <int HD, bool QK_F16, bool PV_F16>
static int launch_cross(const LaunchCtx& c, const CUtensorMap (&tm)[6], const CrossParams& p, const char* tag) {
  using Cfg = CrossCfg<HD>;
  static std::atomic<unsigned long long> smem_set{0};
  const int st = set_smem_limit_once(reinterpret_cast<const void*>(attn_cross_tc_kernel<HD, QK_F16, PV_F16>),
                                     Cfg::SMEM, &smem_set);
  if (st != WAN_OK) return st;
  const int grid = p.n_items < c.num_sms ? p.n_items : c.num_sms;
  count_launch(tag, c.stream, true);
  attn_cross_tc_kernel<HD, QK_F16, PV_F16><<<grid, Cfg::THREADS, Cfg::SMEM, c.stream>>>(tm[0], tm[1], tm[2], tm[3],
                                                                                       tm[4], tm[5], p, c.dev_status);
  count_launch(tag, c.stream, false);
  return cudaGetLastError() == cudaSuccess ? WAN_OK : WAN_ERR_CUDA;
}

int cross_attention_tc(const LaunchCtx& c, const CrossArgs& a) {
  if (a.head_dim != 64 && a.head_dim != 128) return WAN_ERR_UNSUPPORTED;
  if (a.pv_f16 && !a.qk_f16) return WAN_ERR_UNSUPPORTED;
  if (a.L <= 0) return WAN_OK;
  if (a.Lt <= 0 || a.Li < 0 || (a.Li > 0 && (!a.ki || !a.vi))) return WAN_ERR_INVALID_ARG;
  const int HD = a.head_dim;
  const CUtensorMapDataType qkt = a.qk_f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const CUtensorMapDataType pvt = a.pv_f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  CUtensorMap tm[6];
  int st = make_tmap_3d(&tm[0], a.q, qkt, 2, (uint64_t)a.q_row_len, (uint64_t)a.L, (uint64_t)a.B,
                        (uint64_t)a.ldq * 2, (uint64_t)a.ldq * 2 * a.L, 64, 128);
  if (st != WAN_OK) return st;
  st = make_tmap_3d(&tm[1], a.kt, qkt, 2, (uint64_t)a.kt_row_len, (uint64_t)a.Lt, (uint64_t)a.B,
                    (uint64_t)a.ldkt * 2, (uint64_t)a.ldkt * 2 * a.Lt, 64, 128);
  if (st != WAN_OK) return st;
  st = make_tmap_3d(&tm[2], a.vt, pvt, 2, (uint64_t)a.vt_row_len, (uint64_t)a.Lt, (uint64_t)a.B,
                    (uint64_t)a.ldvt * 2, (uint64_t)a.ldvt * 2 * a.Lt, 64, 128);
  if (st != WAN_OK) return st;
  if (a.Li > 0) {
    st = make_tmap_3d(&tm[3], a.ki, qkt, 2, (uint64_t)a.ki_row_len, (uint64_t)a.Li, (uint64_t)a.B,
                      (uint64_t)a.ldki * 2, (uint64_t)a.ldki * 2 * a.Li, 64, 128);
    if (st != WAN_OK) return st;
    st = make_tmap_3d(&tm[4], a.vi, pvt, 2, (uint64_t)a.vi_row_len, (uint64_t)a.Li, (uint64_t)a.B,
                      (uint64_t)a.ldvi * 2, (uint64_t)a.ldvi * 2 * a.Li, 64, 128);
    if (st != WAN_OK) return st;
  } else {
    tm[3] = tm[1];  // unused: no image segment
    tm[4] = tm[2];
  }
  // Output rows [B, L, ldo] (16-bit), 32-row x 64-column boxes: the softmax warps' stores.
  st = make_tmap_3d(&tm[5], a.o, pvt, 2, (uint64_t)a.ldo, (uint64_t)a.L, (uint64_t)a.B, (uint64_t)a.ldo * 2,
                    (uint64_t)a.ldo * 2 * a.L, 64, 32);
  if (st != WAN_OK) return st;
  CrossParams p;
  p.L = a.L;
  p.H = a.H;
  p.Lt = a.Lt;
  p.Li = a.Li;
  p.npairs = ((a.L + 127) / 128 + 1) / 2;
  const long long items = (long long)a.B * a.H * p.npairs;
  if (items > 0x7fffffffLL) return WAN_ERR_UNSUPPORTED;
  p.n_items = (int)items;
  p.q_col = a.q_col;
  p.kt_col = a.kt_col;
  p.vt_col = a.vt_col;
  p.ki_col = a.ki_col;
  p.vi_col = a.vi_col;
  p.scale_log2 = 1.4426950408889634f / sqrtf((float)HD);
  p.o_col = a.o_col;
  p.kt_lens = a.kt_lens;
  const char* tag = a.tag ? a.tag : "attn_cross";
  if (HD == 128) {
    if (a.pv_f16) return launch_cross<128, true, true>(c, tm, p, tag);
    return a.qk_f16 ? launch_cross<128, true, false>(c, tm, p, tag) : launch_cross<128, false, false>(c, tm, p, tag);
  }
  if (a.pv_f16) return launch_cross<64, true, true>(c, tm, p, tag);
  return a.qk_f16 ? launch_cross<64, true, false>(c, tm, p, tag) : launch_cross<64, false, false>(c, tm, p, tag);
}

}  // namespace wan

// fwd_duo.cuh -- attention forward for Dqk = Dv = D in {64, 128} (sm_103a),
// two CTAs per SM.
//   [nemo_automodel.components.attention.ffpa_attention, `_ffpa_varlen_fwd`,
//    `_ffpa_dense_fwd`; causal mask at each segment's bottom-right corner per
//    nemo_automodel.components.attention.fa4, module docstring bullet 2; left
//    window counting the current token per the attention utils page]
//
// Same result as attn_fwd_kernel in fwd.cuh, arranged so that two CTAs share
// an SM: while one CTA's softmax warps work on a score tile, the other CTA's
// MMAs keep the tensor core busy. Each CTA runs, per 128-row query tile,
//   S_j = Q K_j^T  ->  softmax  ->  O += P_j V_j      for every key tile j
// strictly in that order, so a single S buffer suffices.
//   TMEM  256 columns per CTA: S, then P (bf16 over S's first 64 columns)
//         [0, 128) | O [128, 128 + D)
//   Pack  with p.pack = G = Hq / Hkv > 1 the 128-row tile holds the G query
//         heads of one KV head, 128 / G rows each (one TMA box of 128/G rows x G
//         heads), so short segments fill the tile and K/V load once for all G.
//   SMEM  the Q tile and two tile slots that K_j and V_j pass through in turn
//         (D / 64 chunks of 128 rows x 64 columns, 128-byte swizzled each).
//   PV    one N = D MMA chain over a whole V tile: the B operand is MN-major and
//         its 64-column chunks are reached through the leading-byte offset.
//   warps 0-3  softmax, thread t = query row t (TMEM lane t). One pass per
//              key tile: the row of S into registers, its maximum, then P
//              written over S's first columns and the row sum. The running
//              maximum is raised only when it grows by more than 2^8, and only
//              then is O rescaled (the final division by the row sum cancels
//              any common factor). The tile's epilogue divides O by the sum and
//              stores out and lse.
//   warp 4     TMA producer.
//   warp 5     TMEM allocator and MMA issuer.
// The commit that signals S_j also covers PV_{j-1} (a commit tracks every
// earlier MMA of the issuing thread), so the softmax may rescale O as soon as
// S_j is ready.
// Work: each CTA starts on work item blockIdx.x of the heaviest-first list and
// then takes the next untaken item from a global counter, so SMs that finish
// early pick up the remaining items. The producer takes the item, decodes it
// while the previous item's tiles load, and passes index and decoded tile to
// the MMA and softmax warps through a two-entry ring in shared memory (-1 = no
// more work).
// Both softmax passes exist in two forms: one for tiles that cross a mask edge
// and one, free of any mask arithmetic, for the rest.
#pragma once

#include <math_constants.h>

#include "fwd.cuh"

namespace psf {

template <int D>
struct FwdDuoCfg {
  static constexpr int CH = D / 64;
  static constexpr int TILE_BYTES = CH * kChunkBytes;
  static constexpr int Q_OFF = 0;
  static constexpr int SLOT_OFF = TILE_BYTES;  // two slots
  static constexpr int STG_OFF = 3 * TILE_BYTES;  // epilogue staging: 4 softmax warps x (32 rows x 64 B)
  static constexpr int SMEM_USED = STG_OFF + 4 * 2048 + 1024;
  // Never more than two CTAs per SM: a third could not allocate its TMEM.
  static constexpr int SMEM_BYTES = SMEM_USED > 80 * 1024 ? SMEM_USED : 80 * 1024;
  static constexpr int T_S = 0;
  static constexpr int T_O = 128;
  static constexpr int TMEM_COLS = 256;
  static_assert(D == 64 || D == 128, "two-CTA forward covers head dims 64 and 128");
  static_assert(2 * (SMEM_BYTES + 2048) <= 233472, "two CTAs per SM");
  static_assert(3 * (SMEM_BYTES + 1024) > 233472, "at most two CTAs per SM");
};

// CAP: logits softcapped (p.softcap > 0), applied to the score registers in
// place before the row maximum.
template <typename T, int D, bool CAP>
__global__ void __launch_bounds__(192, 2) attn_fwd_duo_kernel(const __grid_constant__ FwdParams p) {
  using C = FwdDuoCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

  __shared__ uint64_t q_full, q_empty, slot_full[2], slot_empty[2], s_full, p_full, pv_done, o_free, drain;
  __shared__ uint64_t work_full[2], work_empty[2];
  __shared__ int work_slot[2];
  __shared__ FwdTile work_tile[2];
  __shared__ uint32_t tmem_base_smem;
  __shared__ int abort_flag;

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  if (threadIdx.x == 0) {
    mbar_init(&q_full, 1);
    mbar_init(&q_empty, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&slot_full[i], 1);
      mbar_init(&slot_empty[i], 1);
    }
    mbar_init(&s_full, 1);
    mbar_init(&p_full, 4);
    mbar_init(&pv_done, 1);
    mbar_init(&o_free, 4);
    mbar_init(&drain, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&work_full[i], 1);
      mbar_init(&work_empty[i], 5);  // the MMA thread and the four softmax warps
    }
    abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 5) {
    tmem_alloc(&tmem_base_smem, C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_smem;
  const Ctl ctl{p.status, p.limit_ns, &abort_flag};
  const int total = (*p.n_items) * (p.Hq / p.pack);
  const int G = p.Hq / p.Hkv;
  // Next work item for the MMA and softmax warps (-1: none left, or abort),
  // with its decoded tile.
  uint32_t nwork = 0;
  auto next_work = [&](bool& ok, FwdTile& t) -> int {
    const int ws = nwork & 1;
    if (!wait_bar(&work_full[ws], (nwork >> 1) & 1, ctl)) {
      ok = false;
      return -1;
    }
    const int w = work_slot[ws];
    t = work_tile[ws];
    __syncwarp(__activemask());
    if (lane == 0) mbar_arrive(&work_empty[ws]);
    ++nwork;
    return w;
  };

  if (warp == 4) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&p.tm_q);
      tma_prefetch_desc(&p.tm_k);
      tma_prefetch_desc(&p.tm_v);
      uint32_t qcnt = 0, it = 0;
      bool ok = true;
      auto load_tile = [&](const CUtensorMap* map, int row, int h, int b) -> bool {
        const int sl = it & 1;
        if (!wait_bar(&slot_empty[sl], ((it >> 1) & 1) ^ 1, ctl)) return false;
        mbar_arrive_expect_tx(&slot_full[sl], C::TILE_BYTES);
        for (int c = 0; c < C::CH; ++c)
          tma_load_4d(smem + C::SLOT_OFF + sl * C::TILE_BYTES + c * kChunkBytes, map, &slot_full[sl], c * 64, row, h,
                      b);
        ++it;
        return true;
      };
      // Each item is decoded (two dependent global reads) while the previous
      // one's tiles are still being loaded, and published decoded.
      int w = blockIdx.x;
      FwdTile tw{};
      if (w < total) tw = fwd_decode(p, w);
      while (true) {
        if (w >= total) w = -1;
        const int ws = nwork & 1;
        if (!wait_bar(&work_empty[ws], ((nwork >> 1) & 1) ^ 1, ctl)) break;
        work_slot[ws] = w;
        work_tile[ws] = tw;
        mbar_arrive(&work_full[ws]);
        ++nwork;
        if (w < 0) break;
        const FwdTile t = tw;
        const int wn = gridDim.x + atomicAdd(p.work_next, 1);
        bool decoded = false;
        if (t.nk > 0) {
          if (!wait_bar(&q_empty, (qcnt & 1) ^ 1, ctl)) break;
          mbar_arrive_expect_tx(&q_full, C::TILE_BYTES);
          const int fq = t.cq0 + t.qt * p.seg.qrows, bq = fq / p.seg.Sq;
          for (int c = 0; c < C::CH; ++c)
            tma_load_4d(smem + C::Q_OFF + c * kChunkBytes, &p.tm_q, &q_full, c * 64, fq - bq * p.seg.Sq, t.h, bq);
          ++qcnt;
          const int hk = t.h / G;
          for (int jj = 0; jj < t.nk && ok; ++jj) {
            const int fk = t.ck0 + (t.kv_t0 + jj) * kBN, bk = fk / p.seg.Sk, sk = fk - bk * p.seg.Sk;
            ok = load_tile(&p.tm_k, sk, hk, bk) && load_tile(&p.tm_v, sk, hk, bk);
            if (jj == 0 && wn < total) {
              tw = fwd_decode(p, wn);
              decoded = true;
            }
          }
          if (!ok) break;
        }
        if (!decoded && wn < total) tw = fwd_decode(p, wn);
        w = wn;
      }
      // Wind down: no copy may still be landing in shared memory.
      for (uint32_t i = it > 2u ? it - 2 : 0; i < it; ++i) wait_bar_drain(&slot_full[i & 1], (i >> 1) & 1, p.limit_ns);
      if (qcnt > 0) wait_bar_drain(&q_full, (qcnt - 1) & 1, p.limit_ns);
    }
  } else if (warp == 5) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t id_qk = idesc_f32acc<T>(128, 128, 0, 0);
      constexpr uint32_t id_pv = idesc_f32acc<T>(128, D, 0, 1);
      const uint32_t q_a = smem_u32(smem + C::Q_OFF), slot_a = smem_u32(smem + C::SLOT_OFF);
      uint32_t qcnt = 0, it = 0, kv = 0, ntile = 0;
      bool ok = true;
      while (ok) {
        FwdTile t;
        const int w = next_work(ok, t);
        if (w < 0) break;
        if (t.nk == 0) continue;
        if (!wait_bar(&q_full, qcnt & 1, ctl)) break;
        tc_fence_after();
        for (int jj = 0; jj < t.nk; ++jj) {
          // S = Q K_j^T
          int sl = it & 1;
          if (!wait_bar(&slot_full[sl], (it >> 1) & 1, ctl)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t k_a = slot_a + sl * C::TILE_BYTES;
#pragma unroll
          for (int c = 0; c < C::CH; ++c)
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              mma_ss(tmem + C::T_S, sdesc_sw128(q_a + c * kChunkBytes + kk * 32, 16, 1024),
                     sdesc_sw128(k_a + c * kChunkBytes + kk * 32, 16, 1024), id_qk, (c | kk) != 0);
          mma_commit(&slot_empty[sl]);
          ++it;
          mma_commit(&s_full);
          if (jj == t.nk - 1) mma_commit(&q_empty);
          // O (+)= P V_j once the softmax has written P (and, on a tile's first
          // key tile, once the previous tile's epilogue has read O). V_j is
          // waited for first: it lands while the softmax runs, so the wait on
          // P is the last step before the PV issue.
          sl = it & 1;
          if (!wait_bar(&slot_full[sl], (it >> 1) & 1, ctl)) {
            ok = false;
            break;
          }
          if (jj == 0 && ntile > 0 && !wait_bar(&o_free, (ntile - 1) & 1, ctl)) {
            ok = false;
            break;
          }
          if (!wait_bar(&p_full, kv & 1, ctl)) {
            ok = false;
            break;
          }
          ++kv;
          tc_fence_after();
          const uint32_t v_a = slot_a + sl * C::TILE_BYTES;
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            mma_ts(tmem + C::T_O, tmem + C::T_S + kk * 8, sdesc_sw128(v_a + kk * 2048, kChunkBytes, 1024), id_pv,
                   (jj > 0 || kk > 0));
          mma_commit(&slot_empty[sl]);
          ++it;
        }
        if (!ok) break;
        mma_commit(&pv_done);
        ++qcnt;
        ++ntile;
      }
      // Wind down: wait until every MMA this thread issued has finished.
      mma_commit(&drain);
      wait_bar_drain(&drain, 0, p.limit_ns);
    }
  } else {
    // ------------------------------------------------------------ softmax warpgroup
    const int row = threadIdx.x;
    const uint32_t lane_base = (uint32_t)(32 * warp) << 16;
    const uint32_t ts = tmem + lane_base + C::T_S, to = tmem + lane_base + C::T_O;
    const float sl2 = p.scale_log2;
    const float2 zero2 = make_float2(0.f, 0.f);
    // With CAP the score registers hold capped logits in log2 units already.
    const float mul = CAP ? 1.f : sl2;
    const float2 mul2 = make_float2(mul, mul);
    const float cap_k1 = CAP ? 2.f * sl2 / p.softcap : 0.f, cap_c2 = CAP ? p.softcap * 1.4426950408889634f : 0.f;
    uint32_t kv = 0, ntile = 0;
    bool ok = true;
    while (ok) {
      FwdTile t;
      const int w = next_work(ok, t);
      if (w < 0) break;
      // TMEM lane / tile row -> (query head, segment-local query index): the
      // tile holds p.pack query heads of qrows rows each, head-major.
      const int qrows = p.seg.qrows;
      const int i = t.qt * qrows + row % qrows;
      const int h = t.h + row / qrows;
      const bool valid = i < t.m;
      const int fq = t.cq0 + i;
      const int bq = fq / p.seg.Sq;
      const int sq = fq - bq * p.seg.Sq;
      T* orow = static_cast<T*>(p.out) + bq * p.o_sb + (int64_t)sq * p.o_ss + h * p.o_sh;
      float* lrow = p.lse + bq * p.l_sb + h * p.l_sh + sq;
      if (t.nk == 0) {
        if (valid) {
          const uint4 z = make_uint4(0, 0, 0, 0);
#pragma unroll
          for (int c = 0; c < D / 8; ++c) reinterpret_cast<uint4*>(orow)[c] = z;
          *lrow = -CUDART_INF_F;
        }
        continue;
      }
      const int delta = t.n - t.m;
      const int jmax_excl = p.seg.causal ? min(t.n, i + delta + 1) : t.n;
      const int jmin = p.seg.window > 0 ? i + delta - p.seg.window + 1 : -0x40000000;
      float m_used = -CUDART_INF_F, l = 0.f;
      for (int jj = 0; jj < t.nk; ++jj) {
        const int c0 = (t.kv_t0 + jj) * kBN;
        const int lo_c = jmin - c0, hi_c = jmax_excl - c0;
        const bool masked = __any_sync(0xffffffffu, lo_c > 0 || hi_c < kBN);
        if (!wait_bar(&s_full, kv & 1, ctl)) {
          ok = false;
          break;
        }
        ++kv;
        tc_fence_after();
        // One pass over the row: the 128 S columns into registers (four loads,
        // one wait), masked columns set to -inf, the row maximum, then
        // P = 2^(S * scale * log2 e - base) as packed T over S's first 64
        // columns and the row sum.
        float m_new = m_used, alpha = 1.f;
        auto softmax_tile = [&](auto tag) -> float {
          constexpr bool MASK = decltype(tag)::value;
          uint32_t s0[32], s1[32], s2[32], s3[32];
          tmem_ld32_async(ts, s0);
          tmem_ld32_async(ts + 32, s1);
          tmem_ld32_async(ts + 64, s2);
          tmem_ld32_async(ts + 96, s3);
          tmem_wait_ld32(s0);
          tmem_wait_ld32(s1);
          tmem_wait_ld32(s2);
          tmem_wait_ld32(s3);
          auto chunk = [&](int c) -> uint32_t(&)[32] { return c == 0 ? s0 : c == 1 ? s1 : c == 2 ? s2 : s3; };
          if constexpr (MASK) {
#pragma unroll
            for (int c = 0; c < 4; ++c) {
              uint32_t(&cur)[32] = chunk(c);
#pragma unroll
              for (int e = 0; e < 32; ++e)
                if (c * 32 + e < lo_c || c * 32 + e >= hi_c) cur[e] = 0xff800000u;  // -inf
            }
          }
          if constexpr (CAP) {
#pragma unroll
            for (int c = 0; c < 4; ++c) {
              uint32_t(&cur)[32] = chunk(c);
#pragma unroll
              for (int e = 0; e < 32; ++e) cur[e] = __float_as_uint(softcap_log2(__uint_as_float(cur[e]), cap_k1, cap_c2));
            }
          }
          float m8[8];
#pragma unroll
          for (int u = 0; u < 8; ++u) m8[u] = -CUDART_INF_F;
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            uint32_t(&cur)[32] = chunk(c);
#pragma unroll
            for (int e = 0; e < 32; e += 4) {
              const int u = ((c * 32 + e) >> 2) & 7;
              m8[u] = fmax3(m8[u], __uint_as_float(cur[e]), __uint_as_float(cur[e + 1]));
              m8[u] = fmax3(m8[u], __uint_as_float(cur[e + 2]), __uint_as_float(cur[e + 3]));
            }
          }
          const float mx =
              fmaxf(fmax3(m8[0], m8[1], m8[2]), fmax3(m8[3], m8[4], fmax3(m8[5], m8[6], m8[7]))) * mul;
          m_new = (mx > m_used + 8.f) ? mx : m_used;
          alpha = (m_new == m_used) ? 1.f : ex2_approx(m_used - m_new);
          const float base = (m_new == -CUDART_INF_F) ? 0.f : m_new;
          const float2 nbase = make_float2(-base, -base);
          float2 r4[4] = {zero2, zero2, zero2, zero2};
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            uint32_t(&cur)[32] = chunk(c);
            uint32_t pk[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              const float2 x =
                  fma2(make_float2(__uint_as_float(cur[2 * e]), __uint_as_float(cur[2 * e + 1])), mul2, nbase);
              const float2 ex = make_float2(ex2_approx(x.x), ex2_approx(x.y));
              r4[e & 3] = add2(r4[e & 3], ex);
              pk[e] = pack2<T>(ex.x, ex.y);
            }
            tmem_st16_async(ts + c * 16, pk);
          }
          tmem_wait_st();
          const float2 r2 = add2(add2(r4[0], r4[1]), add2(r4[2], r4[3]));
          return r2.x + r2.y;
        };
        const float rs = masked ? softmax_tile(MaskTag<true>{}) : softmax_tile(MaskTag<false>{});
        // O holds PV_{jj-1} already (see the header); rescale it if the maximum
        // moved, before PV_jj is released.
        if (jj > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll 1
          for (int c = 0; c < D / 32; ++c) {
            uint32_t r[32];
            tmem_ld32(to + c * 32, r);
#pragma unroll
            for (int e = 0; e < 32; ++e) r[e] = __float_as_uint(__uint_as_float(r[e]) * alpha);
            tmem_st32(to + c * 32, r);
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&p_full);
        l = l * alpha + rs;
        m_used = m_new;
      }
      if (!ok) break;
      if (!wait_bar(&pv_done, ntile & 1, ctl)) break;
      ++ntile;
      tc_fence_after();
      const float inv = l > 0.f ? 1.f / l : 0.f;
      // A warp whose 32 rows are all real rows of one head (all valid, and
      // qrows >= 32) stores them as 32 x 32 boxes: each row's 64 bytes into a
      // 64-byte-swizzled staging buffer, then one TMA store per box. Other
      // warps (a segment's last tile, heads packed 8 or 16 to a tile) store
      // their valid rows directly.
      const bool boxed = qrows >= 32 && __all_sync(0xffffffffu, valid);
      uint8_t* stg = smem + C::STG_OFF + warp * 2048;
      const int s_box = __shfl_sync(0xffffffffu, sq, 0), b_box = __shfl_sync(0xffffffffu, bq, 0);
#pragma unroll 1
      for (int c = 0; c < D / 32; ++c) {
        uint32_t r[32];
        tmem_ld32(to + c * 32, r);
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 16; ++e)
          pk[e] = pack2<T>(__uint_as_float(r[2 * e]) * inv, __uint_as_float(r[2 * e + 1]) * inv);
        if (boxed) {
          if (lane == 0) bulk_wait_group_read0();  // the buffer's previous box has been read
          __syncwarp();
#pragma unroll
          for (int q = 0; q < 4; ++q)
            *reinterpret_cast<uint4*>(stg + lane * 64 + ((q ^ ((lane >> 1) & 3)) << 4)) =
                make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_store_4d(&p.tm_o, stg, c * 32, s_box, h, b_box);
            bulk_commit_group();
          }
        } else if (valid) {
          uint4* dst = reinterpret_cast<uint4*>(orow + c * 32);
#pragma unroll
          for (int e = 0; e < 4; ++e) dst[e] = make_uint4(pk[4 * e], pk[4 * e + 1], pk[4 * e + 2], pk[4 * e + 3]);
        }
      }
      if (valid) *lrow = l > 0.f ? (m_used + __log2f(l)) * 0.69314718055994531f : -CUDART_INF_F;
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&o_free);
    }
    // Every box this warp stored has been written out before the CTA exits.
    if (lane == 0) bulk_wait_group0();
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

}  // namespace psf

// fwd_pair.cuh -- attention forward for Dqk = 192, Dv = 128 (sm_103a): one CTA
// per SM runs two 128-row query tiles of the same segment and query head side
// by side, sharing every K and V tile.
//   [nemo_automodel.components.attention.ffpa_attention, `_ffpa_varlen_fwd`,
//    `_ffpa_dense_fwd`; fa4 page, `document_causal_fa4_attention`: unequal
//    QK/V head dims such as 192/128 run without padding; causal mask at each
//    segment's bottom-right corner per the fa4 module docstring, bullet 2]
//
// A work item is a 256-row query tile of one head: half A (rows 0-127) and half
// B (rows 128-255), each with its own softmax warpgroup, S buffer and O
// accumulator, over the union of the two halves' key ranges (a half skips the
// key tiles it cannot see). Per key tile j each half runs
//   S_X(j) = Q_X K_j^T  ->  softmax  ->  O_X += P_X V_j
// and each half's MMA thread issues PV_X(j) and then S_X(j+1) as soon as that
// half's P_X(j) is written, so one half's softmax overlaps the other half's
// products, neither half's issue waits behind the other's, and both read each
// K_j / V_j from shared memory once.
//   TMEM  S_A [0, 128) | S_B [128, 256) | O_A [256, 256 + Dv) | O_B [256 + Dv, ...);
//         P_X (16-bit) is written over the first 64 columns of S_X.
//   SMEM  Q_A, Q_B (Dqk / 64 chunks each), then a ring of 16 KB chunks that
//         K_0, V_0, K_1, V_1, ... pass through in order.
//   warps 0-3 softmax of half A, 4-7 half B (thread = query row = TMEM lane),
//         8 TMA producer, 9 TMEM allocator and MMA issuer of half A, 10 MMA
//         issuer of half B.
// The commit that signals S_X(j+1) also covers PV_X(j) (a commit tracks every
// earlier MMA of the issuing thread), so the softmax may rescale O_X as soon
// as S_X(j+1) is ready. Items are taken in snake order from the heaviest-first
// list of (segment, 256-row tile) items.
#pragma once

#include <math_constants.h>

#include "fwd.cuh"

namespace psf {

template <int DQK, int DV>
struct FwdPairCfg {
  static constexpr int QCH = DQK / 64;
  static constexpr int VCH = DV / 64;
  static constexpr int Q_BYTES = QCH * kChunkBytes;
  static constexpr int NST = 8;  // ring stages (16 KB chunks)
  static constexpr int RING_OFF = 2 * Q_BYTES;
  static constexpr int SMEM_BYTES = RING_OFF + NST * kChunkBytes + 1024;
  static constexpr int T_O = 256;
  static constexpr int QROWS = 2 * kBM;  // query rows per work item
  static_assert(DQK % 64 == 0 && DV % 64 == 0 && DV <= 128, "two S buffers and two O accumulators in 512 columns");
  static_assert(SMEM_BYTES <= 232448, "shared memory budget");
};

// Key-tile index range [a, b) of one half (relative to the item's first key
// tile t0) and its row offset; empty when the half has no rows or sees no key.
struct PairHalf {
  int i0;    // segment-local first query row
  int a, b;  // key tiles [t0 + a, t0 + b) of the item's union range
};

__device__ __forceinline__ PairHalf pair_half(const FwdParams& p, const FwdTile& t, int x) {
  PairHalf h;
  h.i0 = t.qt * (2 * kBM) + x * kBM;
  h.a = h.b = 0;
  if (h.i0 >= t.m || t.nk == 0) return h;
  int lo, hi;
  kv_range_for_q_tile(t.m, t.n, h.i0, p.seg.causal, p.seg.window, lo, hi, kBM);
  if (hi <= lo) return h;
  h.a = lo / kBN - t.kv_t0;
  h.b = ceil_div(hi, kBN) - t.kv_t0;
  return h;
}

// CAP: logits softcapped (p.softcap > 0), applied to the score registers in
// place before the row maximum.
template <typename T, int DQK, int DV, bool CAP>
__global__ void __launch_bounds__(352, 1) attn_fwd_pair_kernel(const __grid_constant__ FwdParams p) {
  using C = FwdPairCfg<DQK, DV>;
  constexpr int NST = C::NST;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* ring = smem + C::RING_OFF;

  __shared__ uint64_t q_full, q_empty, kv_full[NST], kv_empty[NST];
  __shared__ uint64_t s_full[2], p_full[2], pv_done[2], o_free[2], drain;
  __shared__ uint32_t tmem_base_smem;
  __shared__ int abort_flag;

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  if (threadIdx.x == 0) {
    mbar_init(&q_full, 1);
    mbar_init(&q_empty, 2);  // both MMA issuers
    for (int i = 0; i < NST; ++i) {
      mbar_init(&kv_full[i], 1);
      mbar_init(&kv_empty[i], 2);
    }
    for (int x = 0; x < 2; ++x) {
      mbar_init(&s_full[x], 1);
      mbar_init(&p_full[x], 4);
      mbar_init(&pv_done[x], 1);
      mbar_init(&o_free[x], 4);
    }
    mbar_init(&drain, 2);
    abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 9) {
    tmem_alloc(&tmem_base_smem, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_smem;
  const Ctl ctl{p.status, p.limit_ns, &abort_flag};
  const int total = (*p.n_items) * p.Hq;
  const int G = p.Hq / p.Hkv;

  if (warp == 8) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&p.tm_q);
      tma_prefetch_desc(&p.tm_k);
      tma_prefetch_desc(&p.tm_v);
      uint32_t qcnt = 0, it = 0;
      bool ok = true;
      auto load_chunk = [&](const CUtensorMap* map, int c0, int row, int h, int b) -> bool {
        const int st = it % NST;
        if (!wait_bar(&kv_empty[st], ((it / NST) & 1) ^ 1, ctl)) return false;
        mbar_arrive_expect_tx(&kv_full[st], kChunkBytes);
        tma_load_4d(ring + st * kChunkBytes, map, &kv_full[st], c0, row, h, b);
        ++it;
        return true;
      };
      for (int wi = 0; wi * (int)gridDim.x < total && ok; ++wi) {
        const int w = snake_item(wi);
        if (w >= total) continue;
        const FwdTile t = fwd_decode(p, w);
        if (t.nk == 0) continue;
        const bool have_b = t.qt * (2 * kBM) + kBM < t.m;
        const int hk = t.h / G;
        for (int jj = 0; jj < t.nk && ok; ++jj) {
          const int fk = t.ck0 + (t.kv_t0 + jj) * kBN, bk = fk / p.seg.Sk, sk = fk - bk * p.seg.Sk;
          for (int c = 0; c < C::QCH && ok; ++c) ok = load_chunk(&p.tm_k, c * 64, sk, hk, bk);
          if (jj == 0 && ok) {
            // The item's Q tiles once the previous item's products are done
            // with theirs; its first K tile is already on its way.
            if (!wait_bar(&q_empty, (qcnt & 1) ^ 1, ctl)) {
              ok = false;
              break;
            }
            mbar_arrive_expect_tx(&q_full, (have_b ? 2 : 1) * C::Q_BYTES);
            for (int x = 0; x < (have_b ? 2 : 1); ++x) {
              const int fq = t.cq0 + t.qt * (2 * kBM) + x * kBM, bq = fq / p.seg.Sq;
              for (int c = 0; c < C::QCH; ++c)
                tma_load_4d(smem + x * C::Q_BYTES + c * kChunkBytes, &p.tm_q, &q_full, c * 64, fq - bq * p.seg.Sq,
                            t.h, bq);
            }
            ++qcnt;
          }
          for (int c = 0; c < C::VCH && ok; ++c) ok = load_chunk(&p.tm_v, c * 64, sk, hk, bk);
        }
      }
      // Wind down: no copy may still be landing in shared memory.
      for (uint32_t i = it > (uint32_t)NST ? it - NST : 0; i < it; ++i)
        wait_bar_drain(&kv_full[i % NST], (i / NST) & 1, p.limit_ns);
      if (qcnt > 0) wait_bar_drain(&q_full, (qcnt - 1) & 1, p.limit_ns);
    }
  } else if (warp == 9 || warp == 10) {
    // ------------------------------------------------------------ MMA issuers (warp 9: half A, 10: half B)
    // Each half's products come from its own thread, so one half's issue
    // never waits behind the other half's P. Both walk the ring in load order
    // (per key tile: K_j, then V_j) and each releases every chunk once (the
    // ring's empty barriers count two arrivals): by a commit when its products
    // read the chunk, else by a plain arrival once the chunk has landed (so
    // the arrival cannot count towards the slot's previous round).
    if (lane == 0) {
      const int x = warp - 9;
      constexpr uint32_t id_qk = idesc_f32acc<T>(128, 128, 0, 0);
      constexpr uint32_t id_pv = idesc_f32acc<T>(128, DV, 0, 1);
      constexpr uint32_t id_pv64 = idesc_f32acc<T>(128, 64, 0, 1);
      const uint32_t ring_a = smem_u32(ring), qx = smem_u32(smem) + x * C::Q_BYTES;
      const uint32_t ts = tmem + x * 128, to = tmem + C::T_O + x * DV;
      uint32_t qcnt = 0, it = 0, nkv = 0, ntile = 0;
      bool ok = true;
      // Wait for the next n chunks of the ring (in load order); returns the first one's index.
      auto take = [&](int n) -> uint32_t {
        const uint32_t first = it;
        for (int c = 0; c < n && ok; ++c, ++it)
          if (!wait_bar(&kv_full[it % NST], (it / NST) & 1, ctl)) ok = false;
        tc_fence_after();
        return first;
      };
      auto release = [&](uint32_t first, int n, bool used) {
        for (int c = 0; c < n; ++c) {
          if (used)
            mma_commit(&kv_empty[(first + c) % NST]);
          else
            mbar_arrive(&kv_empty[(first + c) % NST]);
        }
      };
      for (int wi = 0; wi * (int)gridDim.x < total && ok; ++wi) {
        const int w = snake_item(wi);
        if (w >= total) continue;
        const FwdTile t = fwd_decode(p, w);
        if (t.nk == 0) continue;
        const PairHalf hx = pair_half(p, t, x);
        if (!wait_bar(&q_full, qcnt & 1, ctl)) break;
        tc_fence_after();
        bool first_pv = true;
        for (int jj = 0; jj < t.nk && ok; ++jj) {
          const bool act = jj >= hx.a && jj < hx.b;
          // S_X(j) = Q_X K_j^T; its commit also covers PV_X(j-1), issued just before.
          const uint32_t k_first = take(C::QCH);
          if (!ok) break;
          if (act) {
#pragma unroll
            for (int c = 0; c < C::QCH; ++c) {
              const uint32_t k_addr = ring_a + ((k_first + c) % NST) * kChunkBytes;
#pragma unroll
              for (int kk = 0; kk < 4; ++kk)
                mma_ss(ts, sdesc_sw128(qx + c * kChunkBytes + kk * 32, 16, 1024),
                       sdesc_sw128(k_addr + kk * 32, 16, 1024), id_qk, (c | kk) != 0);
            }
            mma_commit(&s_full[x]);
          }
          release(k_first, C::QCH, act);
          // O_X (+)= P_X V_j once the softmax has written P_X (and, on the
          // half's first key tile, once the previous item's epilogue has read O_X).
          const uint32_t v_first = take(C::VCH);
          if (!ok) break;
          if (act) {
            if (!wait_bar(&p_full[x], nkv & 1, ctl)) {
              ok = false;
              break;
            }
            ++nkv;
            if (first_pv && ntile > 0 && !wait_bar(&o_free[x], (ntile - 1) & 1, ctl)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t vs = v_first % NST;
            if (vs + C::VCH <= (uint32_t)NST) {
              // V's chunks sit in consecutive slots: one N = Dv chain, the
              // B operand's 64-column chunks reached through the leading-byte offset.
              const uint32_t v_addr = ring_a + vs * kChunkBytes;
#pragma unroll
              for (int kk = 0; kk < 8; ++kk)
                mma_ts(to, ts + kk * 8, sdesc_sw128(v_addr + kk * 2048, kChunkBytes, 1024), id_pv,
                       !(first_pv && kk == 0));
            } else {
              // V wraps around the ring: one N = 64 chain per chunk.
#pragma unroll
              for (int c = 0; c < C::VCH; ++c) {
                const uint32_t v_addr = ring_a + ((v_first + c) % NST) * kChunkBytes;
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                  mma_ts(to + c * 64, ts + kk * 8, sdesc_sw128(v_addr + kk * 2048, kChunkBytes, 1024), id_pv64,
                         !(first_pv && kk == 0));
              }
            }
            first_pv = false;
          }
          release(v_first, C::VCH, act);
        }
        if (!ok) break;
        mma_commit(&q_empty);
        if (hx.b > hx.a) {
          mma_commit(&pv_done[x]);
          ++ntile;
        }
        ++qcnt;
      }
      // Wind down: wait until every MMA either thread issued has finished.
      mma_commit(&drain);
      wait_bar_drain(&drain, 0, p.limit_ns);
    }
  } else {
    // ------------------------------------------------------------ softmax warpgroups (warps 0-3: A, 4-7: B)
    const int x = warp >> 2;
    const int row = threadIdx.x & 127;
    const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
    const uint32_t ts = tmem + lane_base + x * 128, to = tmem + lane_base + C::T_O + x * DV;
    const float sl2 = p.scale_log2;
    const float2 zero2 = make_float2(0.f, 0.f);
    const float mul = CAP ? 1.f : sl2;  // with CAP the score registers hold capped logits in log2 units
    const float2 mul2 = make_float2(mul, mul);
    const float cap_k1 = CAP ? 2.f * sl2 / p.softcap : 0.f, cap_c2 = CAP ? p.softcap * 1.4426950408889634f : 0.f;
    uint32_t nkv = 0, ntile = 0;
    bool ok = true;
    for (int wi = 0; wi * (int)gridDim.x < total && ok; ++wi) {
      const int w = snake_item(wi);
      if (w >= total) continue;
      const FwdTile t = fwd_decode(p, w);
      const PairHalf hx = pair_half(p, t, x);
      const int i = hx.i0 + row;
      if (hx.i0 >= t.m) continue;  // this half holds no row of the segment
      const bool valid = i < t.m;
      const int fq = t.cq0 + i;
      const int bq = fq / p.seg.Sq;
      const int sq = fq - bq * p.seg.Sq;
      T* orow = static_cast<T*>(p.out) + bq * p.o_sb + (int64_t)sq * p.o_ss + t.h * p.o_sh;
      float* lrow = p.lse + bq * p.l_sb + t.h * p.l_sh + sq;
      if (hx.b <= hx.a) {
        // No key visible to any row of this half: out = 0, lse = -inf.
        if (valid) {
          const uint4 z = make_uint4(0, 0, 0, 0);
#pragma unroll
          for (int c = 0; c < DV / 8; ++c) reinterpret_cast<uint4*>(orow)[c] = z;
          *lrow = -CUDART_INF_F;
        }
        continue;
      }
      const int delta = t.n - t.m;
      const int jmax_excl = p.seg.causal ? min(t.n, i + delta + 1) : t.n;
      const int jmin = p.seg.window > 0 ? i + delta - p.seg.window + 1 : -0x40000000;
      float m_used = -CUDART_INF_F, l = 0.f;
      for (int jj = hx.a; jj < hx.b; ++jj) {
        const int c0 = (t.kv_t0 + jj) * kBN;
        const int lo_c = jmin - c0, hi_c = jmax_excl - c0;
        const bool masked = __any_sync(0xffffffffu, lo_c > 0 || hi_c < kBN);
        if (!wait_bar(&s_full[x], nkv & 1, ctl)) {
          ok = false;
          break;
        }
        ++nkv;
        tc_fence_after();
        // One pass over the row: the 128 S columns into registers, masked
        // columns set to -inf, the row maximum, then P = 2^(S * scale * log2 e
        // - base) as packed 16-bit values over S's first 64 columns, and the row sum.
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
          const float mx = fmaxf(fmax3(m8[0], m8[1], m8[2]), fmax3(m8[3], m8[4], fmax3(m8[5], m8[6], m8[7]))) * mul;
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
              const float2 xv =
                  fma2(make_float2(__uint_as_float(cur[2 * e]), __uint_as_float(cur[2 * e + 1])), mul2, nbase);
              const float2 ex = make_float2(ex2_approx(xv.x), ex2_approx(xv.y));
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
        // O_X holds PV_X of the earlier key tiles already (see the header);
        // rescale it if the maximum moved, before this P is released.
        if (jj > hx.a && __any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll 1
          for (int c = 0; c < DV / 32; ++c) {
            uint32_t r[32];
            tmem_ld32(to + c * 32, r);
#pragma unroll
            for (int e = 0; e < 32; ++e) r[e] = __float_as_uint(__uint_as_float(r[e]) * alpha);
            tmem_st32(to + c * 32, r);
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&p_full[x]);
        l = l * alpha + rs;
        m_used = m_new;
      }
      if (!ok) break;
      if (!wait_bar(&pv_done[x], ntile & 1, ctl)) break;
      ++ntile;
      tc_fence_after();
      const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll 1
      for (int c = 0; c < DV / 32; ++c) {
        uint32_t r[32];
        tmem_ld32(to + c * 32, r);
        if (valid) {
          uint32_t pk[16];
#pragma unroll
          for (int e = 0; e < 16; ++e)
            pk[e] = pack2<T>(__uint_as_float(r[2 * e]) * inv, __uint_as_float(r[2 * e + 1]) * inv);
          uint4* dst = reinterpret_cast<uint4*>(orow + c * 32);
#pragma unroll
          for (int e = 0; e < 4; ++e) dst[e] = make_uint4(pk[4 * e], pk[4 * e + 1], pk[4 * e + 2], pk[4 * e + 3]);
        }
      }
      if (valid) *lrow = l > 0.f ? (m_used + __log2f(l)) * 0.69314718055994531f : -CUDART_INF_F;
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&o_free[x]);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace psf

// bwd192.cuh -- attention backward for Dqk = 192, Dv = 128 (sm_103a): one
// 192-column TMEM region reused for S, dP and dQ in turn.
//   [nemo_automodel.components.attention.ffpa_attention, `_ffpa_varlen_bwd`,
//    `_ffpa_dense_bwd`; the per-step arithmetic is the one bwd.cuh states]
//
// Warps: 0 TMA producer, 1 MMA issuer, 2 TMEM allocator, 4-7 and 12-15
// compute (P, dS, and the dK/dV epilogue), 8-11 dQ read-out.
#pragma once

#include <math_constants.h>

#include <type_traits>

#include "bwd.cuh"

namespace psf {

// Shared-memory and TMEM plan of attn_bwd_kernel (Dqk = 192, Dv = 128).
template <int DQK, int DV>
struct BwdCfg {
  static constexpr int KCH = DQK / 64;
  static constexpr int VCH = DV / 64;
  static constexpr int K_OFF = 0;
  static constexpr int V_OFF = K_OFF + KCH * kChunkBytes;
  static constexpr int Q_OFF = V_OFF + VCH * kChunkBytes;
  static constexpr int DO_OFF = Q_OFF + KCH * kChunkBytes;
  // dS^T (bf16, two 64-query chunks); between steps each compute warp stages
  // its share of the dQ read-out in its own 32 rows of this buffer.
  static constexpr int DS_OFF = DO_OFF + VCH * kChunkBytes;
  static constexpr int STG_OFF = DS_OFF + 2 * kChunkBytes;  // dQ staging of the read-out warps (4 x 4 KB)
  static constexpr int ROWV_OFF = STG_OFF + 4 * 4096;       // -lse log2 e and -Delta, 8 warps x 64 each
  static constexpr int SMEM_BYTES = ROWV_OFF + 2 * 8 * 64 * 4 + 1024;
  // TMEM columns: dV [0, 128) | dK [128, 320) | R [320, 512). R holds S^T
  // (first 128 columns), then dP^T (same columns), then dQ (all 192); P^T
  // (packed 16-bit) sits in its last 64 columns between S^T and dQ.
  static constexpr int T_DV = 0;
  static constexpr int T_DK = 128;
  static constexpr int T_R = 320;
  static constexpr int T_P = T_R + 128;
  static_assert(DQK == 192 && DV == 128, "single-region plan is laid out for (192, 128)");
  static_assert(SMEM_BYTES <= 232448, "shared memory budget");
};

// CAP: logits softcapped (p.softcap > 0); dS carries the cap's 1 - tanh^2.
//
// Per step (one 128-query tile of one query head against the resident key
// tile), thread r of a compute warpgroup owning key row r (TMEM lane r):
//   S^T  = K Q^T -> R[0, 128)          P^T = exp2(S^T scale log2 e - lse log2 e)
//   P^T (16-bit, packed) -> R[128, 192) (the TMEM operand of dV += P^T dO)
//   dP^T = V dO^T -> R[0, 128)          dS^T = P^T (dP^T - Delta) -> shared memory
//   dK  += dS^T Q,  dQ = dS K -> R[0, 192)
// Two compute warpgroups split the 128 query columns of every step (warps
// 4-7 columns 0-63, warps 12-15 columns 64-127); the dQ read-out is split over
// twelve warps (warps 8-11 four 32-column chunks, each compute warpgroup one),
// which release R as soon as their chunks are in registers so that the next
// step's S^T can start while the chunks go out by TMA reduce-add. Q arrives
// and is released in 64-column chunks, so the next step's Q loads while this
// step's dK and dQ products run. Warps: 0 TMA producer, 1 MMA issuer, 2 TMEM
// allocator.
template <typename T, int DQK, int DV, bool CAP>
__global__ void __launch_bounds__(512, 1) attn_bwd_kernel(const __grid_constant__ BwdParams p) {
  using C = BwdCfg<DQK, DV>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  float* l2_s = reinterpret_cast<float*>(smem + C::ROWV_OFF);  // [8 compute warps][64]: lse * log2 e (+inf: no mass)
  float* dl_s = l2_s + 8 * 64;                                   // [8 compute warps][64]: Delta

  // Q moves in its three 64-column chunks, each with its own barriers, so the
  // next step's chunk c loads as soon as this step's dK products are done with it.
  __shared__ uint64_t kv_full, kv_empty, q_full[C::KCH], q_empty[C::KCH], do_full, do_empty, s_full, p_full,
      dp_full, ds_full, dq_full, dq_free, acc_done, acc_free, drain;
  __shared__ uint32_t tmem_base_smem;
  __shared__ int abort_flag;

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  if (threadIdx.x == 0) {
    mbar_init(&kv_full, 1);
    mbar_init(&kv_empty, 1);
    for (int c = 0; c < C::KCH; ++c) {
      mbar_init(&q_full[c], 1);
      mbar_init(&q_empty[c], 1);
    }
    mbar_init(&do_full, 1);
    mbar_init(&do_empty, 1);
    mbar_init(&s_full, 1);
    mbar_init(&p_full, 8);
    mbar_init(&dp_full, 1);
    mbar_init(&ds_full, 8);
    mbar_init(&dq_full, 1);
    mbar_init(&dq_free, 12);
    mbar_init(&acc_done, 1);
    mbar_init(&acc_free, 8);
    mbar_init(&drain, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 2) {
    tmem_alloc(&tmem_base_smem, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_smem;
  const Ctl ctl{p.status, p.limit_ns, &abort_flag};
  const int total = (*p.n_items) * p.Hkv;
  const int G = p.Hq / p.Hkv;
  const uint32_t sbase = smem_u32(smem);

  // One 32 x 32 fp32 chunk of dQ (query rows = TMEM lanes of this warp) into
  // the warp's staging box and on to the accumulator by TMA reduce-add.
  auto reduce_box = [&](uint8_t* box, const uint32_t(&v)[32], int dcol, int sq, int h, int bq) {
#pragma unroll
    for (int u = 0; u < 8; ++u)
      *reinterpret_cast<uint4*>(box + sw128_offset(lane, u)) = make_uint4(v[4 * u], v[4 * u + 1], v[4 * u + 2], v[4 * u + 3]);
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
      tma_reduce_add_4d(&p.tm_dq, box, dcol, sq, h, bq);
      bulk_commit_group();
    }
  };
  // The read-out of one step: this warp's N dQ chunks [c0, c0 + N) (32
  // columns each) into registers, R released, then the chunks staged through
  // `box` in turn (each staging waits until the box's previous reduce has read it).
  auto dq_readout = [&](auto nch, const BwdItem& t, int k, uint32_t gstep, int wq, int c0, uint8_t* box) -> bool {
    constexpr int N = decltype(nch)::value;
    if (!wait_bar(&dq_full, gstep & 1, ctl)) return false;
    tc_fence_after();
    uint32_t a[N][32];
    const uint32_t rq = tmem + ((uint32_t)(32 * wq) << 16) + C::T_R + c0 * 32;
    if constexpr (N == 1) {
      tmem_ld32(rq, a[0]);
    } else {
#pragma unroll
      for (int i = 0; i < N; i += 2) tmem_ld32x2(rq + i * 32, rq + i * 32 + 32, a[i], a[i + 1]);
    }
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(&dq_free);
    const int h = t.hk * G + k / t.nqt, qt = t.qt0 + k % t.nqt;
    const int fq = t.cq0 + qt * kBM + 32 * wq, bq = fq / p.seg.Sq, sq = fq - bq * p.seg.Sq;
#pragma unroll
    for (int i = 0; i < N; ++i) {
      if (lane == 0) bulk_wait_group_read0();
      __syncwarp();
      reduce_box(box, a[i], (c0 + i) * 32, sq, h, bq);
    }
    return true;
  };

  // Register budgets per warpgroup (launch: 128 per thread, 512 threads):
  // warps 0-3 96, compute warpgroups 128, dQ read-out warps 160, which hold
  // four 32-column chunks at once: 96 + 128 + 160 + 128 = 4 x 128.
  if (warp < 4) {
    setmaxnreg_dec<96>();
  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&p.tm_q);
      tma_prefetch_desc(&p.tm_k);
      tma_prefetch_desc(&p.tm_v);
      tma_prefetch_desc(&p.tm_do);
      uint32_t nz = 0, gstep = 0;
      bool ok = true;
      for (int wi = 0; wi * (int)gridDim.x < total && ok; ++wi) {
        const int w = snake_item(wi);
        if (w >= total) continue;
        const BwdItem t = bwd_decode(p, w);
        if (t.k1 == t.k0) continue;
        if (!wait_bar(&kv_empty, (nz & 1) ^ 1, ctl)) break;
        mbar_arrive_expect_tx(&kv_full, (C::KCH + C::VCH) * kChunkBytes);
        const int fk = t.ck0 + t.kt * kBN, bk = fk / p.seg.Sk, sk = fk - bk * p.seg.Sk;
        for (int c = 0; c < C::KCH; ++c)
          tma_load_4d(smem + C::K_OFF + c * kChunkBytes, &p.tm_k, &kv_full, c * 64, sk, t.hk, bk);
        for (int c = 0; c < C::VCH; ++c)
          tma_load_4d(smem + C::V_OFF + c * kChunkBytes, &p.tm_v, &kv_full, c * 64, sk, t.hk, bk);
        ++nz;
        for (int k = t.k0; k < t.k1; ++k, ++gstep) {
          const int h = t.hk * G + k / t.nqt, qt = t.qt0 + k % t.nqt;
          const int fq = t.cq0 + qt * kBM, bq = fq / p.seg.Sq, sq = fq - bq * p.seg.Sq;
          // dO(g) once dV(g-1) has read dO(g-1), then Q(g) once dK(g-1) has read Q(g-1).
          if (!wait_bar(&do_empty, (gstep & 1) ^ 1, ctl)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&do_full, C::VCH * kChunkBytes);
          for (int c = 0; c < C::VCH; ++c)
            tma_load_4d(smem + C::DO_OFF + c * kChunkBytes, &p.tm_do, &do_full, c * 64, sq, h, bq);
          for (int c = 0; c < C::KCH && ok; ++c) {
            if (!wait_bar(&q_empty[c], (gstep & 1) ^ 1, ctl)) {
              ok = false;
              break;
            }
            mbar_arrive_expect_tx(&q_full[c], kChunkBytes);
            tma_load_4d(smem + C::Q_OFF + c * kChunkBytes, &p.tm_q, &q_full[c], c * 64, sq, h, bq);
          }
          if (!ok) break;
        }
      }
      if (nz > 0) wait_bar_drain(&kv_full, (nz - 1) & 1, p.limit_ns);
      if (gstep > 0) {
        wait_bar_drain(&do_full, (gstep - 1) & 1, p.limit_ns);
        for (int c = 0; c < C::KCH; ++c) wait_bar_drain(&q_full[c], (gstep - 1) & 1, p.limit_ns);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t id_sq = idesc_f32acc<T>(128, 128, 0, 0);  // S^T = K Q^T, dP^T = V dO^T
      constexpr uint32_t id_dv = idesc_f32acc<T>(128, DV, 0, 1);   // dV += P^T (TMEM) dO
      constexpr uint32_t id_dk = idesc_f32acc<T>(128, DQK, 0, 1);  // dK += dS^T Q
      constexpr uint32_t id_dq = idesc_f32acc<T>(128, DQK, 1, 1);  // dQ  = dS K
      const uint32_t k_a = sbase + C::K_OFF, v_a = sbase + C::V_OFF, q_a = sbase + C::Q_OFF;
      const uint32_t do_a = sbase + C::DO_OFF, ds_a = sbase + C::DS_OFF;
      const uint32_t rr = tmem + C::T_R, rp = tmem + C::T_P;
      uint32_t nz = 0, gstep = 0;
      bool ok = true;
      for (int wi = 0; wi * (int)gridDim.x < total && ok; ++wi) {
        const int w = snake_item(wi);
        if (w >= total) continue;
        const BwdItem t = bwd_decode(p, w);
        if (t.k1 == t.k0) continue;
        if (!wait_bar(&kv_full, nz & 1, ctl)) break;
        if (nz > 0 && !wait_bar(&acc_free, (nz - 1) & 1, ctl)) break;
        tc_fence_after();
        for (int k = t.k0; k < t.k1 && ok; ++k, ++gstep) {
          // S^T(g) once the previous dQ has left R, chunk by chunk of Q(g) as they land.
          if (gstep > 0 && !wait_bar(&dq_free, (gstep - 1) & 1, ctl)) {
            ok = false;
            break;
          }
          for (int c = 0; c < C::KCH && ok; ++c) {
            if (!wait_bar(&q_full[c], gstep & 1, ctl)) {
              ok = false;
              break;
            }
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              mma_ss(rr, sdesc_sw128(k_a + c * kChunkBytes + kk * 32, 16, 1024),
                     sdesc_sw128(q_a + c * kChunkBytes + kk * 32, 16, 1024), id_sq, (c | kk) != 0);
          }
          if (!ok) break;
          mma_commit(&s_full);
          // dP^T over S^T once the first pass has read it and written P^T;
          // then dV from the packed P^T.
          if (!wait_bar(&do_full, gstep & 1, ctl) || !wait_bar(&p_full, gstep & 1, ctl)) {
            ok = false;
            break;
          }
          tc_fence_after();
          for (int c = 0; c < C::VCH; ++c) {
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              mma_ss(rr, sdesc_sw128(v_a + c * kChunkBytes + kk * 32, 16, 1024),
                     sdesc_sw128(do_a + c * kChunkBytes + kk * 32, 16, 1024), id_sq, (c | kk) != 0);
          }
          mma_commit(&dp_full);
          const uint32_t first = (k == t.k0) ? 1u : 0u;
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            mma_ts(tmem + C::T_DV, rp + kk * 8, sdesc_sw128(do_a + kk * 2048, kChunkBytes, 1024), id_dv,
                   !(first && kk == 0));
          mma_commit(&do_empty);
          // dK, then dQ over all of R, once dS^T is in shared memory.
          if (!wait_bar(&ds_full, gstep & 1, ctl)) {
            ok = false;
            break;
          }
          tc_fence_after();
          // dK over all three 64-column chunks of Q at once (N = 192 products
          // take about the time of N = 64 ones), then Q(g) is released.
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            mma_ss(tmem + C::T_DK, sdesc_sw128(ds_a + (kk >> 2) * kChunkBytes + (kk & 3) * 32, 16, 1024),
                   sdesc_sw128(q_a + kk * 2048, kChunkBytes, 1024), id_dk, !(first && kk == 0));
          for (int c = 0; c < C::KCH; ++c) mma_commit(&q_empty[c]);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            mma_ss(rr, sdesc_sw128(ds_a + kk * 2048, kChunkBytes, 1024), sdesc_sw128(k_a + kk * 2048, kChunkBytes, 1024),
                   id_dq, kk > 0);
          mma_commit(&dq_full);
        }
        if (!ok) break;
        mma_commit(&acc_done);
        mma_commit(&kv_empty);
        ++nz;
      }
      mma_commit(&drain);
      wait_bar_drain(&drain, 0, p.limit_ns);
    }
  }
  } else if (warp >= 4 && (warp < 8 || warp >= 12)) {
    // ------------------------------------------------------------ compute warpgroups
    const int half = warp >= 12 ? 1 : 0;
    const int wq = warp & 3;
    const int cb = half * 64;         // first query column of this warpgroup
    const int r = 32 * wq + lane;     // key row within the tile
    const uint32_t lane_base = (uint32_t)(32 * wq) << 16;
    float* my_l2 = l2_s + (half * 4 + wq) * 64;
    float* my_dl = dl_s + (half * 4 + wq) * 64;
    uint8_t* ds_s = smem + C::DS_OFF + half * kChunkBytes;
    uint8_t* box = ds_s + wq * 4096;  // this warp's own 32 rows of dS^T
    const uint32_t rr = tmem + lane_base + C::T_R + cb, rp = tmem + lane_base + C::T_P + half * 32;
    const float sl2 = p.scale_log2;
    const float cap_c2 = CAP ? p.softcap * 1.4426950408889634f : 0.f;
    const float cap_k1 = CAP ? 2.f * sl2 / p.softcap : 0.f, cap_ic2 = CAP ? 1.f / cap_c2 : 0.f;
    uint32_t nz = 0, gstep = 0;
    bool ok = true;
    for (int wi = 0; wi * (int)gridDim.x < total && ok; ++wi) {
      const int w = snake_item(wi);
      if (w >= total) continue;
      const BwdItem t = bwd_decode(p, w);
      const int j = t.kt * kBN + r;  // segment-local key index
      const bool valid = j < t.n;
      const int fk = t.ck0 + j, bk = fk / p.seg.Sk, sk = fk - bk * p.seg.Sk;
      T* dk_row = static_cast<T*>(p.dk) + bk * p.k_sb + (int64_t)sk * p.k_ss + t.hk * p.k_sh;
      T* dv_row = static_cast<T*>(p.dv) + bk * p.v_sb + (int64_t)sk * p.v_ss + t.hk * p.v_sh;
      if (t.k1 == t.k0) {
        // No query sees this key tile: dV (warps 4-7) and dK (warps 12-15) are zero.
        if (valid) {
          if (half == 0)
            for (int c = 0; c < DV / 8; ++c) reinterpret_cast<uint4*>(dv_row)[c] = make_uint4(0, 0, 0, 0);
          else
            for (int c = 0; c < DQK / 8; ++c) reinterpret_cast<uint4*>(dk_row)[c] = make_uint4(0, 0, 0, 0);
        }
        continue;
      }
      const int delta = t.n - t.m;
      // lse and Delta of 2 of this warpgroup's query columns per lane, loaded
      // one step ahead and left in flight (-inf / 0 outside the segment).
      auto fetch_rows = [&](int k, float (&lv)[2], float (&dv)[2]) {
        const int h = t.hk * G + k / t.nqt, i0 = (t.qt0 + k % t.nqt) * kBM;
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int qc = cb + lane * 2 + e;
          const int f = t.cq0 + i0 + qc;
          const bool in = i0 + qc < t.m && f < p.q_rows;
          const int fs = in ? f : 0;
          const int bq = fs / p.seg.Sq, sq = fs - bq * p.seg.Sq;
          lv[e] = -CUDART_INF_F;
          dv[e] = 0.f;
          ldg_pred_f32(lv[e], p.lse + bq * p.l_sb + h * p.l_sh + sq, in);
          ldg_pred_f32(dv[e], p.delta + (int64_t)h * p.q_rows + fs, in);
        }
      };
      float rlv[2], rdv[2];
      fetch_rows(t.k0, rlv, rdv);
      for (int k = t.k0; k < t.k1; ++k, ++gstep) {
        const int i0 = (t.qt0 + k % t.nqt) * kBM;
        // Visible query columns [q_lo, q_hi) of this key row in the tile.
        int q_lo = p.seg.causal ? j - delta - i0 : -0x40000000;
        int q_hi = t.m - i0;
        if (p.seg.window > 0) q_hi = min(q_hi, j - delta + p.seg.window - i0);
        if (!valid) q_lo = q_hi = 0;
        const bool masked = __any_sync(0xffffffffu, q_lo > cb || q_hi < cb + 64);
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          my_l2[lane * 2 + e] = rlv[e] == -CUDART_INF_F ? CUDART_INF_F : rlv[e] * 1.4426950408889634f;
          my_dl[lane * 2 + e] = rdv[e];
        }
        __syncwarp();
        if (k + 1 < t.k1) fetch_rows(k + 1, rlv, rdv);
        if (!wait_bar(&s_full, gstep & 1, ctl)) {
          ok = false;
          break;
        }
        tc_fence_after();
        // Pass 1: P^T of this warpgroup's 64 columns -> R[128 + 32 half, +32)
        // packed; with CAP the factor P (1 - tanh^2) stays in registers.
        [[maybe_unused]] uint32_t pf_keep[2][16];  // CAP only
        {
          uint32_t sa[32], sb[32];
          tmem_ld32_async(rr, sa);
          tmem_ld32_async(rr + 32, sb);
          tmem_wait_ld32(sa);
          tmem_wait_ld32(sb);
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            uint32_t(&cur)[32] = c ? sb : sa;
            uint32_t pk[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              float pr[2], pf[2];
#pragma unroll
              for (int u = 0; u < 2; ++u) {
                const int ql = c * 32 + 2 * e + u;  // column within this warpgroup's 64
                const float sc = __uint_as_float(cur[2 * e + u]);
                float pe, fac = 1.f;
                if constexpr (CAP) {
                  const float y = softcap_log2(sc, cap_k1, cap_c2);
                  const float tt = y * cap_ic2;
                  fac = fmaf(-tt, tt, 1.f);
                  pe = ex2_approx(y - my_l2[ql]);
                } else {
                  pe = ex2_approx(fmaf(sc, sl2, -my_l2[ql]));
                }
                if (masked && (cb + ql < q_lo || cb + ql >= q_hi)) pe = 0.f;
                pr[u] = pe;
                pf[u] = pe * fac;
              }
              pk[e] = pack2<T>(pr[0], pr[1]);
              if constexpr (CAP) pf_keep[c][e] = pack2<T>(pf[0], pf[1]);
            }
            tmem_st16_async(rp + c * 16, pk);
          }
          tmem_wait_st();
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&p_full);
        // Pass 2: dS^T = P^T (dP^T - Delta) into this warpgroup's 64-column
        // chunk of the dS^T buffer, once dP^T is ready and this warp's
        // previous dQ boxes have been read out of its rows.
        if (lane == 0) bulk_wait_group_read0();
        __syncwarp();
        if (!wait_bar(&dp_full, gstep & 1, ctl)) {
          ok = false;
          break;
        }
        tc_fence_after();
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          uint32_t dpv[32];
          uint32_t pw[16];
          tmem_ld32_async(rr + c * 32, dpv);
          if constexpr (CAP) {
            tmem_wait_ld32(dpv);
#pragma unroll
            for (int e = 0; e < 16; ++e) pw[e] = pf_keep[c][e];
          } else {
            tmem_ld16_async(rp + c * 16, pw);
            tmem_wait_ld32_16(dpv, pw);
          }
          uint32_t dk2[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const int ql = c * 32 + 2 * e;
            const float2 pf = unpack2<T>(pw[e]);
            dk2[e] = pack2<T>(pf.x * (__uint_as_float(dpv[2 * e]) - my_dl[ql]),
                              pf.y * (__uint_as_float(dpv[2 * e + 1]) - my_dl[ql + 1]));
          }
#pragma unroll
          for (int u = 0; u < 4; ++u)
            *reinterpret_cast<uint4*>(ds_s + sw128_offset(r, c * 4 + u)) =
                make_uint4(dk2[4 * u], dk2[4 * u + 1], dk2[4 * u + 2], dk2[4 * u + 3]);
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&ds_full);
        // This warp's share of the dQ read-out: chunk 0 (warps 4-7) or 5
        // (warps 12-15), staged in its own rows of the dS^T buffer, which the
        // dK and dQ products have finished reading when dQ is ready.
        if (!dq_readout(std::integral_constant<int, 1>{}, t, k, gstep, wq, half ? 5 : 0, box)) {
          ok = false;
          break;
        }
      }
      if (!ok) break;
      // dV (warps 4-7) or dK (warps 12-15, scale applied) of this key tile.
      if (!wait_bar(&acc_done, nz & 1, ctl)) break;
      tc_fence_after();
      const int nch = half ? DQK / 32 : DV / 32;
      const float sc = half ? p.scale : 1.f;
      T* row = half ? dk_row : dv_row;
#pragma unroll 1
      for (int c = 0; c < nch; ++c) {
        uint32_t a[32];
        tmem_ld32(tmem + lane_base + (half ? C::T_DK : C::T_DV) + c * 32, a);
        if (valid) {
          uint4* dst = reinterpret_cast<uint4*>(row + c * 32);
#pragma unroll
          for (int u = 0; u < 4; ++u)
            dst[u] = make_uint4(pack2<T>(__uint_as_float(a[8 * u]) * sc, __uint_as_float(a[8 * u + 1]) * sc),
                                pack2<T>(__uint_as_float(a[8 * u + 2]) * sc, __uint_as_float(a[8 * u + 3]) * sc),
                                pack2<T>(__uint_as_float(a[8 * u + 4]) * sc, __uint_as_float(a[8 * u + 5]) * sc),
                                pack2<T>(__uint_as_float(a[8 * u + 6]) * sc, __uint_as_float(a[8 * u + 7]) * sc));
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_free);
      ++nz;
    }
    if (lane == 0) bulk_wait_group0();
  } else {
    // ------------------------------------------------------------ dQ read-out, chunks 1-4
    setmaxnreg_inc<160>();
    const int wq = warp - 8;
    uint8_t* box = smem + C::STG_OFF + wq * 4096;
    uint32_t gstep = 0;
    bool ok = true;
    for (int wi = 0; wi * (int)gridDim.x < total && ok; ++wi) {
      const int w = snake_item(wi);
      if (w >= total) continue;
      const BwdItem t = bwd_decode(p, w);
      for (int k = t.k0; k < t.k1; ++k, ++gstep) {
        if (!dq_readout(std::integral_constant<int, 4>{}, t, k, gstep, wq, 1, box)) {
          ok = false;
          break;
        }
      }
    }
    if (lane == 0) bulk_wait_group0();
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace psf

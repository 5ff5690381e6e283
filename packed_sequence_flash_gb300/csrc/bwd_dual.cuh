// bwd_dual.cuh -- attention backward for Dqk, Dv <= 128 (sm_103a).
//   [nemo_automodel.components.attention.ffpa_attention, `_ffpa_varlen_bwd`,
//    `_ffpa_dense_bwd`: gradients from the caller-supplied out/lse, dK/dV
//    reduced to the KV heads]
//
// Same arithmetic as bwd.cuh, laid out for head dims up to 128 so that every
// operand stream overlaps the tensor core:
//   TMEM   dV [0, Dv) | dK [Dv, Dv + Dqk) | region A [256, 384) | region B [384, 512)
//          A holds S^T, then P^T (bf16; query columns 0-63 at A[0, 32),
//          64-127 at A[64, 96)) as the TMEM operand of dV += P^T dO; B holds
//          dP^T (two N = 64 halves), then dQ = dS K.
//   Order  per step g the MMA warp issues dP(g) -> B, dV(g) once P^T is
//          written, then, as soon as dS^T(g) is in shared memory, S(g+1) -> A
//          ahead of dQ(g) -> B and dK(g), so the next step's element-wise pass
//          runs while the tensor core finishes this one, and the dQ read-out
//          (which frees B for dP(g+1)) overlaps the dK MMAs.
//   SMEM   K, V resident per key tile; Q double-buffered; dO single-buffered
//          but released right after dV, its last reader; dS^T (bf16, 128-byte
//          swizzled) read K-major by dK and M-major by dQ; a 16 KB area stages
//          the dQ read-out's fp32 boxes; the dK/dV epilogue stages in the dS^T
//          buffer, which the compute warps own between steps.
//   Steps  the compute warps make two passes: P^T (stored to A as packed
//          bf16), then dS^T from dP^T and the stored P^T. TMEM reads run one
//          32-column chunk ahead of the arithmetic; S(g+1) is issued only after
//          dS^T(g), so the second pass can still read P^T(g) from A.
//   Work   a unit is a key tile of one KV head and a range of its (query head,
//          query tile) steps; the scheduler cuts heavy key tiles into several
//          ranges so that the SMs finish together. dV and dK accumulate in
//          TMEM across the range (all query heads of the GQA group when the
//          range covers them); a whole key tile writes them to the outputs
//          from TMEM, a cut tile's sub-ranges store fp32 partial sums to
//          slots of their own, which the convert kernel adds up.
//   Warps  0 TMA producer, 1 MMA issuer, 2 TMEM allocator, 4-7 compute
//          (thread = key row: P, dS, then the dK/dV epilogue), 8-11 dQ read-out.
//   Work   a CTA starts on unit blockIdx.x of the heaviest-first list, then takes
//          the next untaken unit from a global counter; the producer decodes
//          each unit while the previous one's first step loads and passes its
//          index and decoded unit to the other warps through a two-entry ring
//          in shared memory (-1 = no more work).
// The compute warps load the next step's lse and Delta one step ahead and
// leave the loads in flight until the step begins.
#pragma once

#include <math_constants.h>

#include "bwd.cuh"

namespace psf {

template <int DQK, int DV>
struct BwdDualCfg {
  static constexpr int KCH = DQK / 64;
  static constexpr int VCH = DV / 64;
  static constexpr int K_OFF = 0;
  static constexpr int V_OFF = K_OFF + KCH * kChunkBytes;
  static constexpr int Q_OFF = V_OFF + VCH * kChunkBytes;  // two slots
  static constexpr int Q_SLOT = KCH * kChunkBytes;
  static constexpr int DO_OFF = Q_OFF + 2 * Q_SLOT;
  static constexpr int DS_OFF = DO_OFF + VCH * kChunkBytes;  // dS^T; the dK/dV epilogue stages here (8 x 4 KB)
  static constexpr int STG_OFF = DS_OFF + 2 * kChunkBytes;   // dQ read-out staging (4 warps x 4 KB)
  static constexpr int ROWV_OFF = STG_OFF + 4 * 4096;
  static constexpr int SMEM_BYTES = ROWV_OFF + 2 * 8 * 64 * 4 + 1024;
  static constexpr int T_DV = 0;
  static constexpr int T_DK = DV;
  static constexpr int T_A = 256;
  static constexpr int T_B = 384;
  static_assert(DQK <= 128 && DV <= 128, "dual-region plan needs Dqk, Dv <= 128");
  static_assert(SMEM_BYTES <= 232448, "shared memory budget");
};

// CAP: logits softcapped (p.softcap > 0). Pass 1 then also writes
// P (1 - tanh^2) of the capped logit, packed, into the other 32 columns of
// its half of region A (S^T columns it has already read and dV never reads),
// and pass 2 takes dS^T from those instead of from P^T.
// PACK: a step takes the p.pack query heads of its KV head (p.seg.qrows rows
// each); without it one head of 128 rows, with compile-time tile arithmetic.
template <typename T, int DQK, int DV, bool CAP, bool PACK>
__global__ void __launch_bounds__(512, 1) attn_bwd_dual_kernel(const __grid_constant__ BwdParams p) {
  using C = BwdDualCfg<DQK, DV>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  float* nlse_s = reinterpret_cast<float*>(smem + C::ROWV_OFF);  // [8 compute warps][64]: -lse * log2(e)
  float* ndl_s = nlse_s + 8 * 64;                                 // [8 compute warps][64]: -Delta

  __shared__ uint64_t kv_full, kv_empty, q_full[2], q_empty[2], do_full, do_empty, s_full, dp_full[2], p_full,
      ds_full, ds_free, dq_full, dq_free[2], acc_done, acc_free, drain, work_full[2], work_empty[2];
  __shared__ int work_slot[2];
  __shared__ BwdItem work_tile[2];
  __shared__ uint32_t tmem_base_smem;
  __shared__ int abort_flag;

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  if (threadIdx.x == 0) {
    mbar_init(&kv_full, 1);
    mbar_init(&kv_empty, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&q_full[i], 1);
      mbar_init(&q_empty[i], 1);
    }
    mbar_init(&do_full, 1);
    mbar_init(&do_empty, 1);
    mbar_init(&s_full, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&dp_full[i], 1);
      mbar_init(&dq_free[i], 4);
    }
    mbar_init(&p_full, 8);
    mbar_init(&ds_full, 8);
    mbar_init(&ds_free, 1);
    mbar_init(&dq_full, 1);
    mbar_init(&acc_done, 1);
    mbar_init(&acc_free, 8);
    mbar_init(&drain, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&work_full[i], 1);
      mbar_init(&work_empty[i], 13);  // the MMA thread, eight compute and four dQ warps
    }
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
  const int hpack = PACK ? p.pack : 1;        // query heads per step
  const int qrows = PACK ? p.seg.qrows : kBM;  // rows of each of them
  const uint32_t sbase = smem_u32(smem);
  // Next work item for the MMA, compute and dQ warps (-1: none left, or
  // abort), with its decoded unit.
  uint32_t nwork = 0;
  auto next_work = [&](bool& ok, BwdItem& t) -> int {
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

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&p.tm_q);
      tma_prefetch_desc(&p.tm_k);
      tma_prefetch_desc(&p.tm_v);
      tma_prefetch_desc(&p.tm_do);
      uint32_t nz = 0, gstep = 0;
      bool ok = true;
      // Each unit is decoded (two dependent global reads) while the previous
      // one's first step loads, and published decoded.
      int w = blockIdx.x;
      BwdItem tw{};
      if (w < total) tw = bwd_decode(p, w);
      while (ok) {
        if (w >= total) w = -1;
        const int ws = nwork & 1;
        if (!wait_bar(&work_empty[ws], ((nwork >> 1) & 1) ^ 1, ctl)) break;
        work_slot[ws] = w;
        work_tile[ws] = tw;
        mbar_arrive(&work_full[ws]);
        ++nwork;
        if (w < 0) break;
        const BwdItem t = tw;
        const int wn = gridDim.x + atomicAdd(p.work_next, 1);
        bool decoded = false;
        if (t.k1 > t.k0) {
          if (!wait_bar(&kv_empty, (nz & 1) ^ 1, ctl)) break;
          mbar_arrive_expect_tx(&kv_full, (C::KCH + C::VCH) * kChunkBytes);
          const int fk = t.ck0 + t.kt * kBN, bk = fk / p.seg.Sk, sk = fk - bk * p.seg.Sk;
          for (int c = 0; c < C::KCH; ++c)
            tma_load_4d(smem + C::K_OFF + c * kChunkBytes, &p.tm_k, &kv_full, c * 64, sk, t.hk, bk);
          for (int c = 0; c < C::VCH; ++c)
            tma_load_4d(smem + C::V_OFF + c * kChunkBytes, &p.tm_v, &kv_full, c * 64, sk, t.hk, bk);
          ++nz;
          for (int k = t.k0; k < t.k1; ++k, ++gstep) {
            // the step's first query head (p.pack heads per step) and query tile
            const int h = t.hk * G + (k / t.nqt) * hpack, qt = t.qt0 + k % t.nqt;
            const int fq = t.cq0 + qt * qrows, bq = fq / p.seg.Sq, sq = fq - bq * p.seg.Sq;
            const int qs = gstep & 1;
            if (!wait_bar(&q_empty[qs], ((gstep >> 1) & 1) ^ 1, ctl)) {
              ok = false;
              break;
            }
            mbar_arrive_expect_tx(&q_full[qs], C::KCH * kChunkBytes);
            for (int c = 0; c < C::KCH; ++c)
              tma_load_4d(smem + C::Q_OFF + qs * C::Q_SLOT + c * kChunkBytes, &p.tm_q, &q_full[qs], c * 64, sq, h, bq);
            if (!wait_bar(&do_empty, (gstep & 1) ^ 1, ctl)) {
              ok = false;
              break;
            }
            mbar_arrive_expect_tx(&do_full, C::VCH * kChunkBytes);
            for (int c = 0; c < C::VCH; ++c)
              tma_load_4d(smem + C::DO_OFF + c * kChunkBytes, &p.tm_do, &do_full, c * 64, sq, h, bq);
            if (k == t.k0 && wn < total) {
              tw = bwd_decode(p, wn);
              decoded = true;
            }
          }
        }
        if (!ok) break;
        if (!decoded && wn < total) tw = bwd_decode(p, wn);
        w = wn;
      }
      if (nz > 0) wait_bar_drain(&kv_full, (nz - 1) & 1, p.limit_ns);
      for (uint32_t i = gstep > 2 ? gstep - 2 : 0; i < gstep; ++i) wait_bar_drain(&q_full[i & 1], (i >> 1) & 1, p.limit_ns);
      if (gstep > 0) wait_bar_drain(&do_full, (gstep - 1) & 1, p.limit_ns);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t id_sq = idesc_f32acc<T>(128, 128, 0, 0);  // S^T = K Q^T
      constexpr uint32_t id_dp = idesc_f32acc<T>(128, 64, 0, 0);   // one half of dP^T = V dO^T
      constexpr uint32_t id_dv = idesc_f32acc<T>(128, DV, 0, 1);   // dV += P^T (TMEM) dO
      constexpr uint32_t id_dk = idesc_f32acc<T>(128, DQK, 0, 1);  // dK += dS^T Q
      constexpr uint32_t id_dq = idesc_f32acc<T>(128, DQK, 1, 1);  // dQ  = dS K
      const uint32_t k_a = sbase + C::K_OFF, v_a = sbase + C::V_OFF, q_a0 = sbase + C::Q_OFF;
      const uint32_t do_a = sbase + C::DO_OFF, ds_a = sbase + C::DS_OFF;
      const uint32_t ra = tmem + C::T_A, rb = tmem + C::T_B;
      uint32_t nz = 0, gstep = 0;
      bool ok = true;
      while (ok) {
        BwdItem t;
        const int w = next_work(ok, t);
        if (w < 0) break;
        if (t.k1 == t.k0) continue;
        if (!wait_bar(&kv_full, nz & 1, ctl)) break;
        if (nz > 0 && !wait_bar(&acc_free, (nz - 1) & 1, ctl)) break;
        tc_fence_after();
        // S of the range's first step; later ones are issued inside the loop.
        {
          const int qs = gstep & 1;
          if (!wait_bar(&q_full[qs], (gstep >> 1) & 1, ctl)) break;
          tc_fence_after();
          for (int c = 0; c < C::KCH; ++c) {
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              mma_ss(ra, sdesc_sw128(k_a + c * kChunkBytes + kk * 32, 16, 1024),
                     sdesc_sw128(q_a0 + qs * C::Q_SLOT + c * kChunkBytes + kk * 32, 16, 1024), id_sq, (c | kk) != 0);
          }
          mma_commit(&s_full);
        }
        for (int k = t.k0; k < t.k1 && ok; ++k, ++gstep) {
          const int qs = gstep & 1;
          const uint32_t q_a = q_a0 + qs * C::Q_SLOT;
          // dP^T in two N = 64 halves (query rows 0-63, 64-127), each issued
          // as soon as the dQ read-out has freed its columns of B; each
          // compute warpgroup waits only for its own half.
          if (!wait_bar(&do_full, gstep & 1, ctl)) {
            ok = false;
            break;
          }
          for (int hh = 0; hh < 2 && ok; ++hh) {
            if (gstep > 0 && (hh == 0 || DQK > 64) && !wait_bar(&dq_free[hh], (gstep - 1) & 1, ctl)) {
              ok = false;
              break;
            }
            tc_fence_after();
            for (int c = 0; c < C::VCH; ++c) {
#pragma unroll
              for (int kk = 0; kk < 4; ++kk)
                mma_ss(rb + hh * 64, sdesc_sw128(v_a + c * kChunkBytes + kk * 32, 16, 1024),
                       sdesc_sw128(do_a + c * kChunkBytes + hh * 8192 + kk * 32, 16, 1024), id_dp, (c | kk) != 0);
            }
            mma_commit(&dp_full[hh]);
          }
          if (!ok) break;
          if (!wait_bar(&p_full, gstep & 1, ctl)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t first = (k == t.k0) ? 1u : 0u;
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            mma_ts(tmem + C::T_DV, ra + kk * 8 + (kk >= 4 ? 32 : 0), sdesc_sw128(do_a + kk * 2048, kChunkBytes, 1024), id_dv,
                   !(first && kk == 0));
          mma_commit(&do_empty);
          if (!wait_bar(&ds_full, gstep & 1, ctl)) {
            ok = false;
            break;
          }
          tc_fence_after();
          if (k + 1 < t.k1) {
            // Next step's S into A: P^T(g) there has been read by dV(g), issued before.
            const int qn = (gstep + 1) & 1;
            if (!wait_bar(&q_full[qn], ((gstep + 1) >> 1) & 1, ctl)) {
              ok = false;
              break;
            }
            tc_fence_after();
            for (int c = 0; c < C::KCH; ++c) {
#pragma unroll
              for (int kk = 0; kk < 4; ++kk)
                mma_ss(ra, sdesc_sw128(k_a + c * kChunkBytes + kk * 32, 16, 1024),
                       sdesc_sw128(q_a0 + qn * C::Q_SLOT + c * kChunkBytes + kk * 32, 16, 1024), id_sq,
                       (c | kk) != 0);
            }
            mma_commit(&s_full);
          }
          // dQ before dK: its read-out, which frees region B for the next dP,
          // then overlaps the dK MMAs.
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            mma_ss(rb, sdesc_sw128(ds_a + kk * 2048, kChunkBytes, 1024), sdesc_sw128(k_a + kk * 2048, kChunkBytes, 1024),
                   id_dq, kk > 0);
          mma_commit(&dq_full);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            mma_ss(tmem + C::T_DK, sdesc_sw128(ds_a + (kk >> 2) * kChunkBytes + (kk & 3) * 32, 16, 1024),
                   sdesc_sw128(q_a + kk * 2048, kChunkBytes, 1024), id_dk, !(first && kk == 0));
          mma_commit(&q_empty[qs]);
          mma_commit(&ds_free);
        }
        if (!ok) break;
        mma_commit(&acc_done);
        mma_commit(&kv_empty);
        ++nz;
      }
      mma_commit(&drain);
      wait_bar_drain(&drain, 0, p.limit_ns);
    }
  } else if (warp >= 4 && (warp < 8 || warp >= 12)) {
    // ------------------------------------------------------------ compute warpgroups
    // Warps 4-7 take query columns [0, 64) of every step, warps 12-15 columns
    // [64, 128); thread = key row in both.
    const int half = warp >= 12 ? 1 : 0;
    const int wq = warp & 3;
    const int cb = half * 64;                       // first query column of this half
    const uint32_t pofs = half ? 64 : 0;            // where this half's P^T sits in A
    const int r = 32 * wq + lane;                   // key row within the tile
    const uint32_t lane_base = (uint32_t)(32 * wq) << 16;
    float* my_nlse = nlse_s + (half * 4 + wq) * 64;
    float* my_ndl = ndl_s + (half * 4 + wq) * 64;
    uint8_t* ds_s = smem + C::DS_OFF + half * kChunkBytes;
    uint8_t* epi = smem + C::DS_OFF + (half * 4 + wq) * 4096;  // one 4 KB box per warp, used between units
    const float sl2 = p.scale_log2;
    const float2 sl2x2 = make_float2(sl2, sl2), one2 = make_float2(1.f, 1.f), zero2 = make_float2(0.f, 0.f);
    const float cap_c2 = CAP ? p.softcap * 1.4426950408889634f : 0.f;
    const float cap_k1 = CAP ? 2.f * sl2 / p.softcap : 0.f, cap_ic2 = CAP ? 1.f / cap_c2 : 0.f;
    // Query column qc of a step is row i0 + (qc & rmask) of query head
    // h0 + qc / qrows (qrows = 128 unless a KV head's query heads share a tile).
    const int rmask = qrows - 1, qshift = PACK ? 31 - __clz(qrows) : 7;  // qrows is a power of two
    uint32_t nz = 0, gstep = 0;
    bool ok = true;
    // lse and Delta of 2 of this half's query columns per lane for one step,
    // loaded one step ahead and left in flight (-inf / 0 outside the segment).
    auto fetch_rows = [&](const BwdItem& t, int k, float (&lv)[2], float (&dv)[2]) {
      const int h0 = t.hk * G + (k / t.nqt) * hpack, i0 = (t.qt0 + k % t.nqt) * qrows;
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int qc = cb + lane * 2 + e;
        const int h = h0 + (qc >> qshift), ri = qc & rmask;
        const int f = t.cq0 + i0 + ri;
        const bool in = i0 + ri < t.m && f < p.q_rows;
        const int fs = in ? f : 0;
        const int bq = fs / p.seg.Sq, sq = fs - bq * p.seg.Sq;
        lv[e] = -CUDART_INF_F;
        dv[e] = 0.f;
        ldg_pred_f32(lv[e], p.lse + bq * p.l_sb + h * p.l_sh + sq, in);
        ldg_pred_f32(dv[e], p.delta + (int64_t)h * p.q_rows + fs, in);
      }
    };
    // -lse * log2(e) (-inf where the row carries no probability, so P = 0).
    auto neg_lse2 = [](float x) { return x == -CUDART_INF_F ? -CUDART_INF_F : -x * 1.4426950408889634f; };
    while (ok) {
      BwdItem t;
      const int w = next_work(ok, t);
      if (w < 0) break;
      const int j = t.kt * kBN + r;  // segment-local key index
      const bool valid = j < t.n;
      // This key row's dV (warps 4-7) or dK (warps 12-15) in the output.
      const int fk = t.ck0 + j, bk = fk / p.seg.Sk, sk = fk - bk * p.seg.Sk;
      T* const out_row = half ? static_cast<T*>(p.dk) + bk * p.k_sb + (int64_t)sk * p.k_ss + t.hk * p.k_sh
                              : static_cast<T*>(p.dv) + bk * p.v_sb + (int64_t)sk * p.v_ss + t.hk * p.v_sh;
      if (t.k1 == t.k0) {
        // No query sees this key tile (never cut): its dK and dV are zero.
        if (valid)
          for (int c = 0; c < (half ? DQK : DV) / 8; ++c) reinterpret_cast<uint4*>(out_row)[c] = make_uint4(0, 0, 0, 0);
        continue;
      }
      const int delta = t.n - t.m;
      float nlv[2], ndv[2];
      fetch_rows(t, t.k0, nlv, ndv);
      for (int k = t.k0; k < t.k1; ++k, ++gstep) {
        const int i0 = (t.qt0 + k % t.nqt) * qrows;
        *reinterpret_cast<float2*>(my_nlse + lane * 2) = make_float2(neg_lse2(nlv[0]), neg_lse2(nlv[1]));
        *reinterpret_cast<float2*>(my_ndl + lane * 2) = make_float2(-ndv[0], -ndv[1]);
        __syncwarp();
        if (k + 1 < t.k1) fetch_rows(t, k + 1, nlv, ndv);
        // Per-key visible query rows [q_lo, q_hi) of the tile, relative to i0
        // (the same rows in every head block of a packed tile); this half's
        // columns cover rows [rstart, rend) of each of its head blocks.
        int q_lo = p.seg.causal ? j - delta - i0 : -0x40000000;
        int q_hi = t.m - i0;
        if (p.seg.window > 0) q_hi = min(q_hi, j - delta + p.seg.window - i0);
        if (!valid) q_lo = q_hi = 0;
        const int rstart = cb & rmask, rend = rstart + min(64, qrows);
        const bool masked = __any_sync(0xffffffffu, q_lo > rstart || q_hi < rend);
        if (!wait_bar(&s_full, gstep & 1, ctl)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t ra = tmem + lane_base + C::T_A, rb = tmem + lane_base + C::T_B;
        // Pass 1: P^T = exp2(S^T * scale * log2 e - lse * log2 e) as packed bf16;
        // chunk c of this half's S^T columns -> A[pofs + 16c, pofs + 16c + 16),
        // columns this half has already read.
        auto pass1 = [&](auto tag) {
          constexpr bool MASK = decltype(tag)::value;
          uint32_t sa[32], sb[32];
          tmem_ld32_async(ra + cb, sa);
          tmem_ld32_async(ra + cb + 32, sb);
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            uint32_t(&cur)[32] = c ? sb : sa;
            tmem_wait_ld32(cur);
            uint32_t pk[16];
            [[maybe_unused]] uint32_t pfk[16];  // CAP only
#pragma unroll
            for (int e4 = 0; e4 < 8; ++e4) {
              const float4 nl = *reinterpret_cast<const float4*>(my_nlse + c * 32 + e4 * 4);
#pragma unroll
              for (int hf = 0; hf < 2; ++hf) {
                const int e = e4 * 2 + hf;
                const float2 nl2 = hf ? make_float2(nl.z, nl.w) : make_float2(nl.x, nl.y);
                float2 x;
                [[maybe_unused]] float2 fac = one2;  // CAP only
                if constexpr (CAP) {
                  const float2 y = make_float2(softcap_log2(__uint_as_float(cur[2 * e]), cap_k1, cap_c2),
                                               softcap_log2(__uint_as_float(cur[2 * e + 1]), cap_k1, cap_c2));
                  x = fma2(y, one2, nl2);
                  const float2 tt = make_float2(y.x * cap_ic2, y.y * cap_ic2);
                  fac = make_float2(fmaf(-tt.x, tt.x, 1.f), fmaf(-tt.y, tt.y, 1.f));
                } else {
                  x = fma2(make_float2(__uint_as_float(cur[2 * e]), __uint_as_float(cur[2 * e + 1])), sl2x2, nl2);
                }
                float p0 = ex2_approx(x.x), p1 = ex2_approx(x.y);
                if constexpr (MASK) {
                  const int rc = (cb + c * 32 + 2 * e) & rmask;  // row of the column pair's first column
                  p0 = (rc < q_lo || rc >= q_hi) ? 0.f : p0;
                  p1 = (rc + 1 < q_lo || rc + 1 >= q_hi) ? 0.f : p1;
                }
                pk[e] = pack2<T>(p0, p1);
                if constexpr (CAP) pfk[e] = pack2<T>(p0 * fac.x, p1 * fac.y);
              }
            }
            tmem_st16_async(ra + pofs + c * 16, pk);
            if constexpr (CAP) tmem_st16_async(ra + pofs + 32 + c * 16, pfk);
          }
          tmem_wait_st();
        };
        if (masked)
          pass1(MaskTag<true>{});
        else
          pass1(MaskTag<false>{});
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&p_full);
        // Pass 2: dS^T = P^T (dP^T - Delta) into this half's 64 columns of the
        // dS^T buffer (bf16, 128-byte swizzled).
        if (!wait_bar(&dp_full[half], gstep & 1, ctl) || (gstep > 0 && !wait_bar(&ds_free, (gstep - 1) & 1, ctl))) {
          ok = false;
          break;
        }
        tc_fence_after();
        {
          // Four 16-column pieces, the next one's TMEM loads in flight.
          uint32_t da[16], db[16], pa[8], pb[8];
          tmem_ld16_async(rb + cb, da);
          constexpr uint32_t kPsrc = CAP ? 32 : 0;  // P^T, or P^T (1 - tanh^2) with a cap
          tmem_ld8_async(ra + pofs + kPsrc, pa);
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            uint32_t(&dcur)[16] = (c & 1) ? db : da;
            uint32_t(&dnxt)[16] = (c & 1) ? da : db;
            uint32_t(&pcur)[8] = (c & 1) ? pb : pa;
            uint32_t(&pnxt)[8] = (c & 1) ? pa : pb;
            tmem_wait_ld16_8(dcur, pcur);
            if (c + 1 < 4) {
              tmem_ld16_async(rb + cb + (c + 1) * 16, dnxt);
              tmem_ld8_async(ra + pofs + kPsrc + (c + 1) * 8, pnxt);
            }
            uint32_t dk2[8];
#pragma unroll
            for (int e4 = 0; e4 < 4; ++e4) {
              const float4 nd = *reinterpret_cast<const float4*>(my_ndl + c * 16 + e4 * 4);
#pragma unroll
              for (int hf = 0; hf < 2; ++hf) {
                const int e = e4 * 2 + hf;
                const float2 nd2 = hf ? make_float2(nd.z, nd.w) : make_float2(nd.x, nd.y);
                const float2 pf = unpack2<T>(pcur[e]);
                const float2 dd =
                    fma2(make_float2(__uint_as_float(dcur[2 * e]), __uint_as_float(dcur[2 * e + 1])), one2, nd2);
                const float2 ds = fma2(pf, dd, zero2);
                dk2[e] = pack2<T>(ds.x, ds.y);
              }
            }
#pragma unroll
            for (int u = 0; u < 2; ++u)
              *reinterpret_cast<uint4*>(ds_s + sw128_offset(r, c * 2 + u)) =
                  make_uint4(dk2[4 * u], dk2[4 * u + 1], dk2[4 * u + 2], dk2[4 * u + 3]);
          }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&ds_full);
      }
      if (!ok) break;
      // Epilogue: this range's dV (warps 4-7) or dK (warps 12-15). A whole key
      // tile writes its rows straight to the output (dK scaled); a cut tile's
      // sub-range stores its fp32 partial sums to its own slot in 32 x 32
      // boxes, and the convert adds the slots up.
      if (!wait_bar(&acc_done, nz & 1, ctl)) break;
      tc_fence_after();
      constexpr int NCV = DV / 32, NCK = DQK / 32;
      const int nc = half ? NCK : NCV;
      if (t.slot < 0) {
        const float sc = half ? p.scale : 1.f;
#pragma unroll 1
        for (int c = 0; c < nc; ++c) {
          uint32_t a[32];
          tmem_ld32(tmem + lane_base + (half ? C::T_DK : C::T_DV) + c * 32, a);
          if (c == nc - 1) {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&acc_free);
          }
          if (valid) {
            uint4* dst = reinterpret_cast<uint4*>(out_row + c * 32);
#pragma unroll
            for (int u = 0; u < 4; ++u)
              dst[u] = make_uint4(pack2<T>(__uint_as_float(a[8 * u]) * sc, __uint_as_float(a[8 * u + 1]) * sc),
                                  pack2<T>(__uint_as_float(a[8 * u + 2]) * sc, __uint_as_float(a[8 * u + 3]) * sc),
                                  pack2<T>(__uint_as_float(a[8 * u + 4]) * sc, __uint_as_float(a[8 * u + 5]) * sc),
                                  pack2<T>(__uint_as_float(a[8 * u + 6]) * sc, __uint_as_float(a[8 * u + 7]) * sc));
          }
        }
      } else {
#pragma unroll 1
        for (int c = 0; c < nc; ++c) {
          uint32_t a[32];
          tmem_ld32(tmem + lane_base + (half ? C::T_DK : C::T_DV) + c * 32, a);
          if (c == nc - 1) {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&acc_free);
          }
          if (c >= 1) {
            if (lane == 0) bulk_wait_group_read0();
            __syncwarp();
          }
#pragma unroll
          for (int u = 0; u < 8; ++u)
            *reinterpret_cast<uint4*>(epi + sw128_offset(lane, u)) =
                make_uint4(a[4 * u], a[4 * u + 1], a[4 * u + 2], a[4 * u + 3]);
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_store_4d(half ? &p.tm_dk : &p.tm_dv, epi, c * 32, 32 * wq, t.hk, t.slot);
            bulk_commit_group();
          }
        }
        // The boxes sit in the dS^T buffer: drain them before the next dS^T.
        if (lane == 0) bulk_wait_group_read0();
        __syncwarp();
      }
      ++nz;
    }
    if (lane == 0) bulk_wait_group0();
  } else if (warp >= 8 && warp < 12) {
    // ------------------------------------------------------------ dQ read-out
    const int wq = warp - 8;
    const uint32_t lane_base = (uint32_t)(32 * wq) << 16;
    uint8_t* box = smem + C::STG_OFF + wq * 4096;
    uint32_t gstep = 0;
    bool ok = true;
    while (ok) {
      BwdItem t;
      const int w = next_work(ok, t);
      if (w < 0) break;
      if (t.k1 == t.k0) continue;
      for (int k = t.k0; k < t.k1; ++k, ++gstep) {
        // this warp's 32 rows lie in one head block (packing keeps qrows >= 32)
        const int h = t.hk * G + (k / t.nqt) * hpack + (32 * wq) / qrows, qt = t.qt0 + k % t.nqt;
        if (!wait_bar(&dq_full, gstep & 1, ctl)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t rq = tmem + lane_base + C::T_B;
        const int fq = t.cq0 + qt * qrows + ((32 * wq) & (qrows - 1)), bq = fq / p.seg.Sq, sq = fq - bq * p.seg.Sq;
        // One 32 x 32 fp32 box of dQ into the staging box and on to the
        // accumulator by TMA reduce-add (after the box's previous reduce has
        // read it).
        auto reduce_box = [&](const uint32_t(&v)[32], int cchunk) {
          if (lane == 0) bulk_wait_group_read0();
          __syncwarp();
#pragma unroll
          for (int u = 0; u < 8; ++u)
            *reinterpret_cast<uint4*>(box + sw128_offset(lane, u)) =
                make_uint4(v[4 * u], v[4 * u + 1], v[4 * u + 2], v[4 * u + 3]);
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_reduce_add_4d(&p.tm_dq, box, cchunk * 32, sq, h, bq);
            bulk_commit_group();
          }
        };
        // Columns 0-63 of B, then (Dqk = 128) columns 64-127 as soon as the
        // first box is on its way, so both dP halves can follow the dQ MMA
        // without waiting for the boxes' reduce traffic.
        uint32_t a[2][32];
        tmem_ld32x2(rq, rq + 32, a[0], a[1]);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&dq_free[0]);
        reduce_box(a[0], 0);
        if constexpr (DQK > 64) {
          uint32_t b[2][32];
          tmem_ld32x2(rq + 64, rq + 96, b[0], b[1]);
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&dq_free[1]);
          reduce_box(a[1], 1);
          reduce_box(b[0], 2);
          reduce_box(b[1], 3);
        } else {
          reduce_box(a[1], 1);
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

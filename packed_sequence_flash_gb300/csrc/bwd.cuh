// bwd.cuh -- attention backward for sm_103a, from the caller-supplied out/lse.
//   [nemo_automodel.components.attention.ffpa_attention, `_ffpa_varlen_bwd`,
//    `_ffpa_dense_bwd`: gradients "using the caller-supplied out/lse", "dK/dV
//    reduced to Hkv for GQA"]
//
// Per (segment, KV head, 128-row key tile) a CTA keeps K and V in shared
// memory and walks every (query head of the GQA group, 128-row query tile)
// that can see the key tile. For each step, with thread r of the compute
// warpgroup owning key row r (TMEM lane r):
//   S^T  = K Q^T           (tcgen05, fp32 in TMEM)
//   dP^T = V dO^T          (tcgen05)
//   P^T  = exp2(S^T * scale * log2 e - lse * log2 e), 0 where masked or lse = -inf
//   dS^T = P^T (dP^T - Delta),  Delta = rowsum(dO * out) from the preprocess
//   dV  += P^T dO          (tcgen05, accumulated in TMEM across the whole group)
//   dK  += dS^T Q          (idem; the scale is applied once in the epilogue)
//   dQ   = dS K            (tcgen05 into TMEM, then added to an fp32 global
//                           accumulator with TMA reduce-add, 32 x 32 boxes)
// P^T and dS^T are written to shared memory as bf16 in the 128-byte-swizzled
// layout, which the MMAs read K-major (as P^T, dS^T) or M-major (as dS).
//
// TMEM plans: with Dqk, Dv <= 128 two 128-column regions alternate between S
// and dP so the next step's S^T overlaps the dQ read-out ("dual"); with
// Dqk = 192 a single 192-column region is reused for S, dP and dQ in turn.
//
// Warps: 0 TMA producer, 1 MMA issuer, 2 TMEM allocator, 4-7 compute
// (P, dS, and the dK/dV epilogue), 8-11 dQ read-out.
#pragma once

#include <math_constants.h>

#include "common.cuh"

namespace psf {

struct BwdParams {
  CUtensorMap tm_q, tm_k, tm_v, tm_do;  // bf16 (d, s, h, b) views, box (64, 128)
  CUtensorMap tm_dq;                    // fp32 dQ accumulator [rows][Hq][Dqk], box (32, 32)
  CUtensorMap tm_dk, tm_dv;             // fp32 dK / dV accumulators [rows][Hkv][D], box (32, 32)
  SegInfo seg;
  const float* lse;
  int64_t l_sb, l_sh;
  const float* delta;  // [Hq][q_rows]
  int q_rows;
  void* dk;  // T
  int64_t k_sb, k_ss, k_sh;  // element strides of dk (batch, row, head)
  void* dv;  // T
  int64_t v_sb, v_ss, v_sh;  // element strides of dv
  int Hq, Hkv;
  float scale, scale_log2;
  int pack;       // query heads per step: 1, or Hq / Hkv when a KV head's query heads share one tile
  float softcap;  // > 0: logits capped as softcap * tanh(logit / softcap) (the CAP kernels)
  const int4* items;  // (segment, key tile, first step, end step), heaviest first
  const int* n_items;
  int* work_next;  // zeroed by the schedule kernel; kernels that take work dynamically count on it
  int* status;
  uint64_t limit_ns;
};

template <int DQK, int DV>
struct BwdCfg {
  static constexpr int KCH = DQK / 64;
  static constexpr int VCH = DV / 64;
  static constexpr bool DUAL = DQK <= 128 && DV <= 128;
  static constexpr int K_OFF = 0;
  static constexpr int V_OFF = K_OFF + KCH * kChunkBytes;
  static constexpr int Q_OFF = V_OFF + VCH * kChunkBytes;
  static constexpr int DO_OFF = Q_OFF + KCH * kChunkBytes;
  static constexpr int PT_OFF = DO_OFF + VCH * kChunkBytes;
  // The single-region plan writes dS^T over P^T once the dV MMA has read it,
  // and stages dQ in that same buffer once the dQ MMA has read dS.
  static constexpr int DS_OFF = DUAL ? PT_OFF + 2 * kChunkBytes : PT_OFF;
  static constexpr int STG_OFF = DUAL ? DS_OFF + 2 * kChunkBytes : PT_OFF;  // 4 x 4 KB dQ staging
  static constexpr int ROWV_OFF = DUAL ? STG_OFF + 4 * 4096 : PT_OFF + 2 * kChunkBytes;
  static constexpr int SMEM_BYTES = ROWV_OFF + 2 * 4 * 128 * 4 + 1024;
  // TMEM columns
  static constexpr int T_DV = 0;
  static constexpr int T_DK = DUAL ? DV : 128;
  static constexpr int T_A = DUAL ? 256 : 320;
  static constexpr int T_B = DUAL ? 384 : 320;
  // Single-region plan with a softcap: P^T (1 - tanh^2), packed, between the passes.
  static constexpr int T_PF = 448;
  static_assert(SMEM_BYTES <= 232448, "shared memory budget");
  static_assert(DUAL || (DQK == 192 && DV == 128), "single-region plan is laid out for (192, 128)");
};

// One work unit: a key tile of one KV head and a range [k0, k1) of its steps.
// Step k is query head hk * G + k / nqt and query tile qt0 + k % nqt.
struct BwdItem {
  int s, kt, hk;
  int cq0, ck0, m, n;
  int qt0, nqt;  // query tiles [qt0, qt0 + nqt) (of p.seg.qrows rows) see this key tile
  int k0, k1;
};

__device__ __forceinline__ BwdItem bwd_decode(const BwdParams& p, int w) {
  BwdItem t;
  const int item = w / p.Hkv;
  t.hk = w - item * p.Hkv;
  const int4 it = p.items[item];
  t.s = it.x;
  t.kt = it.y;
  t.k0 = it.z;
  t.k1 = it.w;
  t.cq0 = cu_q_at(p.seg, t.s);
  t.ck0 = cu_k_at(p.seg, t.s);
  t.m = cu_q_at(p.seg, t.s + 1) - t.cq0;
  t.n = cu_k_at(p.seg, t.s + 1) - t.ck0;
  int lo, hi;
  q_range_for_kv_tile(t.m, t.n, t.kt * kBN, p.seg.causal, p.seg.window, lo, hi);
  t.qt0 = lo / p.seg.qrows;
  t.nqt = hi > lo ? ceil_div(hi, p.seg.qrows) - t.qt0 : 0;
  return t;
}

// CAP: logits softcapped (p.softcap > 0); dS carries the cap's 1 - tanh^2.
template <typename T, int DQK, int DV, bool CAP>
__global__ void __launch_bounds__(384, 1) attn_bwd_kernel(const __grid_constant__ BwdParams p) {
  using C = BwdCfg<DQK, DV>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  float* lse_s = reinterpret_cast<float*>(smem + C::ROWV_OFF);  // [4 warps][128]
  float* dl_s = lse_s + 4 * 128;

  __shared__ uint64_t kv_full, kv_empty, q_full, q_empty, s_full, dp_full, p_full, pt_read, ds_full, ds_free,
      dq_full, dq_free, acc_done, acc_free, drain;
  __shared__ uint32_t tmem_base_smem;
  __shared__ int abort_flag;

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  if (threadIdx.x == 0) {
    mbar_init(&kv_full, 1);
    mbar_init(&kv_empty, 1);
    mbar_init(&q_full, 1);
    mbar_init(&q_empty, 1);
    mbar_init(&s_full, 1);
    mbar_init(&dp_full, 1);
    mbar_init(&p_full, 4);
    mbar_init(&pt_read, 1);
    mbar_init(&ds_full, 4);
    mbar_init(&ds_free, 1);
    mbar_init(&dq_full, 1);
    mbar_init(&dq_free, 4);
    mbar_init(&acc_done, 1);
    mbar_init(&acc_free, 4);
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
        for (int k = t.k0; k < t.k1; ++k) {
          const int h = t.hk * G + k / t.nqt, qt = t.qt0 + k % t.nqt;
          if (!wait_bar(&q_empty, (gstep & 1) ^ 1, ctl)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&q_full, (C::KCH + C::VCH) * kChunkBytes);
          const int fq = t.cq0 + qt * kBM, bq = fq / p.seg.Sq, sq = fq - bq * p.seg.Sq;
          for (int c = 0; c < C::KCH; ++c)
            tma_load_4d(smem + C::Q_OFF + c * kChunkBytes, &p.tm_q, &q_full, c * 64, sq, h, bq);
          for (int c = 0; c < C::VCH; ++c)
            tma_load_4d(smem + C::DO_OFF + c * kChunkBytes, &p.tm_do, &q_full, c * 64, sq, h, bq);
          ++gstep;
        }
      }
      if (nz > 0) wait_bar_drain(&kv_full, (nz - 1) & 1, p.limit_ns);
      if (gstep > 0) wait_bar_drain(&q_full, (gstep - 1) & 1, p.limit_ns);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t id_sq = idesc_f32acc<T>(128, 128, 0, 0);  // S^T, dP^T
      constexpr uint32_t id_dv = idesc_f32acc<T>(128, DV, 0, 1);   // dV += P^T dO
      constexpr uint32_t id_dk = idesc_f32acc<T>(128, DQK, 0, 1);  // dK += dS^T Q
      constexpr uint32_t id_dq = idesc_f32acc<T>(128, DQK, 1, 1);  // dQ = dS K
      const uint32_t k_a = sbase + C::K_OFF, v_a = sbase + C::V_OFF, q_a = sbase + C::Q_OFF;
      const uint32_t do_a = sbase + C::DO_OFF, pt_a = sbase + C::PT_OFF, ds_a = sbase + C::DS_OFF;
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
          if (!wait_bar(&q_full, gstep & 1, ctl)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t rs = tmem + (C::DUAL ? ((gstep & 1) ? C::T_B : C::T_A) : C::T_A);  // S (and dQ)
          const uint32_t rp = tmem + (C::DUAL ? ((gstep & 1) ? C::T_A : C::T_B) : C::T_A);  // dP
          if (!C::DUAL && gstep > 0 && !wait_bar(&dq_free, (gstep - 1) & 1, ctl)) {
            ok = false;
            break;
          }
          for (int c = 0; c < C::KCH; ++c) {
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              mma_ss(rs, sdesc_sw128(k_a + c * kChunkBytes + kk * 32, 16, 1024),
                     sdesc_sw128(q_a + c * kChunkBytes + kk * 32, 16, 1024), id_sq, (c | kk) != 0);
          }
          mma_commit(&s_full);
          if (C::DUAL) {
            if (gstep > 0 && !wait_bar(&dq_free, (gstep - 1) & 1, ctl)) {
              ok = false;
              break;
            }
          } else {
            if (!wait_bar(&p_full, gstep & 1, ctl)) {
              ok = false;
              break;
            }
          }
          tc_fence_after();
          for (int c = 0; c < C::VCH; ++c) {
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              mma_ss(rp, sdesc_sw128(v_a + c * kChunkBytes + kk * 32, 16, 1024),
                     sdesc_sw128(do_a + c * kChunkBytes + kk * 32, 16, 1024), id_sq, (c | kk) != 0);
          }
          mma_commit(&dp_full);
          const uint32_t first = (k == t.k0) ? 1u : 0u;
          if (!C::DUAL) {
            // P^T is already in shared memory: dV can start while dS is computed.
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
              mma_ss(tmem + C::T_DV, sdesc_sw128(pt_a + (kk >> 2) * kChunkBytes + (kk & 3) * 32, 16, 1024),
                     sdesc_sw128(do_a + kk * 2048, kChunkBytes, 1024), id_dv, !(first && kk == 0));
            mma_commit(&pt_read);
          }
          if (!wait_bar(&ds_full, gstep & 1, ctl)) {
            ok = false;
            break;
          }
          tc_fence_after();
          if (C::DUAL) {
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
              mma_ss(tmem + C::T_DV, sdesc_sw128(pt_a + (kk >> 2) * kChunkBytes + (kk & 3) * 32, 16, 1024),
                     sdesc_sw128(do_a + kk * 2048, kChunkBytes, 1024), id_dv, !(first && kk == 0));
          }
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            mma_ss(tmem + C::T_DK, sdesc_sw128(ds_a + (kk >> 2) * kChunkBytes + (kk & 3) * 32, 16, 1024),
                   sdesc_sw128(q_a + kk * 2048, kChunkBytes, 1024), id_dk, !(first && kk == 0));
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            mma_ss(rs, sdesc_sw128(ds_a + kk * 2048, kChunkBytes, 1024), sdesc_sw128(k_a + kk * 2048, kChunkBytes, 1024),
                   id_dq, kk > 0);
          mma_commit(&ds_free);
          mma_commit(&dq_full);
          mma_commit(&q_empty);
        }
        if (!ok) break;
        mma_commit(&acc_done);
        mma_commit(&kv_empty);
        ++nz;
      }
      mma_commit(&drain);
      wait_bar_drain(&drain, 0, p.limit_ns);
    }
  } else if (warp >= 4 && warp < 8) {
    // ------------------------------------------------------------ compute warpgroup
    const int wq = warp - 4;
    const int r = threadIdx.x - 128;  // key row within the tile
    const uint32_t lane_base = (uint32_t)(32 * wq) << 16;
    float* my_lse = lse_s + wq * 128;
    float* my_dl = dl_s + wq * 128;
    uint8_t* pt_s = smem + C::PT_OFF;
    uint8_t* ds_s = smem + C::DS_OFF;
    const float sl2 = p.scale_log2;
    const float cap_c2 = CAP ? p.softcap * 1.4426950408889634f : 0.f;
    const float cap_k1 = CAP ? 2.f * sl2 / p.softcap : 0.f, cap_ic2 = CAP ? 1.f / cap_c2 : 0.f;
    // P (and, with CAP, the factor 1 - tanh^2 of the capped logit) of score s
    // for a row whose lse (log2 units) is l2.
    auto prob = [&](float s, float l2, float& fac) -> float {
      if constexpr (CAP) {
        const float y = softcap_log2(s, cap_k1, cap_c2);
        const float tt = y * cap_ic2;
        fac = fmaf(-tt, tt, 1.f);
        return ex2_approx(y - l2);
      } else {
        fac = 1.f;
        return ex2_approx(fmaf(s, sl2, -l2));
      }
    };
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
        if (valid) {
          for (int c = 0; c < DQK / 8; ++c) reinterpret_cast<uint4*>(dk_row)[c] = make_uint4(0, 0, 0, 0);
          for (int c = 0; c < DV / 8; ++c) reinterpret_cast<uint4*>(dv_row)[c] = make_uint4(0, 0, 0, 0);
        }
        continue;
      }
      const int delta = t.n - t.m;
      // lse and Delta of 4 query columns per lane, loaded one step ahead and
      // left in flight until the step stages them (-inf / 0 outside the segment).
      auto fetch_rows = [&](int k, float (&lv)[4], float (&dv)[4]) {
        const int h = t.hk * G + k / t.nqt, i0 = (t.qt0 + k % t.nqt) * kBM;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int qc = lane * 4 + e;
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
      float rlv[4], rdv[4];
      fetch_rows(t.k0, rlv, rdv);
      {
        for (int k = t.k0; k < t.k1; ++k, ++gstep) {
          const int i0 = (t.qt0 + k % t.nqt) * kBM;
          // Per-key visible query columns [q_lo, q_hi) of this tile.
          int q_lo = p.seg.causal ? j - delta - i0 : -0x40000000;
          int q_hi = t.m - i0;
          if (p.seg.window > 0) q_hi = min(q_hi, j - delta + p.seg.window - i0);
          if (!valid) q_lo = q_hi = 0;
          const bool masked = q_lo > 0 || q_hi < kBM;
          // lse * log2(e) (+inf for rows without mass) and Delta for this step.
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int qc = lane * 4 + e;
            my_lse[qc] = rlv[e] == -CUDART_INF_F ? CUDART_INF_F : rlv[e] * 1.4426950408889634f;
            my_dl[qc] = rdv[e];
          }
          if (k + 1 < t.k1) fetch_rows(k + 1, rlv, rdv);
          __syncwarp();
          if (!wait_bar(&s_full, gstep & 1, ctl)) {
            ok = false;
            break;
          }
          if (gstep > 0 && !wait_bar(&ds_free, (gstep - 1) & 1, ctl)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t rs = tmem + lane_base + (C::DUAL ? ((gstep & 1) ? C::T_B : C::T_A) : C::T_A);
          const uint32_t rp = tmem + lane_base + (C::DUAL ? ((gstep & 1) ? C::T_A : C::T_B) : C::T_A);
          if (C::DUAL) {
            if (!wait_bar(&dp_full, gstep & 1, ctl)) {
              ok = false;
              break;
            }
            tc_fence_after();
#pragma unroll 1
            for (int c = 0; c < 4; ++c) {
              uint32_t sv[32], pv[32];
              tmem_ld32(rs + c * 32, sv);
              tmem_ld32(rp + c * 32, pv);
              uint32_t pk[16], dk2[16];
#pragma unroll
              for (int e = 0; e < 16; ++e) {
                float pr[2], dr[2];
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                  const int qc = c * 32 + 2 * e + u;
                  float fe;
                  float pe = prob(__uint_as_float(sv[2 * e + u]), my_lse[qc], fe);
                  if (masked && (qc < q_lo || qc >= q_hi)) pe = 0.f;
                  pr[u] = pe;
                  dr[u] = pe * fe * (__uint_as_float(pv[2 * e + u]) - my_dl[qc]);
                }
                pk[e] = pack2<T>(pr[0], pr[1]);
                dk2[e] = pack2<T>(dr[0], dr[1]);
              }
              const int chunk = c >> 1, g0 = (c & 1) * 4;
#pragma unroll
              for (int u = 0; u < 4; ++u) {
                const uint32_t off = chunk * kChunkBytes + sw128_offset(r, g0 + u);
                *reinterpret_cast<uint4*>(pt_s + off) = make_uint4(pk[4 * u], pk[4 * u + 1], pk[4 * u + 2], pk[4 * u + 3]);
                *reinterpret_cast<uint4*>(ds_s + off) =
                    make_uint4(dk2[4 * u], dk2[4 * u + 1], dk2[4 * u + 2], dk2[4 * u + 3]);
              }
            }
          } else {
#pragma unroll 1
            for (int c = 0; c < 4; ++c) {
              uint32_t sv[32];
              tmem_ld32(rs + c * 32, sv);
              uint32_t pk[16], pfk[16];
#pragma unroll
              for (int e = 0; e < 16; ++e) {
                float pr[2], pf[2];
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                  const int qc = c * 32 + 2 * e + u;
                  float fe;
                  float pe = prob(__uint_as_float(sv[2 * e + u]), my_lse[qc], fe);
                  if (masked && (qc < q_lo || qc >= q_hi)) pe = 0.f;
                  pr[u] = pe;
                  pf[u] = pe * fe;
                }
                pk[e] = pack2<T>(pr[0], pr[1]);
                if constexpr (CAP) pfk[e] = pack2<T>(pf[0], pf[1]);
              }
              const int chunk = c >> 1, g0 = (c & 1) * 4;
#pragma unroll
              for (int u = 0; u < 4; ++u) {
                const uint32_t off = chunk * kChunkBytes + sw128_offset(r, g0 + u);
                *reinterpret_cast<uint4*>(pt_s + off) = make_uint4(pk[4 * u], pk[4 * u + 1], pk[4 * u + 2], pk[4 * u + 3]);
              }
              // With CAP, P^T (1 - tanh^2) waits in TMEM (the dS^T buffer is
              // P^T's own in this plan) for the second pass.
              if constexpr (CAP) tmem_st16(tmem + lane_base + C::T_PF + c * 16, pfk);
            }
            fence_proxy_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&p_full);
            if (!wait_bar(&dp_full, gstep & 1, ctl) || !wait_bar(&pt_read, gstep & 1, ctl)) {
              ok = false;
              break;
            }
            tc_fence_after();
#pragma unroll 1
            for (int c = 0; c < 4; ++c) {
              uint32_t pv[32];
              tmem_ld32(rp + c * 32, pv);
              const int chunk = c >> 1, g0 = (c & 1) * 4;
              uint32_t dk2[16], pfw[16];
              if constexpr (CAP) tmem_ld16(tmem + lane_base + C::T_PF + c * 16, pfw);
#pragma unroll
              for (int u = 0; u < 4; ++u) {
                const uint4 pp = CAP ? make_uint4(pfw[4 * u], pfw[4 * u + 1], pfw[4 * u + 2], pfw[4 * u + 3])
                                     : *reinterpret_cast<const uint4*>(pt_s + chunk * kChunkBytes + sw128_offset(r, g0 + u));
                const uint32_t pw[4] = {pp.x, pp.y, pp.z, pp.w};
#pragma unroll
                for (int e2 = 0; e2 < 4; ++e2) {
                  const int e = 4 * u + e2;
                  float2 pf = unpack2<T>(pw[e2]);
                  const int qc = c * 32 + 2 * e;
                  dk2[e] = pack2<T>(pf.x * (__uint_as_float(pv[2 * e]) - my_dl[qc]),
                                       pf.y * (__uint_as_float(pv[2 * e + 1]) - my_dl[qc + 1]));
                }
              }
#pragma unroll
              for (int u = 0; u < 4; ++u)
                *reinterpret_cast<uint4*>(ds_s + chunk * kChunkBytes + sw128_offset(r, g0 + u)) =
                    make_uint4(dk2[4 * u], dk2[4 * u + 1], dk2[4 * u + 2], dk2[4 * u + 3]);
            }
          }
          fence_proxy_async_smem();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&ds_full);
        }
      }
      if (!ok) break;
      // dK / dV epilogue for this key tile.
      if (!wait_bar(&acc_done, nz & 1, ctl)) break;
      tc_fence_after();
#pragma unroll 1
      for (int c = 0; c < DV / 32; ++c) {
        uint32_t a[32];
        tmem_ld32(tmem + lane_base + C::T_DV + c * 32, a);
        if (valid) {
          uint4* dst = reinterpret_cast<uint4*>(dv_row + c * 32);
#pragma unroll
          for (int u = 0; u < 4; ++u)
            dst[u] = make_uint4(pack2<T>(__uint_as_float(a[8 * u]), __uint_as_float(a[8 * u + 1])),
                                pack2<T>(__uint_as_float(a[8 * u + 2]), __uint_as_float(a[8 * u + 3])),
                                pack2<T>(__uint_as_float(a[8 * u + 4]), __uint_as_float(a[8 * u + 5])),
                                pack2<T>(__uint_as_float(a[8 * u + 6]), __uint_as_float(a[8 * u + 7])));
        }
      }
      const float sc = p.scale;
#pragma unroll 1
      for (int c = 0; c < DQK / 32; ++c) {
        uint32_t a[32];
        tmem_ld32(tmem + lane_base + C::T_DK + c * 32, a);
        if (valid) {
          uint4* dst = reinterpret_cast<uint4*>(dk_row + c * 32);
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
  } else if (warp >= 8) {
    // ------------------------------------------------------------ dQ read-out
    const int wq = warp - 8;
    const uint32_t lane_base = (uint32_t)(32 * wq) << 16;
    uint8_t* stg = smem + C::STG_OFF + wq * 4096;
    uint32_t gstep = 0;
    bool ok = true;
    for (int wi = 0; wi * (int)gridDim.x < total && ok; ++wi) {
      const int w = snake_item(wi);
      if (w >= total) continue;
      const BwdItem t = bwd_decode(p, w);
      if (t.k1 == t.k0) continue;
      {
        for (int k = t.k0; k < t.k1; ++k, ++gstep) {
          const int h = t.hk * G + k / t.nqt, qt = t.qt0 + k % t.nqt;
          if (!wait_bar(&dq_full, gstep & 1, ctl)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t rq = tmem + lane_base + (C::DUAL ? ((gstep & 1) ? C::T_B : C::T_A) : C::T_A);
          const int fq = t.cq0 + qt * kBM + 32 * wq, bq = fq / p.seg.Sq, sq = fq - bq * p.seg.Sq;
#pragma unroll 1
          for (int c = 0; c < DQK / 32; ++c) {
            uint32_t a[32];
            tmem_ld32(rq + c * 32, a);
            if (c > 0) {
              if (lane == 0) bulk_wait_group_read0();
              __syncwarp();
            }
#pragma unroll
            for (int u = 0; u < 8; ++u)
              *reinterpret_cast<uint4*>(stg + sw128_offset(lane, u)) =
                  make_uint4(a[4 * u], a[4 * u + 1], a[4 * u + 2], a[4 * u + 3]);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              tma_reduce_add_4d(&p.tm_dq, stg, c * 32, sq, h, bq);
              bulk_commit_group();
            }
          }
          if (lane == 0) bulk_wait_group_read0();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&dq_free);
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

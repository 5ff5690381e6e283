// bwd_wide.cuh -- attention backward for Dqk = Dv = 512 (sm_103a), one
// four-CTA thread-block cluster per (key tile, KV head).
//   [nemo_automodel.components.attention.ffpa_attention: the FFPA kernel the
//    page routes head_dim = 512 layers to; `_ffpa_dense_bwd`,
//    `_ffpa_varlen_bwd`: gradients from the caller-supplied out/lse]
//
// The dK and dV accumulators of a 128-row key tile at head dim 512 would need
// 1024 TMEM columns, twice what an SM has. The four CTAs of a cluster each own
// one 128-column part r of the head dim -- the slices K_r, V_r, Q_r, dO_r and
// part r of dV, dK and dQ -- and split the 512-wide contractions of S and dP:
//   S_r^T  = K_r Q_r^T,   dP_r^T = V_r dO_r^T        (partial sums over part r)
// CTA r owns the query columns [32r, 32r + 32) of a step. Every CTA stores the
// other CTAs' columns of its partial S^T, then of its partial dP^T, into their
// shared memory (st.async, counted in bytes on the receiver's mbarrier) and
// adds the three partials it receives to its own columns:
//   P^T  = exp2(S^T scale log2 e - lse log2 e),   dS^T = P^T (dP^T - Delta)
// It writes its columns of P^T, as soon as they exist, and then of dS^T
// (16-bit) into all four CTAs' P^T / dS^T buffers, and each CTA runs
//   dV_r += P^T dO_r (once P^T is complete),
//   dK_r += dS^T Q_r,  dQ_r = dS K_r (once dS^T is complete).
// Each of the five products is computed once, and a CTA streams only its
// quarter of Q, dO and V per step (K_r stays for the whole key tile). The
// exchange of S^T overlaps the dP product, the exchange of dP^T the dV
// product, and the next step's S^T product (its Q_r in the buffer this
// step's dO_r leaves after dV) the exchange of dP^T and dS^T.
//
// TMEM: dV_r [0,128) | dK_r [128,256) | S_r^T [256,384) | dP_r^T, then dQ_r [384,512)
// Shared memory: K_r, two buffers that take Q_r and dO_r in turn, P^T (32 KB
// each); the dS^T buffer (32 KB), which holds V_r until the step's dP product
// has read it; X (48 KB), the columns received from the three other CTAs
// (S^T, then dP^T); dQ staging (4 KB per read-out warp). P^T and dS^T are four
// 32-query chunks of 64-byte rows (64-byte swizzle), so CTA r's columns are
// chunk r: one contiguous 8 KB block.
// Warps: 0 TMA producer, 1 MMA issuer, 2 TMEM allocator, 4-7 compute (the
// exchange, P, dS, the dK/dV epilogue), 8-11 dQ read-out (TMA reduce-add).
//
// Signals between the CTAs of a cluster (every wait bounded):
//   rx_s[q]  CTA q has summed the dP^T columns of the previous step: its X
//            may take this step's S^T columns
//   rx_d[q]  CTA q has summed this step's S^T columns: its X may take dP^T
//   recv_full  the three others' columns (48 KB) have landed in X
//   p_full / ds_full  the three others' P^T / dS^T columns (24 KB each) and
//            this CTA's own are in place
// The P^T and dS^T buffers need no signal of their own: a CTA sends its P^T
// (dS^T) columns of a step only once it holds every other CTA's S^T (dP^T)
// columns of that step, each sent after that CTA's S (dP) product of the
// step, which completed after the products that last read its P^T (its V_r,
// then dS^T).
#pragma once

#include <math_constants.h>

#include "bwd.cuh"
#include "cluster.cuh"

namespace psf {

template <int D>
struct BwdWideCfg {
  static constexpr int NP = D / 128;    // column parts = CTAs per cluster
  static constexpr int OWN = kBM / NP;  // query columns a CTA owns per step
  static constexpr int K_OFF = 0;
  // Two 32 KB buffers that take Q_r and dO_r in turn: step g's Q_r in buffer
  // g & 1 and its dO_r in the other, so the next step's Q_r loads as soon as
  // this step's dV product has read dO_r.
  static constexpr int QD_OFF = K_OFF + 2 * kChunkBytes;
  static constexpr int QD_BYTES = 2 * kChunkBytes;
  static constexpr int PT_OFF = QD_OFF + 2 * QD_BYTES;
  static constexpr int DS_OFF = PT_OFF + 2 * kChunkBytes;  // V_r, then dS^T
  static constexpr int X_OFF = DS_OFF + 2 * kChunkBytes;
  static constexpr int SLOT_BYTES = kBN * OWN * 4;  // one sender's columns, fp32
  static constexpr int X_BYTES = (NP - 1) * SLOT_BYTES;
  static constexpr int STG_OFF = X_OFF + X_BYTES;
  static constexpr int COL_BYTES = kBN * OWN * 2;           // one CTA's P^T (or dS^T) columns, 16-bit
  static constexpr int HALF_TX = (NP - 1) * COL_BYTES;      // the three others' columns
  // The barriers the other CTAs signal, at fixed offsets so that one mapped
  // base address per CTA reaches them: recv_full, p_full, ds_full, rx_s[4], rx_d[4].
  static constexpr int BAR_OFF = STG_OFF + 4 * 4096;
  static constexpr int B_RECV = BAR_OFF, B_P = BAR_OFF + 8, B_DS = BAR_OFF + 16, B_RXS = BAR_OFF + 24,
                       B_RXD = BAR_OFF + 56;
  static constexpr int SMEM_BYTES = BAR_OFF + 88 + 1024;
  static constexpr int T_DV = 0, T_DK = 128, T_S = 256, T_DP = 384;  // T_DP: dP^T, then dQ
  static_assert(NP == 4 && OWN == 32, "laid out for a four-CTA cluster");
  static_assert(SMEM_BYTES + 512 <= 232448, "shared memory budget (dynamic + static)");
};

// CAP: logits softcapped (p.softcap > 0); dS carries the cap's 1 - tanh^2.
template <typename T, int D, bool CAP>
__global__ void __cluster_dims__(4, 1, 1) __launch_bounds__(384, 1)
    attn_bwd_wide_kernel(const __grid_constant__ BwdParams p) {
  using C = BwdWideCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

  __shared__ uint64_t k_full, k_empty, qd_full[2], qd_empty[2], v_full, v_free, s_full, s_read, dp_full;
  __shared__ uint64_t dq_full, dq_free, acc_done, acc_free, drain;
  uint64_t& recv_full = *reinterpret_cast<uint64_t*>(smem + C::B_RECV);
  uint64_t& p_full = *reinterpret_cast<uint64_t*>(smem + C::B_P);
  uint64_t& ds_full = *reinterpret_cast<uint64_t*>(smem + C::B_DS);
  uint64_t* rx_s = reinterpret_cast<uint64_t*>(smem + C::B_RXS);
  uint64_t* rx_d = reinterpret_cast<uint64_t*>(smem + C::B_RXD);
  __shared__ uint32_t tmem_base_smem;
  __shared__ int abort_flag;

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int rank = (int)cluster_ctarank();
  const int ncl = (int)cluster_count_x(), cid = (int)cluster_id_x();
  if (threadIdx.x == 0) {
    mbar_init(&k_full, 1);
    mbar_init(&k_empty, 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(&qd_full[b], 1);
      mbar_init(&qd_empty[b], 1);
    }
    mbar_init(&s_read, 4);
    mbar_init(&v_full, 1);
    mbar_init(&v_free, 1);
    mbar_init(&s_full, 1);
    mbar_init(&dp_full, 1);
    mbar_init(&dq_full, 1);
    mbar_init(&dq_free, 4);
    mbar_init(&acc_done, 1);
    mbar_init(&acc_free, 4);
    mbar_init(&drain, 1);
    mbar_init(&recv_full, 1);
    mbar_init(&p_full, 4);
    mbar_init(&ds_full, 4);
    for (int q = 0; q < 4; ++q) {
      mbar_init(&rx_s[q], 4);
      mbar_init(&rx_d[q], 4);
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
  cluster_sync();  // every CTA's barriers exist before any other CTA signals them
  tc_fence_after();
  const uint32_t tmem = tmem_base_smem;
  const Ctl ctl{p.status, p.limit_ns, &abort_flag};
  const int total = (*p.n_items) * p.Hkv;
  const int G = p.Hq / p.Hkv;
  const uint32_t sbase = smem_u32(smem);
  // The four CTAs of a cluster walk the same (key tile, KV head) units: in
  // round i cluster c takes unit i * ncl + c (i even) or i * ncl + ncl - 1 - c.
  auto unit = [&](int i) { return i * ncl + ((i & 1) ? ncl - 1 - cid : cid); };
  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&p.tm_q);
      tma_prefetch_desc(&p.tm_k);
      tma_prefetch_desc(&p.tm_v);
      tma_prefetch_desc(&p.tm_do);
      uint32_t nk = 0, nv = 0, ng = 0, nqd[2] = {0, 0};
      bool ok = true;
      for (int wi = 0; wi * ncl < total && ok; ++wi) {
        const int w = unit(wi);
        if (w >= total) continue;
        const BwdItem t = bwd_decode(p, w);
        if (t.k1 == t.k0) continue;
        const int fk = t.ck0 + t.kt * kBN, bk = fk / p.seg.Sk, sk = fk - bk * p.seg.Sk;
        if (nk > 0 && !wait_bar(&k_empty, (nk - 1) & 1, ctl)) break;
        mbar_arrive_expect_tx(&k_full, 2 * kChunkBytes);
        for (int c = 0; c < 2; ++c)
          tma_load_4d(smem + C::K_OFF + c * kChunkBytes, &p.tm_k, &k_full, rank * 128 + c * 64, sk, t.hk, bk);
        ++nk;
        for (int k = t.k0; k < t.k1; ++k) {
          const int h = t.hk * G + k / t.nqt, qt = t.qt0 + k % t.nqt;
          const int fq = t.cq0 + qt * kBM, bq = fq / p.seg.Sq, sq = fq - bq * p.seg.Sq;
          // Q_r into buffer g & 1 (it held dO_r of step g - 1: free after that
          // step's dV), dO_r into the other (it held Q_r of step g - 1: free
          // after that step's dK).
          const int b0 = ng & 1;
          for (int x = 0; x < 2 && ok; ++x) {
            const int b = b0 ^ x;
            if (ng > 0 && !wait_bar(&qd_empty[b], (ng - 1) & 1, ctl)) {
              ok = false;
              break;
            }
            mbar_arrive_expect_tx(&qd_full[b], C::QD_BYTES);
            for (int c = 0; c < 2; ++c)
              tma_load_4d(smem + C::QD_OFF + b * C::QD_BYTES + c * kChunkBytes, x == 0 ? &p.tm_q : &p.tm_do,
                          &qd_full[b], rank * 128 + c * 64, sq, h, bq);
            ++nqd[b];
          }
          if (!ok) break;
          ++ng;
          // V_r of the step goes into the dS^T buffer once the previous step's dQ product has read it.
          if (nv > 0 && !wait_bar(&v_free, (nv - 1) & 1, ctl)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&v_full, 2 * kChunkBytes);
          for (int c = 0; c < 2; ++c)
            tma_load_4d(smem + C::DS_OFF + c * kChunkBytes, &p.tm_v, &v_full, rank * 128 + c * 64, sk, t.hk, bk);
          ++nv;
        }
      }
      // Loads still in flight after an abort land before the CTA leaves.
      if (nk > 0) wait_bar_drain(&k_full, (nk - 1) & 1, p.limit_ns);
      if (nv > 0) wait_bar_drain(&v_full, (nv - 1) & 1, p.limit_ns);
      for (int b = 0; b < 2; ++b)
        if (nqd[b] > 0) wait_bar_drain(&qd_full[b], (nqd[b] - 1) & 1, p.limit_ns);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t id_sq = idesc_f32acc<T>(128, 128, 0, 0);
      constexpr uint32_t id_part = idesc_f32acc<T>(128, 128, 0, 1);  // dV, dK parts: B MN-major
      constexpr uint32_t id_dq = idesc_f32acc<T>(128, 128, 1, 1);    // dQ part: A (dS) M-major
      const uint32_t k_a = sbase + C::K_OFF, qd_a = sbase + C::QD_OFF;
      const uint32_t pt_a = sbase + C::PT_OFF, ds_a = sbase + C::DS_OFF;  // ds_a: V_r first
      // S_r^T = K_r Q_r^T (128-wide contraction) from the buffer at q_a
      auto issue_s = [&](uint32_t q_a) {
#pragma unroll
        for (int c = 0; c < 2; ++c)
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_ss(tmem + C::T_S, sdesc_sw128(k_a + c * kChunkBytes + kk * 32, 16, 1024),
                   sdesc_sw128(q_a + c * kChunkBytes + kk * 32, 16, 1024), id_sq, (c | kk) != 0);
        mma_commit(&s_full);
      };
      uint32_t ni = 0, gstep = 0;
      bool ok = true;
      for (int wi = 0; wi * ncl < total && ok; ++wi) {
        const int w = unit(wi);
        if (w >= total) continue;
        const BwdItem t = bwd_decode(p, w);
        if (t.k1 == t.k0) continue;
        if (!wait_bar(&k_full, ni & 1, ctl)) break;
        bool s_issued = false;  // this step's S^T already issued during the previous step
        for (int k = t.k0; k < t.k1; ++k, ++gstep) {
          const int b = gstep & 1;
          const uint32_t q_a = qd_a + b * C::QD_BYTES, do_a = qd_a + (b ^ 1) * C::QD_BYTES;
          if (!s_issued) {
            if (!wait_bar(&qd_full[b], gstep & 1, ctl) || (gstep > 0 && !wait_bar(&s_read, (gstep - 1) & 1, ctl))) {
              ok = false;
              break;
            }
            tc_fence_after();
            issue_s(q_a);
          }
          s_issued = false;
          // dP^T's columns hold the previous step's dQ until it has been read out.
          if (!wait_bar(&v_full, gstep & 1, ctl) || !wait_bar(&qd_full[b ^ 1], gstep & 1, ctl) ||
              (gstep > 0 && !wait_bar(&dq_free, (gstep - 1) & 1, ctl))) {
            ok = false;
            break;
          }
          tc_fence_after();
          // dP_r^T = V_r dO_r^T
#pragma unroll
          for (int c = 0; c < 2; ++c)
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              mma_ss(tmem + C::T_DP, sdesc_sw128(ds_a + c * kChunkBytes + kk * 32, 16, 1024),
                     sdesc_sw128(do_a + c * kChunkBytes + kk * 32, 16, 1024), id_sq, (c | kk) != 0);
          mma_commit(&dp_full);
          const bool first = k == t.k0;
          if ((first && ni > 0 && !wait_bar(&acc_free, (ni - 1) & 1, ctl)) || !wait_bar_cl(&p_full, gstep & 1, ctl)) {
            ok = false;
            break;
          }
          // The other CTAs' columns arrived by st.async: make them visible to the tensor core's reads.
          fence_proxy_async_smem();
          tc_fence_after();
          // dV_r += P^T dO_r (B: the two 64-column chunks of dO_r, kChunkBytes apart)
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            mma_ss(tmem + C::T_DV, sdesc_sw64(pt_a + (kk >> 1) * C::COL_BYTES + (kk & 1) * 32, 16, 512),
                   sdesc_sw128(do_a + kk * 2048, kChunkBytes, 1024), id_part, !(first && kk == 0));
          mma_commit(&qd_empty[b ^ 1]);
          // The next step's S^T (same key tile) as soon as its Q_r has landed
          // and this step's S^T has been read out, ahead of dK and dQ.
          if (k + 1 < t.k1) {
            if (!wait_bar(&qd_full[b ^ 1], (gstep + 1) & 1, ctl) || !wait_bar(&s_read, gstep & 1, ctl)) {
              ok = false;
              break;
            }
            tc_fence_after();
            issue_s(do_a);
            s_issued = true;
          }
          if (!wait_bar_cl(&ds_full, gstep & 1, ctl)) {
            ok = false;
            break;
          }
          fence_proxy_async_smem();
          tc_fence_after();
          // dK_r += dS^T Q_r
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            mma_ss(tmem + C::T_DK, sdesc_sw64(ds_a + (kk >> 1) * C::COL_BYTES + (kk & 1) * 32, 16, 512),
                   sdesc_sw128(q_a + kk * 2048, kChunkBytes, 1024), id_part, !(first && kk == 0));
          mma_commit(&qd_empty[b]);
          // dQ_r = dS K_r, into the dP^T columns (already read out)
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            mma_ss(tmem + C::T_DP, sdesc_sw64(ds_a + kk * 1024, C::COL_BYTES, 512),
                   sdesc_sw128(k_a + kk * 2048, kChunkBytes, 1024), id_dq, kk > 0);
          mma_commit(&dq_full);
          mma_commit(&v_free);
        }
        if (!ok) break;
        mma_commit(&acc_done);
        mma_commit(&k_empty);
        ++ni;
      }
      mma_commit(&drain);
      wait_bar_drain(&drain, 0, p.limit_ns);
    }
  } else if (warp >= 4 && warp < 8) {
    // ------------------------------------------------------------ compute warpgroup
    const int wq = warp - 4;
    const int r = threadIdx.x - 128;  // key row of the tile (TMEM lane)
    const uint32_t lane_base = (uint32_t)(32 * wq) << 16;
    const int c0 = rank * C::OWN;  // this CTA's query columns [c0, c0 + 32)
    const float sl2 = p.scale_log2;
    const float cap_c2 = CAP ? p.softcap * 1.4426950408889634f : 0.f;
    const float cap_k1 = CAP ? 2.f * sl2 / p.softcap : 0.f, cap_ic2 = CAP ? 1.f / cap_c2 : 0.f;
    // Shared-memory base of the other CTAs, in the order rank + 1, rank + 2,
    // rank + 3; this CTA's columns go to slot 2 - i of the i-th one's X.
    uint32_t pbase[3];
    for (int i = 0; i < 3; ++i) pbase[i] = mapa_shared(sbase, (uint32_t)(rank + 1 + i) & 3u);
    // A slot holds granule u (four consecutive columns) of row r at byte
    // (u * 128 + r) * 16, so each store instruction of a warp covers 512
    // contiguous bytes of the receiver's slot.
    auto px = [&](int i) { return pbase[i] + C::X_OFF + (2 - i) * C::SLOT_BYTES + r * 16; };
    const uint32_t xrow = sbase + C::X_OFF + r * 16;  // this row of slot 0 (slots SLOT_BYTES apart)
    // Granule u (8 columns) of row r of this CTA's chunk of P^T / dS^T (64-byte swizzle).
    auto col_off = [&](int u) { return (uint32_t)(rank * C::COL_BYTES + r * 64 + ((u ^ ((r >> 1) & 3)) << 4)); };
    // Columns 32 q .. 32 q + 31 of a partial sum in TMEM, to the q-th CTA's X.
    auto send_cols = [&](int i, uint32_t tcol) {
      uint32_t v[32];
      tmem_ld32(tmem + lane_base + tcol, v);
#pragma unroll
      for (int u = 0; u < 8; ++u)
        st_async_v4(px(i) + u * (kBN * 16), make_uint4(v[4 * u], v[4 * u + 1], v[4 * u + 2], v[4 * u + 3]),
                    pbase[i] + C::B_RECV);
    };
    auto add_recv = [&](float (&a)[32]) {
#pragma unroll
      for (int s = 0; s < 3; ++s)
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const uint4 x = lds_v4(xrow + s * C::SLOT_BYTES + u * (kBN * 16));
          a[4 * u] += __uint_as_float(x.x);
          a[4 * u + 1] += __uint_as_float(x.y);
          a[4 * u + 2] += __uint_as_float(x.z);
          a[4 * u + 3] += __uint_as_float(x.w);
        }
    };
    // This CTA's 16-bit columns (16 packed pairs) into its chunk of the
    // buffer at `off0` of all four CTAs: the warp writes its 32 rows (2 KB,
    // contiguous) here, reads them back four 512-byte rows at a time, arrives
    // on the local barrier at `bar_off` (warp 4 with the three others' bytes)
    // and only then stores them into the other CTAs, so that the arrival does
    // not wait for those stores.
    auto share_cols = [&](const uint32_t (&pk)[16], int off0, int bar_off) {
#pragma unroll
      for (int u = 0; u < 4; ++u)
        *reinterpret_cast<uint4*>(smem + off0 + col_off(u)) =
            make_uint4(pk[4 * u], pk[4 * u + 1], pk[4 * u + 2], pk[4 * u + 3]);
      __syncwarp();
      const uint32_t rows = off0 + rank * C::COL_BYTES + wq * 2048;
      uint4 v[4];
#pragma unroll
      for (int m = 0; m < 4; ++m) v[m] = lds_v4(sbase + rows + m * 512 + lane * 16);
      // The local copy is read by this CTA's tensor core.
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        uint64_t* b = reinterpret_cast<uint64_t*>(smem + bar_off);
        if (wq == 0)
          mbar_arrive_expect_tx(b, C::HALF_TX);
        else
          mbar_arrive(b);
      }
#pragma unroll
      for (int m = 0; m < 4; ++m)
#pragma unroll
        for (int i = 0; i < 3; ++i)
          st_async_v4(pbase[i] + rows + m * 512 + lane * 16, v[m], pbase[i] + bar_off);
    };
    // Every lane of the warp: a bounded wait by lane 0 on barrier `bar`.
    auto warp_wait_cl = [&](uint64_t* bar, uint32_t parity) {
      bool good = true;
      if (lane == 0) good = wait_bar_cl(bar, parity, ctl);
      return __shfl_sync(0xffffffffu, good, 0) != 0;
    };
    uint32_t ni = 0, gstep = 0;
    bool ok = true;
    for (int wi = 0; wi * ncl < total && ok; ++wi) {
      const int w = unit(wi);
      if (w >= total) continue;
      const BwdItem t = bwd_decode(p, w);
      const int j = t.kt * kBN + r;
      const bool valid = j < t.n;
      const int fk = t.ck0 + j, bk = fk / p.seg.Sk, sk = fk - bk * p.seg.Sk;
      T* dk_row = static_cast<T*>(p.dk) + bk * p.k_sb + (int64_t)sk * p.k_ss + t.hk * p.k_sh + rank * 128;
      T* dv_row = static_cast<T*>(p.dv) + bk * p.v_sb + (int64_t)sk * p.v_ss + t.hk * p.v_sh + rank * 128;
      if (t.k1 == t.k0) {
        if (valid) {
          for (int c = 0; c < 16; ++c) {
            reinterpret_cast<uint4*>(dk_row)[c] = make_uint4(0, 0, 0, 0);
            reinterpret_cast<uint4*>(dv_row)[c] = make_uint4(0, 0, 0, 0);
          }
        }
        continue;
      }
      const int delta = t.n - t.m;
      // lse and Delta of query column c0 + lane, loaded one step ahead and
      // left in flight until the step reads them (-inf / 0 outside the segment).
      auto fetch_col = [&](int k, float& lv, float& dv) {
        const int h = t.hk * G + k / t.nqt, i0 = (t.qt0 + k % t.nqt) * kBM;
        const int qc = c0 + lane;
        const int f = t.cq0 + i0 + qc;
        const bool in = i0 + qc < t.m && f < p.q_rows;
        const int fs = in ? f : 0;
        const int bq = fs / p.seg.Sq, sq = fs - bq * p.seg.Sq;
        lv = -CUDART_INF_F;
        dv = 0.f;
        ldg_pred_f32(lv, p.lse + bq * p.l_sb + h * p.l_sh + sq, in);
        ldg_pred_f32(dv, p.delta + (int64_t)h * p.q_rows + fs, in);
      };
      float rlv, rdv;
      fetch_col(t.k0, rlv, rdv);
      for (int k = t.k0; k < t.k1; ++k, ++gstep) {
        const int i0 = (t.qt0 + k % t.nqt) * kBM;
        int q_lo = p.seg.causal ? j - delta - i0 : -0x40000000;
        int q_hi = t.m - i0;
        if (p.seg.window > 0) q_hi = min(q_hi, j - delta + p.seg.window - i0);
        if (!valid) q_lo = q_hi = 0;
        const bool masked = q_lo > c0 || q_hi < c0 + C::OWN;
        const float l2 = rlv == -CUDART_INF_F ? CUDART_INF_F : rlv * 1.4426950408889634f;
        const float dl = rdv;
        if (k + 1 < t.k1) fetch_col(k + 1, rlv, rdv);
        if (!wait_bar(&s_full, gstep & 1, ctl)) {
          ok = false;
          break;
        }
        tc_fence_after();
        // Arm the receive barrier for this step's S^T columns before this
        // thread's own stores, so that the arming does not wait for them.
        if (wq == 0 && lane == 0) mbar_arrive_expect_tx(&recv_full, C::X_BYTES);
        // ---- S^T: the other CTAs' columns of the partial sum go to them
        bool good = true;
        for (int i = 0; i < 3 && good; ++i) {
          const int q = (rank + 1 + i) & 3;
          if (gstep > 0 && !(good = warp_wait_cl(&rx_s[q], (gstep - 1) & 1))) break;
          send_cols(i, C::T_S + 32 * q);
        }
        if (!good) {
          ok = false;
          break;
        }
        float acc[32];
        {
          uint32_t v[32];
          tmem_ld32(tmem + lane_base + C::T_S + c0, v);
#pragma unroll
          for (int e = 0; e < 32; ++e) acc[e] = __uint_as_float(v[e]);
        }
        // S^T is read out: the next step's S^T may take its columns.
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&s_read);
        if (!wait_bar_cl(&recv_full, 0, ctl)) {
          ok = false;
          break;
        }
        // The S^T phase is complete: arm the barrier for the dP^T columns.
        if (wq == 0 && lane == 0) mbar_arrive_expect_tx(&recv_full, C::X_BYTES);
        add_recv(acc);
        // P (16-bit, packed, for P^T) and P (1 - tanh^2) in acc (for dS)
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          float pr[2];
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            const int jj = 2 * e + u, qc = c0 + jj;
            const float l2j = __shfl_sync(0xffffffffu, l2, jj);
            float pe, fe = 1.f;
            if constexpr (CAP) {
              const float y = softcap_log2(acc[jj], cap_k1, cap_c2);
              const float tt = y * cap_ic2;
              fe = fmaf(-tt, tt, 1.f);
              pe = ex2_approx(y - l2j);
            } else {
              pe = ex2_approx(fmaf(acc[jj], sl2, -l2j));
            }
            if (masked && (qc < q_lo || qc >= q_hi)) pe = 0.f;
            pr[u] = pe;
            acc[jj] = pe * fe;
          }
          pk[e] = pack2<T>(pr[0], pr[1]);
        }
        // This warp's rows of X are summed: the others may send dP^T columns.
        // (A relaxed arrive: it only releases slots whose values are already
        // in registers, and must not wait for this thread's S^T stores.)
        __syncwarp();
        if (lane == 0)
          for (int i = 0; i < 3; ++i) mbar_arrive_remote_relaxed(pbase[i] + C::B_RXD + 8 * rank);
        // ---- P^T columns to all four CTAs (the dV product can start); the dP
        // product, whose dO_r and V_r load only after the previous step's dK
        // and dQ, is usually still running
        share_cols(pk, C::PT_OFF, C::B_P);
        // ---- dP^T: the same exchange as S^T
        if (!wait_bar(&dp_full, gstep & 1, ctl)) {
          ok = false;
          break;
        }
        tc_fence_after();
        for (int i = 0; i < 3 && good; ++i) {
          const int q = (rank + 1 + i) & 3;
          if (!(good = warp_wait_cl(&rx_d[q], gstep & 1))) break;
          send_cols(i, C::T_DP + 32 * q);
        }
        if (!good) {
          ok = false;
          break;
        }
        float dpa[32];
        {
          uint32_t v[32];
          tmem_ld32(tmem + lane_base + C::T_DP + c0, v);
#pragma unroll
          for (int e = 0; e < 32; ++e) dpa[e] = __uint_as_float(v[e]);
        }
        // Last TMEM read of the step: the MMA may overwrite S^T and dP^T once
        // the ds_full arrival below is seen.
        tc_fence_before();
        if (!wait_bar_cl(&recv_full, 1, ctl)) {
          ok = false;
          break;
        }
        add_recv(dpa);
        // This warp's rows of X are summed: the others may send the next step's S^T columns.
        __syncwarp();
        if (lane == 0)
          for (int i = 0; i < 3; ++i) mbar_arrive_remote_relaxed(pbase[i] + C::B_RXS + 8 * rank);
        uint32_t dk2[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const float d0 = acc[2 * e] * (dpa[2 * e] - __shfl_sync(0xffffffffu, dl, 2 * e));
          const float d1 = acc[2 * e + 1] * (dpa[2 * e + 1] - __shfl_sync(0xffffffffu, dl, 2 * e + 1));
          dk2[e] = pack2<T>(d0, d1);
        }
        // ---- dS^T columns to all four CTAs (dK and dQ can start)
        share_cols(dk2, C::DS_OFF, C::B_DS);
      }
      if (!ok) break;
      if (!wait_bar(&acc_done, ni & 1, ctl)) break;
      tc_fence_after();
      const float sc = p.scale;
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        uint32_t a[32], b[32];
        tmem_ld32(tmem + lane_base + C::T_DV + c * 32, a);
        tmem_ld32(tmem + lane_base + C::T_DK + c * 32, b);
        if (valid) {
          uint4* dv_dst = reinterpret_cast<uint4*>(dv_row + c * 32);
          uint4* dk_dst = reinterpret_cast<uint4*>(dk_row + c * 32);
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            dv_dst[u] = make_uint4(pack2<T>(__uint_as_float(a[8 * u]), __uint_as_float(a[8 * u + 1])),
                                   pack2<T>(__uint_as_float(a[8 * u + 2]), __uint_as_float(a[8 * u + 3])),
                                   pack2<T>(__uint_as_float(a[8 * u + 4]), __uint_as_float(a[8 * u + 5])),
                                   pack2<T>(__uint_as_float(a[8 * u + 6]), __uint_as_float(a[8 * u + 7])));
            dk_dst[u] = make_uint4(pack2<T>(__uint_as_float(b[8 * u]) * sc, __uint_as_float(b[8 * u + 1]) * sc),
                                   pack2<T>(__uint_as_float(b[8 * u + 2]) * sc, __uint_as_float(b[8 * u + 3]) * sc),
                                   pack2<T>(__uint_as_float(b[8 * u + 4]) * sc, __uint_as_float(b[8 * u + 5]) * sc),
                                   pack2<T>(__uint_as_float(b[8 * u + 6]) * sc, __uint_as_float(b[8 * u + 7]) * sc));
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_free);
      ++ni;
    }
  } else if (warp >= 8) {
    // ------------------------------------------------------------ dQ read-out
    const int wq = warp - 8;
    const uint32_t lane_base = (uint32_t)(32 * wq) << 16;
    uint8_t* box = smem + C::STG_OFF + wq * 4096;
    uint32_t gstep = 0;
    bool ok = true;
    for (int wi = 0; wi * ncl < total && ok; ++wi) {
      const int w = unit(wi);
      if (w >= total) continue;
      const BwdItem t = bwd_decode(p, w);
      if (t.k1 == t.k0) continue;
      for (int k = t.k0; k < t.k1; ++k, ++gstep) {
        const int h = t.hk * G + k / t.nqt, qt = t.qt0 + k % t.nqt;
        if (!wait_bar(&dq_full, gstep & 1, ctl)) {
          ok = false;
          break;
        }
        tc_fence_after();
        uint32_t a[4][32];
#pragma unroll
        for (int c = 0; c < 4; ++c) tmem_ld32(tmem + lane_base + C::T_DP + c * 32, a[c]);
        // dQ is in registers: the next step's dP^T may take its columns.
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&dq_free);
        const int fq = t.cq0 + qt * kBM + 32 * wq, bq = fq / p.seg.Sq, sq = fq - bq * p.seg.Sq;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          if (lane == 0) bulk_wait_group_read0();
          __syncwarp();
#pragma unroll
          for (int u = 0; u < 8; ++u)
            *reinterpret_cast<uint4*>(box + sw128_offset(lane, u)) =
                make_uint4(a[c][4 * u], a[c][4 * u + 1], a[c][4 * u + 2], a[c][4 * u + 3]);
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_reduce_add_4d(&p.tm_dq, box, rank * 128 + c * 32, sq, h, bq);
            bulk_commit_group();
          }
        }
      }
    }
    if (lane == 0) bulk_wait_group0();
  }
  tc_fence_before();
  __syncthreads();
  // No CTA leaves while another may still store into or signal its shared memory.
  cluster_sync();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace psf

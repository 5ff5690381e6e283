// bwd_wide.cuh -- attention backward for Dqk = Dv = 512 (sm_103a).
//   [nemo_automodel.components.attention.ffpa_attention: the FFPA kernel the
//    page routes head_dim = 512 layers to; `_ffpa_dense_bwd`,
//    `_ffpa_varlen_bwd`: gradients from the caller-supplied out/lse]
//
// The dK and dV accumulators of a 128-row key tile at head dim 512 would need
// 1024 TMEM columns, twice what an SM has. Each CTA therefore owns one
// 128-column slice ("part") of dV, dK and dQ and recomputes the full S^T and
// dP^T for it:
//   TMEM  dV part [0,128) | dK part [128,256) | S^T, then dQ part [256,384) | dP^T [384,512)
//   per step (query head of the group x query tile):
//     S^T  = sum_c K_c Q_c^T over eight 64-column chunks c
//     dP^T = sum_c V_c dO_c^T
//     P^T, dS^T -> shared memory (bf16, 128-byte swizzled)
//     dV_part += P^T dO_part, dK_part += dS^T Q_part, dQ_part = dS K_part
// K, Q, V and dO all stream through one ring of 16 KB chunks in the order the
// MMA warp consumes them; nothing but P^T and dS^T stays in shared memory.
// Roles as in bwd.cuh: warp 0 producer, warp 1 MMA, warp 2 TMEM, warps 4-7
// compute (+ dK/dV epilogue), warps 8-11 dQ read-out (TMA reduce-add).
#pragma once

#include <math_constants.h>

#include "bwd.cuh"

namespace psf {

template <int D>
struct BwdWideCfg {
  static constexpr int NCH = D / 64;   // chunks per full operand row
  static constexpr int NP = D / 128;   // column parts
  static constexpr int NST = 8;        // ring stages
  static constexpr int RING_OFF = 0;
  static constexpr int PT_OFF = RING_OFF + NST * kChunkBytes;  // P^T; dQ staging after the dQ MMA
  static constexpr int DS_OFF = PT_OFF + 2 * kChunkBytes;
  static constexpr int ROWV_OFF = DS_OFF + 2 * kChunkBytes;
  static constexpr int SMEM_BYTES = ROWV_OFF + 2 * 4 * 128 * 4 + 1024;
  static constexpr int T_DV = 0, T_DK = 128, T_S = 256, T_DP = 384;
  static constexpr int CHUNKS_PER_STEP = 4 * NCH + 6;
  static_assert(SMEM_BYTES <= 232448, "shared memory budget");
};

// CAP: logits softcapped (p.softcap > 0); dS carries the cap's 1 - tanh^2.
template <typename T, int D, bool CAP>
__global__ void __launch_bounds__(384, 1) attn_bwd_wide_kernel(const __grid_constant__ BwdParams p) {
  using C = BwdWideCfg<D>;
  constexpr int NST = C::NST;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  float* lse_s = reinterpret_cast<float*>(smem + C::ROWV_OFF);
  float* dl_s = lse_s + 4 * 128;

  __shared__ uint64_t ring_full[NST], ring_empty[NST];
  __shared__ uint64_t s_full, dp_full, ds_full, ds_free, dq_full, dq_free, acc_done, acc_free, drain;
  __shared__ uint32_t tmem_base_smem;
  __shared__ int abort_flag;

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  if (threadIdx.x == 0) {
    for (int i = 0; i < NST; ++i) {
      mbar_init(&ring_full[i], 1);
      mbar_init(&ring_empty[i], 1);
    }
    mbar_init(&s_full, 1);
    mbar_init(&dp_full, 1);
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
  const int per_item = p.Hkv * C::NP;
  const int total = (*p.n_items) * per_item;
  const int G = p.Hq / p.Hkv;
  const uint32_t sbase = smem_u32(smem);

  // Work w -> (key tile item, KV head, column part).
  auto decode = [&](int w, int& part) {
    const int item = w / per_item;
    const int rem = w - item * per_item;
    part = rem % C::NP;
    return bwd_decode(p, item * p.Hkv + rem / C::NP);
  };

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&p.tm_q);
      tma_prefetch_desc(&p.tm_k);
      tma_prefetch_desc(&p.tm_v);
      tma_prefetch_desc(&p.tm_do);
      uint32_t it = 0;
      bool ok = true;
      auto load = [&](const CUtensorMap* map, int c0, int row, int h, int b) -> bool {
        const int st = it % NST;
        if (!wait_bar(&ring_empty[st], ((it / NST) & 1) ^ 1, ctl)) return false;
        mbar_arrive_expect_tx(&ring_full[st], kChunkBytes);
        tma_load_4d(smem + C::RING_OFF + st * kChunkBytes, map, &ring_full[st], c0, row, h, b);
        ++it;
        return true;
      };
      for (int wi = 0; wi * (int)gridDim.x < total && ok; ++wi) {
        const int w = snake_item(wi);
        if (w >= total) continue;
        int part;
        const BwdItem t = decode(w, part);
        if (t.k1 == t.k0) continue;
        const int fk = t.ck0 + t.kt * kBN, bk = fk / p.seg.Sk, sk = fk - bk * p.seg.Sk;
        {
          for (int k = t.k0; k < t.k1 && ok; ++k) {
            const int h = t.hk * G + k / t.nqt, qt = t.qt0 + k % t.nqt;
            const int fq = t.cq0 + qt * kBM, bq = fq / p.seg.Sq, sq = fq - bq * p.seg.Sq;
            for (int c = 0; c < C::NCH && ok; ++c) {
              ok = load(&p.tm_k, c * 64, sk, t.hk, bk) && load(&p.tm_q, c * 64, sq, h, bq);
            }
            for (int c = 0; c < C::NCH && ok; ++c) {
              ok = load(&p.tm_v, c * 64, sk, t.hk, bk) && load(&p.tm_do, c * 64, sq, h, bq);
            }
            for (int c = 0; c < 2 && ok; ++c) ok = load(&p.tm_do, part * 128 + c * 64, sq, h, bq);
            for (int c = 0; c < 2 && ok; ++c) ok = load(&p.tm_q, part * 128 + c * 64, sq, h, bq);
            for (int c = 0; c < 2 && ok; ++c) ok = load(&p.tm_k, part * 128 + c * 64, sk, t.hk, bk);
          }
        }
      }
      for (uint32_t i = it > (uint32_t)NST ? it - NST : 0; i < it; ++i)
        wait_bar_drain(&ring_full[i % NST], (i / NST) & 1, p.limit_ns);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t id_sq = idesc_f32acc<T>(128, 128, 0, 0);
      constexpr uint32_t id_part64 = idesc_f32acc<T>(128, 64, 0, 1);  // dV, dK parts: B MN-major, N = 64
      constexpr uint32_t id_dq64 = idesc_f32acc<T>(128, 64, 1, 1);         // dQ part: A (dS) M-major
      const uint32_t ring = sbase + C::RING_OFF, pt_a = sbase + C::PT_OFF, ds_a = sbase + C::DS_OFF;
      uint32_t it = 0, nz = 0, gstep = 0;
      bool ok = true;
      auto take = [&](uint32_t& addr) -> bool {
        const int st = it % NST;
        if (!wait_bar(&ring_full[st], (it / NST) & 1, ctl)) return false;
        tc_fence_after();
        addr = ring + st * kChunkBytes;
        return true;
      };
      auto give = [&]() {
        mma_commit(&ring_empty[it % NST]);
        ++it;
      };
      for (int wi = 0; wi * (int)gridDim.x < total && ok; ++wi) {
        const int w = snake_item(wi);
        if (w >= total) continue;
        int part;
        const BwdItem t = decode(w, part);
        if (t.k1 == t.k0) continue;
        if (nz > 0 && !wait_bar(&acc_free, (nz - 1) & 1, ctl)) break;
        for (int k = t.k0; k < t.k1 && ok; ++k, ++gstep) {
          if (gstep > 0 && !wait_bar(&dq_free, (gstep - 1) & 1, ctl)) {
            ok = false;
            break;
          }
          tc_fence_after();
          // S^T = sum_c K_c Q_c^T
          for (int c = 0; c < C::NCH && ok; ++c) {
            uint32_t ka, qa;
            if (!take(ka)) { ok = false; break; }
            const int st_k = it % NST;
            ++it;
            if (!take(qa)) { ok = false; break; }
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              mma_ss(tmem + C::T_S, sdesc_sw128(ka + kk * 32, 16, 1024), sdesc_sw128(qa + kk * 32, 16, 1024), id_sq,
                     (c | kk) != 0);
            mma_commit(&ring_empty[st_k]);
            give();
          }
          if (!ok) break;
          mma_commit(&s_full);
          // dP^T = sum_c V_c dO_c^T
          for (int c = 0; c < C::NCH && ok; ++c) {
            uint32_t va, da;
            if (!take(va)) { ok = false; break; }
            const int st_v = it % NST;
            ++it;
            if (!take(da)) { ok = false; break; }
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              mma_ss(tmem + C::T_DP, sdesc_sw128(va + kk * 32, 16, 1024), sdesc_sw128(da + kk * 32, 16, 1024), id_sq,
                     (c | kk) != 0);
            mma_commit(&ring_empty[st_v]);
            give();
          }
          if (!ok) break;
          mma_commit(&dp_full);
          if (!wait_bar(&ds_full, gstep & 1, ctl)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t first = (k == t.k0) ? 1u : 0u;
          // dV_part += P^T dO_part (two 64-column halves)
          for (int hh = 0; hh < 2 && ok; ++hh) {
            uint32_t da;
            if (!take(da)) { ok = false; break; }
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
              mma_ss(tmem + C::T_DV + hh * 64, sdesc_sw128(pt_a + (kk >> 2) * kChunkBytes + (kk & 3) * 32, 16, 1024),
                     sdesc_sw128(da + kk * 2048, kChunkBytes, 1024), id_part64, !(first && kk == 0));
            give();
          }
          // dK_part += dS^T Q_part
          for (int hh = 0; hh < 2 && ok; ++hh) {
            uint32_t qa;
            if (!take(qa)) { ok = false; break; }
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
              mma_ss(tmem + C::T_DK + hh * 64, sdesc_sw128(ds_a + (kk >> 2) * kChunkBytes + (kk & 3) * 32, 16, 1024),
                     sdesc_sw128(qa + kk * 2048, kChunkBytes, 1024), id_part64, !(first && kk == 0));
            give();
          }
          // dQ_part = dS K_part, into the S^T columns (already consumed)
          for (int hh = 0; hh < 2 && ok; ++hh) {
            uint32_t ka;
            if (!take(ka)) { ok = false; break; }
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
              mma_ss(tmem + C::T_S + hh * 64, sdesc_sw128(ds_a + kk * 2048, kChunkBytes, 1024),
                     sdesc_sw128(ka + kk * 2048, kChunkBytes, 1024), id_dq64, kk > 0);
            give();
          }
          if (!ok) break;
          mma_commit(&ds_free);
          mma_commit(&dq_full);
        }
        if (!ok) break;
        mma_commit(&acc_done);
        ++nz;
      }
      mma_commit(&drain);
      wait_bar_drain(&drain, 0, p.limit_ns);
    }
  } else if (warp >= 4 && warp < 8) {
    // ------------------------------------------------------------ compute warpgroup
    const int wq = warp - 4;
    const int r = threadIdx.x - 128;
    const uint32_t lane_base = (uint32_t)(32 * wq) << 16;
    float* my_lse = lse_s + wq * 128;
    float* my_dl = dl_s + wq * 128;
    uint8_t* pt_s = smem + C::PT_OFF;
    uint8_t* ds_s = smem + C::DS_OFF;
    const float sl2 = p.scale_log2;
    const float cap_c2 = CAP ? p.softcap * 1.4426950408889634f : 0.f;
    const float cap_k1 = CAP ? 2.f * sl2 / p.softcap : 0.f, cap_ic2 = CAP ? 1.f / cap_c2 : 0.f;
    uint32_t nz = 0, gstep = 0;
    bool ok = true;
    for (int wi = 0; wi * (int)gridDim.x < total && ok; ++wi) {
      const int w = snake_item(wi);
      if (w >= total) continue;
      int part;
      const BwdItem t = decode(w, part);
      const int j = t.kt * kBN + r;
      const bool valid = j < t.n;
      const int fk = t.ck0 + j, bk = fk / p.seg.Sk, sk = fk - bk * p.seg.Sk;
      T* dk_row = static_cast<T*>(p.dk) + bk * p.k_sb + (int64_t)sk * p.k_ss + t.hk * p.k_sh + part * 128;
      T* dv_row = static_cast<T*>(p.dv) + bk * p.v_sb + (int64_t)sk * p.v_ss + t.hk * p.v_sh + part * 128;
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
          if (!wait_bar(&s_full, gstep & 1, ctl) || !wait_bar(&dp_full, gstep & 1, ctl) ||
              (gstep > 0 && !wait_bar(&ds_free, (gstep - 1) & 1, ctl))) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll 1
          for (int c = 0; c < 4; ++c) {
            uint32_t sv[32], pv[32];
            tmem_ld32(tmem + lane_base + C::T_S + c * 32, sv);
            tmem_ld32(tmem + lane_base + C::T_DP + c * 32, pv);
            uint32_t pk[16], dk2[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              float pr[2], dr[2];
#pragma unroll
              for (int u = 0; u < 2; ++u) {
                const int qc = c * 32 + 2 * e + u;
                float pe, fe = 1.f;
                if constexpr (CAP) {
                  const float y = softcap_log2(__uint_as_float(sv[2 * e + u]), cap_k1, cap_c2);
                  const float tt = y * cap_ic2;
                  fe = fmaf(-tt, tt, 1.f);
                  pe = ex2_approx(y - my_lse[qc]);
                } else {
                  pe = ex2_approx(fmaf(__uint_as_float(sv[2 * e + u]), sl2, -my_lse[qc]));
                }
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
              *reinterpret_cast<uint4*>(ds_s + off) = make_uint4(dk2[4 * u], dk2[4 * u + 1], dk2[4 * u + 2], dk2[4 * u + 3]);
            }
          }
          fence_proxy_async_smem();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&ds_full);
        }
      }
      if (!ok) break;
      if (!wait_bar(&acc_done, nz & 1, ctl)) break;
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
      ++nz;
    }
  } else if (warp >= 8) {
    // ------------------------------------------------------------ dQ read-out
    const int wq = warp - 8;
    const uint32_t lane_base = (uint32_t)(32 * wq) << 16;
    uint8_t* stg = smem + C::PT_OFF + wq * 8192;
    uint32_t gstep = 0;
    bool ok = true;
    for (int wi = 0; wi * (int)gridDim.x < total && ok; ++wi) {
      const int w = snake_item(wi);
      if (w >= total) continue;
      int part;
      const BwdItem t = decode(w, part);
      if (t.k1 == t.k0) continue;
      {
        for (int k = t.k0; k < t.k1; ++k, ++gstep) {
          const int h = t.hk * G + k / t.nqt, qt = t.qt0 + k % t.nqt;
          if (!wait_bar(&dq_full, gstep & 1, ctl)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const int fq = t.cq0 + qt * kBM + 32 * wq, bq = fq / p.seg.Sq, sq = fq - bq * p.seg.Sq;
#pragma unroll 1
          for (int c = 0; c < 4; ++c) {
            uint32_t a[32];
            tmem_ld32(tmem + lane_base + C::T_S + c * 32, a);
            uint8_t* box = stg + (c & 1) * 4096;
            if (c >= 2) {
              if (lane == 0) asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
              __syncwarp();
            }
#pragma unroll
            for (int u = 0; u < 8; ++u)
              *reinterpret_cast<uint4*>(box + sw128_offset(lane, u)) =
                  make_uint4(a[4 * u], a[4 * u + 1], a[4 * u + 2], a[4 * u + 3]);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              tma_reduce_add_4d(&p.tm_dq, box, part * 128 + c * 32, sq, h, bq);
              bulk_commit_group();
            }
          }
          // The staging sits in the P^T buffer: the next step may write P^T
          // only after these reduces have read it.
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

// fwd512.cuh -- attention forward for Dqk = 512 (Dv = 512 as two 256-column
// halves), sm_103a; the arithmetic is the one fwd.cuh states.
//
// Structure (one CTA per SM, persistent over a heaviest-first tile list):
//   warp 0      TMA producer: Q tile once per work tile, then K and V tiles as
//               16 KB chunks (128 rows x 64 columns, 128-byte swizzled) through
//               an NST-deep ring, in the order the MMA warp consumes them.
//   warp 1      one thread issues every tcgen05.mma: S = Q K^T into one of two
//               TMEM S buffers (fp32, 128 columns each), then O += P V with P
//               read from TMEM (bf16, written over the S buffer it came from).
//               Issue order QK(j+1) before PV(j) lets the tensor core compute
//               the next logits while the softmax works on the current ones.
//   warp 2      allocates / frees TMEM (512 columns).
//   warps 4-7   softmax warpgroup: thread t owns query row t (TMEM lane t). It
//               reads S, applies the mask only on tiles that cross a mask edge,
//               keeps the running max in log2 units with the scale folded in,
//               rescales O in TMEM only when the max grows by more than 2^8
//               (exact: the final division by the running sum cancels any
//               common factor), writes P, and at the end of the tile divides
//               O by the row sum and stores out and lse.
#pragma once

#include <math_constants.h>

#include "fwd.cuh"

namespace psf {

template <int DQK, int DVC>
struct FwdCfg {
  static constexpr int QCH = DQK / 64;  // 16 KB chunks per Q (or K) tile
  static constexpr int VCH = DVC / 64;  // chunks per V tile slice
  static constexpr int NQB = DQK >= 512 ? 1 : 2;
  static constexpr int NST = DQK >= 512 ? 6 : (DQK >= 192 ? 7 : 8);
  static constexpr int Q_BYTES = QCH * kChunkBytes;
  static constexpr int SMEM_BYTES = NQB * Q_BYTES + NST * kChunkBytes + 1024;
  static constexpr int TMEM_O = 256;
  static_assert(DVC <= 256, "O must fit next to two S buffers");
  static_assert(SMEM_BYTES + 512 <= 232448, "shared memory budget (dynamic + static)");
};

// CAP: logits softcapped (p.softcap > 0), applied to the score registers in
// place before the row maximum.
template <typename T, int DQK, int DVC, bool CAP>
__global__ void __launch_bounds__(256, 1) attn_fwd_kernel(const __grid_constant__ FwdParams p) {
  using C = FwdCfg<DQK, DVC>;
  constexpr int NST = C::NST, NQB = C::NQB;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* q_smem = smem;
  uint8_t* kv_smem = smem + NQB * C::Q_BYTES;

  __shared__ uint64_t q_full[NQB], q_empty[NQB], kv_full[NST], kv_empty[NST];
  __shared__ uint64_t s_full[2], p_full[2], pv_done, o_free, drain;
  __shared__ uint32_t tmem_base_smem;
  __shared__ int abort_flag;

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  if (threadIdx.x == 0) {
    for (int i = 0; i < NQB; ++i) {
      mbar_init(&q_full[i], 1);
      mbar_init(&q_empty[i], 1);
    }
    for (int i = 0; i < NST; ++i) {
      mbar_init(&kv_full[i], 1);
      mbar_init(&kv_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&p_full[i], 4);
    }
    mbar_init(&pv_done, 1);
    mbar_init(&o_free, 4);
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
  const int total = (*p.n_items) * (p.Hq / p.pack) * p.dv_parts;  // p.pack is 1 for this kernel
  const int G = p.Hq / p.Hkv;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&p.tm_q);
      tma_prefetch_desc(&p.tm_k);
      tma_prefetch_desc(&p.tm_v);
      uint32_t qcnt = 0, kvit = 0;
      bool ok = true;
      auto load_chunk = [&](const CUtensorMap* map, int c0, int row, int h, int b) -> bool {
        int st = kvit % NST;
        if (!wait_bar(&kv_empty[st], ((kvit / NST) & 1) ^ 1, ctl)) return false;
        mbar_arrive_expect_tx(&kv_full[st], kChunkBytes);
        tma_load_4d(kv_smem + st * kChunkBytes, map, &kv_full[st], c0, row, h, b);
        ++kvit;
        return true;
      };
      for (int wi = 0; wi * (int)gridDim.x < total && ok; ++wi) {
        const int w = snake_item(wi);
        if (w >= total) continue;
        FwdTile t = fwd_decode(p, w);
        if (t.nk == 0) continue;
        int qb = qcnt % NQB;
        if (!wait_bar(&q_empty[qb], ((qcnt / NQB) & 1) ^ 1, ctl)) break;
        mbar_arrive_expect_tx(&q_full[qb], C::Q_BYTES);
        int fq = t.cq0 + t.qt * kBM;
        int bq = fq / p.seg.Sq;
        for (int c = 0; c < C::QCH; ++c)
          tma_load_4d(q_smem + qb * C::Q_BYTES + c * kChunkBytes, &p.tm_q, &q_full[qb], c * 64, fq - bq * p.seg.Sq,
                      t.h, bq);
        ++qcnt;
        const int hk = t.h / G, dv0 = t.part * DVC;
        for (int jj = 0; jj <= t.nk && ok; ++jj) {
          if (jj < t.nk) {
            int fk = t.ck0 + (t.kv_t0 + jj) * kBN;
            int bk = fk / p.seg.Sk;
            for (int c = 0; c < C::QCH && ok; ++c) ok = load_chunk(&p.tm_k, c * 64, fk - bk * p.seg.Sk, hk, bk);
          }
          if (jj >= 1) {
            int fk = t.ck0 + (t.kv_t0 + jj - 1) * kBN;
            int bk = fk / p.seg.Sk;
            for (int c = 0; c < C::VCH && ok; ++c) ok = load_chunk(&p.tm_v, dv0 + c * 64, fk - bk * p.seg.Sk, hk, bk);
          }
        }
      }
      // Wind down: make sure no copy is still landing in shared memory.
      for (uint32_t i = kvit > (uint32_t)NST ? kvit - NST : 0; i < kvit; ++i)
        wait_bar_drain(&kv_full[i % NST], (i / NST) & 1, p.limit_ns);
      for (uint32_t i = qcnt > (uint32_t)NQB ? qcnt - NQB : 0; i < qcnt; ++i)
        wait_bar_drain(&q_full[i % NQB], (i / NQB) & 1, p.limit_ns);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_qk = idesc_f32acc<T>(128, 128, 0, 0);
      constexpr uint32_t idesc_pv = idesc_f32acc<T>(128, 64, 0, 1);
      constexpr uint32_t idesc_pv128 = idesc_f32acc<T>(128, 128, 0, 1);
      static_assert(C::VCH % 2 == 0, "V chunks go in pairs");
      uint32_t qcnt = 0, kvit = 0, scnt = 0, pcnt = 0, ntile = 0;
      bool ok = true;
      for (int wi = 0; wi * (int)gridDim.x < total && ok; ++wi) {
        const int w = snake_item(wi);
        if (w >= total) continue;
        FwdTile t = fwd_decode(p, w);
        if (t.nk == 0) continue;
        int qb = qcnt % NQB;
        if (!wait_bar(&q_full[qb], (qcnt / NQB) & 1, ctl)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t q_addr = smem_u32(q_smem + qb * C::Q_BYTES);
        for (int jj = 0; jj <= t.nk && ok; ++jj) {
          if (jj < t.nk) {
            const uint32_t sbuf = tmem + (scnt & 1) * 128;
            for (int c = 0; c < C::QCH; ++c) {
              int st = kvit % NST;
              if (!wait_bar(&kv_full[st], (kvit / NST) & 1, ctl)) {
                ok = false;
                break;
              }
              tc_fence_after();
              const uint32_t k_addr = smem_u32(kv_smem + st * kChunkBytes);
#pragma unroll
              for (int kk = 0; kk < 4; ++kk)
                mma_ss(sbuf, sdesc_sw128(q_addr + c * kChunkBytes + kk * 32, 16, 1024),
                       sdesc_sw128(k_addr + kk * 32, 16, 1024), idesc_qk, (c | kk) != 0);
              mma_commit(&kv_empty[st]);
              ++kvit;
            }
            if (!ok) break;
            mma_commit(&s_full[scnt & 1]);
            ++scnt;
            if (jj == t.nk - 1) mma_commit(&q_empty[qb]);
          }
          if (jj >= 1) {
            const int pb = pcnt & 1;
            if (!wait_bar(&p_full[pb], (pcnt >> 1) & 1, ctl)) {
              ok = false;
              break;
            }
            if (jj == 1 && ntile > 0 && !wait_bar(&o_free, (ntile - 1) & 1, ctl)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t p_tmem = tmem + pb * 128;
            // V chunks in pairs: two chunks in neighbouring ring slots make one
            // N = 128 chain (the second reached through the leading-byte
            // offset), which runs in about the time of one N = 64 chain.
            for (int c = 0; c < C::VCH; c += 2) {
              const int st0 = kvit % NST, st1 = (kvit + 1) % NST;
              if (!wait_bar(&kv_full[st0], (kvit / NST) & 1, ctl) ||
                  !wait_bar(&kv_full[st1], ((kvit + 1) / NST) & 1, ctl)) {
                ok = false;
                break;
              }
              tc_fence_after();
              const uint32_t v0 = smem_u32(kv_smem + st0 * kChunkBytes);
              if (st1 == st0 + 1) {
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                  mma_ts(tmem + C::TMEM_O + c * 64, p_tmem + kk * 8, sdesc_sw128(v0 + kk * 2048, kChunkBytes, 1024),
                         idesc_pv128, (jj > 1 || kk > 0));
              } else {
                const uint32_t v1 = smem_u32(kv_smem + st1 * kChunkBytes);
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                  mma_ts(tmem + C::TMEM_O + c * 64, p_tmem + kk * 8, sdesc_sw128(v0 + kk * 2048, kChunkBytes, 1024),
                         idesc_pv, (jj > 1 || kk > 0));
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                  mma_ts(tmem + C::TMEM_O + c * 64 + 64, p_tmem + kk * 8,
                         sdesc_sw128(v1 + kk * 2048, kChunkBytes, 1024), idesc_pv, (jj > 1 || kk > 0));
              }
              mma_commit(&kv_empty[st0]);
              mma_commit(&kv_empty[st1]);
              kvit += 2;
            }
            if (!ok) break;
            mma_commit(&pv_done);
            ++pcnt;
          }
        }
        ++qcnt;
        ++ntile;
      }
      // Wind down: wait until every MMA this thread issued has finished.
      mma_commit(&drain);
      wait_bar_drain(&drain, 0, p.limit_ns);
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ softmax warpgroup
    const int row = threadIdx.x - 128;
    const uint32_t lane_base = (uint32_t)(32 * (warp - 4)) << 16;
    const float sl2 = p.scale_log2;
    uint32_t scnt = 0, pvcnt = 0;
    bool ok = true;
    for (int wi = 0; wi * (int)gridDim.x < total && ok; ++wi) {
      const int w = snake_item(wi);
      if (w >= total) continue;
      FwdTile t = fwd_decode(p, w);
      const int i = t.qt * kBM + row;  // segment-local query index
      const bool valid = i < t.m;
      const int fq = t.cq0 + i;
      const int bq = fq / p.seg.Sq;
      const int sq = fq - bq * p.seg.Sq;
      T* orow = static_cast<T*>(p.out) + bq * p.o_sb + (int64_t)sq * p.o_ss + t.h * p.o_sh + t.part * DVC;
      float* lrow = p.lse + bq * p.l_sb + t.h * p.l_sh + sq;
      if (t.nk == 0) {
        if (valid) {
          uint4 z = make_uint4(0, 0, 0, 0);
#pragma unroll
          for (int c = 0; c < DVC / 8; ++c) reinterpret_cast<uint4*>(orow)[c] = z;
          if (t.part == 0) *lrow = -CUDART_INF_F;
        }
        continue;
      }
      const int delta = t.n - t.m;
      const int jmax_excl = p.seg.causal ? min(t.n, i + delta + 1) : t.n;
      const int jmin = p.seg.window > 0 ? i + delta - p.seg.window + 1 : -0x40000000;
      float m_used = -CUDART_INF_F, l = 0.f;
      for (int jj = 0; jj < t.nk; ++jj) {
        const int sb = scnt & 1;
        if (!wait_bar(&s_full[sb], (scnt >> 1) & 1, ctl)) {
          ok = false;
          break;
        }
        tc_fence_after();
        float s[128];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t r[32];
          tmem_ld32(tmem + lane_base + sb * 128 + c * 32, r);
#pragma unroll
          for (int j = 0; j < 32; ++j) s[c * 32 + j] = __uint_as_float(r[j]);
        }
        const int c0 = (t.kv_t0 + jj) * kBN;
        const int lo_c = jmin - c0, hi_c = jmax_excl - c0;
        if (lo_c > 0 || hi_c < kBN) {
#pragma unroll
          for (int j = 0; j < 128; ++j) s[j] = (j < lo_c || j >= hi_c) ? -CUDART_INF_F : s[j];
        }
        if constexpr (CAP) {
          // capped logits in log2 units; the multiplier below becomes 1
          const float k1 = 2.f * sl2 / p.softcap, c2 = p.softcap * 1.4426950408889634f;
#pragma unroll
          for (int j = 0; j < 128; ++j) s[j] = softcap_log2(s[j], k1, c2);
        }
        // Row maximum with eight independent chains (one warp per SM
        // sub-partition: latency, not throughput, bounds a single chain).
        float m8[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) m8[u] = s[u];
#pragma unroll
        for (int j = 8; j < 128; ++j) m8[j & 7] = fmaxf(m8[j & 7], s[j]);
        float mx = fmaxf(fmaxf(fmaxf(m8[0], m8[1]), fmaxf(m8[2], m8[3])), fmaxf(fmaxf(m8[4], m8[5]), fmaxf(m8[6], m8[7])));
        if constexpr (!CAP) mx *= sl2;
        const float m_new = (mx > m_used + 8.f) ? mx : m_used;
        const float alpha = (m_new == m_used) ? 1.f : ex2_approx(m_used - m_new);
        const float base = (m_new == -CUDART_INF_F) ? 0.f : m_new;
        float r8[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        uint32_t pa[32], pb2[32];
        const float2 sl2x2 = CAP ? make_float2(1.f, 1.f) : make_float2(sl2, sl2), nbase = make_float2(-base, -base);
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const float2 x = fma2(make_float2(s[2 * j], s[2 * j + 1]), sl2x2, nbase);
          const float e0 = ex2_approx(x.x), e1 = ex2_approx(x.y);
          r8[(2 * j) & 7] += e0;
          r8[(2 * j + 1) & 7] += e1;
          pa[j] = pack2<T>(e0, e1);
        }
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const float2 x = fma2(make_float2(s[64 + 2 * j], s[64 + 2 * j + 1]), sl2x2, nbase);
          const float e0 = ex2_approx(x.x), e1 = ex2_approx(x.y);
          r8[(2 * j) & 7] += e0;
          r8[(2 * j + 1) & 7] += e1;
          pb2[j] = pack2<T>(e0, e1);
        }
        const float rs = ((r8[0] + r8[1]) + (r8[2] + r8[3])) + ((r8[4] + r8[5]) + (r8[6] + r8[7]));
        if (jj > 0) {
          // O must hold PV(jj-1) before it is rescaled.
          if (!wait_bar(&pv_done, pvcnt & 1, ctl)) {
            ok = false;
            break;
          }
          ++pvcnt;
          tc_fence_after();
          if (__any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll 1
            for (int c = 0; c < DVC / 32; ++c) {
              uint32_t r[32];
              const uint32_t ta = tmem + lane_base + C::TMEM_O + c * 32;
              tmem_ld32(ta, r);
#pragma unroll
              for (int j = 0; j < 32; ++j) r[j] = __float_as_uint(__uint_as_float(r[j]) * alpha);
              tmem_st32(ta, r);
            }
          }
        }
        tmem_st32(tmem + lane_base + sb * 128, pa);
        tmem_st32(tmem + lane_base + sb * 128 + 32, pb2);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&p_full[sb]);
        l = l * alpha + rs;
        m_used = m_new;
        ++scnt;
      }
      if (!ok) break;
      if (!wait_bar(&pv_done, pvcnt & 1, ctl)) break;
      ++pvcnt;
      tc_fence_after();
      const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll 1
      for (int c = 0; c < DVC / 32; ++c) {
        uint32_t r[32];
        tmem_ld32(tmem + lane_base + C::TMEM_O + c * 32, r);
        if (valid) {
          uint32_t pk[16];
#pragma unroll
          for (int j = 0; j < 16; ++j)
            pk[j] = pack2<T>(__uint_as_float(r[2 * j]) * inv, __uint_as_float(r[2 * j + 1]) * inv);
          uint4* dst = reinterpret_cast<uint4*>(orow + c * 32);
#pragma unroll
          for (int j = 0; j < 4; ++j) dst[j] = make_uint4(pk[4 * j], pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]);
        }
      }
      if (valid && t.part == 0) *lrow = l > 0.f ? (m_used + __log2f(l)) * 0.69314718055994531f : -CUDART_INF_F;
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&o_free);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace psf

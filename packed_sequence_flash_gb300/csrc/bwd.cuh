// bwd.cuh -- what the attention backward kernels share: their parameter
// block and the decoding of a work unit.
//   [nemo_automodel.components.attention.ffpa_attention, `_ffpa_varlen_bwd`,
//    `_ffpa_dense_bwd`: gradients from the out and lse the caller passes in,
//    dK/dV summed over the query heads of each KV head]
//
// Per (segment, KV head, 128-row key tile) a CTA (or, at head dim 512, a
// cluster) walks every (query head of the GQA group, 128-row query tile) that
// can see the key tile. For each step, with thread r of a compute warpgroup
// owning key row r (TMEM lane r):
//   S^T  = K Q^T           (tcgen05, fp32 in TMEM)
//   dP^T = V dO^T          (tcgen05)
//   P^T  = exp2(S^T * scale * log2 e - lse * log2 e), 0 where masked or lse = -inf
//   dS^T = P^T (dP^T - Delta),  Delta = rowsum(dO * out) from the preprocess
//   dV  += P^T dO          (tcgen05, accumulated in TMEM across the whole group)
//   dK  += dS^T Q          (idem; the scale is applied once in the epilogue)
//   dQ   = dS K            (tcgen05 into TMEM, then added to an fp32 global
//                           accumulator with TMA reduce-add, 32 x 32 boxes)
// P^T and dS^T are written to shared memory as 16-bit values, which the MMAs
// read K-major (as P^T, dS^T) or M-major (as dS). The kernels: bwd_dual.cuh
// (Dqk, Dv <= 128), bwd192.cuh (192/128), bwd_wide.cuh (512).
#pragma once

#include <math_constants.h>

#include <type_traits>

#include "common.cuh"

namespace psf {

struct BwdParams {
  CUtensorMap tm_q, tm_k, tm_v, tm_do;  // bf16 (d, s, h, b) views, box (64, 128)
  CUtensorMap tm_dq;                    // fp32 dQ accumulator [rows][Hq][Dqk], box (32, 32)
  CUtensorMap tm_dk, tm_dv;             // fp32 dK / dV partial-sum slots [slot][Hkv][128][D], box (32, 32)
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
  const int* item_slot;  // per item: its dK/dV partial-sum slot, -1 when its key tile is whole
  const int* n_items;
  int* work_next;  // zeroed by the schedule kernel; kernels that take work dynamically count on it
  int* status;
  uint64_t limit_ns;
};

// One work unit: a key tile of one KV head and a range [k0, k1) of its steps.
// Step k is query head hk * G + k / nqt and query tile qt0 + k % nqt.
struct BwdItem {
  int s, kt, hk;
  int cq0, ck0, m, n;
  int qt0, nqt;  // query tiles [qt0, qt0 + nqt) (of p.seg.qrows rows) see this key tile
  int k0, k1;
  int slot;  // dK/dV partial-sum slot of a cut key tile's sub-range; -1: the whole tile
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
  t.slot = p.item_slot[item];
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

}  // namespace psf

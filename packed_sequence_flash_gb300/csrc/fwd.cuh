// fwd.cuh -- what the attention forward kernels share: their parameter block
// and the decoding of a work tile.
//
// Computes, per (segment, query head, 128-row query tile), the exact softmax
// attention out = softmax(scale * Q K^T) V over the keys each query may see and
// lse = log sum exp(scale * Q K^T) (natural log, fp32).
//   [nemo_automodel.components.attention.ffpa_attention, `_ffpa_varlen_fwd`,
//    `_ffpa_dense_fwd`; causal mask at each segment's bottom-right corner per
//    nemo_automodel.components.attention.fa4, module docstring bullet 2; left
//    window counting the current token per the attention utils page]
//
// The kernels: fwd_duo.cuh (head dims 64, 128), fwd_pair.cuh (192/128),
// fwd512.cuh (512).

#pragma once

#include <math_constants.h>

#include "common.cuh"

namespace psf {

struct FwdParams {
  CUtensorMap tm_q, tm_k, tm_v;  // (d, s, h, b) views, box (64, 128), 128B swizzle, bf16
  CUtensorMap tm_o;              // out, box (32, 32), 64B swizzle (the two-CTA kernel's epilogue stores)
  SegInfo seg;
  void* out;  // T (bf16 or fp16), the inputs' type
  int64_t o_sb, o_ss, o_sh;  // element strides of out (batch, row, head)
  float* lse;
  int64_t l_sb, l_sh;  // element strides of lse (batch, head); rows are contiguous
  int Hq, Hkv;
  int pack;      // query heads per tile: 1, or Hq / Hkv when a KV head's query heads share one tile
  int dv_parts;  // value-dim slices computed by separate tiles (each DVC wide)
  float scale_log2;
  float softcap;      // > 0: logits capped as softcap * tanh(logit / softcap) (the CAP kernels)
  const int2* items;  // (segment, q tile), heaviest first
  const int* n_items;
  int* work_next;  // zeroed by the schedule kernel; kernels that take work dynamically count on it
  int* status;
  uint64_t limit_ns;
};

struct FwdTile {
  int s, qt, h, part;  // h: the tile's first query head
  int cq0, ck0, m, n;
  int kv_t0, nk;
};

__device__ __forceinline__ FwdTile fwd_decode(const FwdParams& p, int w) {
  FwdTile t;
  const int hp = (p.Hq / p.pack) * p.dv_parts;
  int item = w / hp;
  int r = w - item * hp;
  const int hg = r / p.dv_parts;
  t.part = r - hg * p.dv_parts;
  t.h = hg * p.pack;
  int2 it = p.items[item];
  t.s = it.x;
  t.qt = it.y;
  t.cq0 = cu_q_at(p.seg, t.s);
  t.ck0 = cu_k_at(p.seg, t.s);
  t.m = cu_q_at(p.seg, t.s + 1) - t.cq0;
  t.n = cu_k_at(p.seg, t.s + 1) - t.ck0;
  int lo, hi;
  kv_range_for_q_tile(t.m, t.n, t.qt * p.seg.qrows, p.seg.causal, p.seg.window, lo, hi, p.seg.qrows);
  t.kv_t0 = lo / kBN;
  t.nk = hi > lo ? ceil_div(hi, kBN) - t.kv_t0 : 0;
  return t;
}

}  // namespace psf

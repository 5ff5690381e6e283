// aux.cu -- memory-bound kernels around the attention kernels: the tile
// schedulers, the doc-id segment builder, pad fixup, lse merge, the backward
// preprocess (Delta = rowsum(dO * O), zeroed accumulators) and the backward
// convert (fp32 accumulators -> bf16 dQ, dK, dV).
#include <math_constants.h>

#include "launch.h"

namespace psf {

namespace {

constexpr int kScanThreads = 1024;
constexpr int kBuckets = 1024;
// Per-segment tile prefixes live in shared memory when they fit (the common
// case); the workspace copy is used beyond that.
constexpr int kSmemPrefix = 6144;
// Tiles shorter than this many steps are never cut to fill the last wave (a
// cut costs a partial-sum slot round trip; short tiles leave short tails).
constexpr int kWaveFillMinSteps = 256;

// Exclusive block-wide prefix sum over kScanThreads threads; *total gets the sum.
__device__ int block_excl_scan(int v, int* total) {
  __shared__ int warp_tot[32];
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_tot[wid] = x;
  __syncthreads();
  if (wid == 0) {
    int t = warp_tot[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int y = __shfl_up_sync(0xffffffffu, t, o);
      if (lane >= o) t += y;
    }
    warp_tot[lane] = t;
  }
  __syncthreads();
  int res = (wid > 0 ? warp_tot[wid - 1] : 0) + x - v;
  *total = warp_tot[31];
  __syncthreads();
  return res;
}

__device__ int block_max(int v) {
  __shared__ int warp_max[32];
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = max(v, __shfl_xor_sync(0xffffffffu, v, o));
  if (lane == 0) warp_max[wid] = v;
  __syncthreads();
  int r = warp_max[0];
  for (int i = 1; i < 32; ++i) r = max(r, warp_max[i]);
  __syncthreads();
  return r;
}

// Largest s in [0, nseg) with prefix[s] <= x.
__device__ int find_segment(const int* prefix, int nseg, int x) {
  int lo = 0, hi = nseg - 1;
  while (lo < hi) {
    int mid = (lo + hi + 1) >> 1;
    if (prefix[mid] <= x)
      lo = mid;
    else
      hi = mid - 1;
  }
  return lo;
}

__device__ int tile_cost(const SegInfo& g, int s, int t, int over_keys) {
  int m = cu_q_at(g, s + 1) - cu_q_at(g, s);
  int n = cu_k_at(g, s + 1) - cu_k_at(g, s);
  int lo, hi;
  if (over_keys) {
    q_range_for_kv_tile(m, n, t * kBN, g.causal, g.window, lo, hi);
    return hi > lo ? ceil_div(hi, g.qrows) - lo / g.qrows : 0;
  }
  kv_range_for_q_tile(m, n, t * g.qrows, g.causal, g.window, lo, hi, g.qrows);
  return hi > lo ? ceil_div(hi, kBN) - lo / kBN : 0;
}

// Runs in one 1024-thread block (block 0 of fwd_prep_kernel).
__device__ void schedule_body(SegInfo g, int over_keys, int2* items, int* n_items,
                                                                int* seg_prefix, int item_cap, int* status) {
  __shared__ int hist[kBuckets];
  __shared__ int start[kBuckets];
  __shared__ int bad;
  const int tid = threadIdx.x;
  const int nseg = seg_count(g);
  __shared__ int prefix_smem[kSmemPrefix];
  int* pref = nseg + 1 <= kSmemPrefix ? prefix_smem : seg_prefix;
  const int max_q = g.dev_meta ? g.dev_meta[1] : g.max_q;
  const int max_k = g.dev_meta ? g.dev_meta[2] : g.max_k;
  const int Tq = g.B * g.Sq, Tk = g.B * g.Sk;
  hist[tid] = 0;
  if (tid == 0) {
    n_items[1] = 0;  // work counter of kernels that take items dynamically
    n_items[2] = 0;  // cut tiles
  }
  if (tid == 0) bad = (g.cu_q && nseg >= 0 && (g.cu_q[0] != 0 || g.cu_k[0] != 0)) ? 1 : 0;
  __syncthreads();
  int carry = 0;
  for (int base = 0; base < nseg; base += kScanThreads) {
    const int s = base + tid;
    int cnt = 0;
    if (s < nseg) {
      const int q0 = cu_q_at(g, s), q1 = cu_q_at(g, s + 1);
      const int k0 = cu_k_at(g, s), k1 = cu_k_at(g, s + 1);
      const int m = q1 - q0, n = k1 - k0;
      bool ok = m >= 0 && n >= 0 && q1 <= Tq && k1 <= Tk && (max_q < 0 || m <= max_q) && (max_k < 0 || n <= max_k);
      if (ok && g.B > 1)
        ok = (m == 0 || q0 / g.Sq == (q1 - 1) / g.Sq) && (n == 0 || k0 / g.Sk == (k1 - 1) / g.Sk);
      if (!ok) bad = 1;
      else cnt = over_keys ? ceil_div(n, kBN) : ceil_div(m, g.qrows);
    }
    int tot;
    const int ex = block_excl_scan(cnt, &tot);
    if (s < nseg) pref[s] = carry + ex;
    carry += tot;
  }
  if (tid == 0) pref[nseg] = carry;
  __syncthreads();
  if (bad || carry > item_cap) {
    if (tid == 0) {
      record_status(status, kStatusDeviceArgs);
      *n_items = 0;
    }
    return;
  }
  for (int x = tid; x < carry; x += kScanThreads) {
    const int s = find_segment(pref, nseg, x);
    const int c = tile_cost(g, s, x - pref[s], over_keys);
    atomicAdd(&hist[min(c, kBuckets - 1)], 1);
  }
  __syncthreads();
  // Heaviest bucket first: start[b] = number of items in buckets above b.
  int tot;
  const int rb = kBuckets - 1 - tid;
  const int ex = block_excl_scan(hist[rb], &tot);
  start[rb] = ex;
  hist[rb] = 0;
  __syncthreads();
  for (int x = tid; x < carry; x += kScanThreads) {
    const int s = find_segment(pref, nseg, x);
    const int t = x - pref[s];
    const int b = min(tile_cost(g, s, t, over_keys), kBuckets - 1);
    const int pos = start[b] + atomicAdd(&hist[b], 1);
    items[pos] = make_int2(s, t);
  }
  if (tid == 0) *n_items = carry;
}

// Backward work list: key tiles, each cut into sub-ranges of its G * nqt
// (query head, query tile) steps when it holds more than its share of the
// total (split_target > 0: aim at split_target sub-items' worth of steps),
// heaviest first. Items are (segment, key tile, first step, end step).
// The sub-ranges of a cut tile write their dK/dV partial sums to slots of
// their own: item_slot[i] is item i's slot (-1: the tile is whole and its
// unit writes dK/dV itself), and splits[0, n_items[2]) lists the cut tiles as
// (first key row, key rows, first slot, slot count) for the convert kernel.
// When tiles of one size carry most of the work, their units (tiles x KV
// heads) fill whole waves of the nctas CTAs but the last: if that wave is less
// than half full, enough of those tiles are cut into four that its units
// become quarter-length ones, which the heaviest-first order takes last.
// Runs in one 1024-thread block (block 0 of bwd_prep_kernel).
__device__ void bwd_schedule_body(SegInfo g, int G, int Hkv, int split_target, int nctas, int4* items,
                                  int* item_slot, int4* splits, int slot_cap, int* n_items, int* seg_prefix,
                                  int item_cap, int* status) {
  __shared__ int hist[kBuckets];
  __shared__ int start[kBuckets];
  __shared__ int bad;
  __shared__ unsigned long long total_steps;
  const int tid = threadIdx.x;
  const int nseg = seg_count(g);
  __shared__ int prefix_smem[kSmemPrefix];
  int* pref = nseg + 1 <= kSmemPrefix ? prefix_smem : seg_prefix;
  const int max_q = g.dev_meta ? g.dev_meta[1] : g.max_q;
  const int max_k = g.dev_meta ? g.dev_meta[2] : g.max_k;
  const int Tq = g.B * g.Sq, Tk = g.B * g.Sk;
  // Steps of a key tile: (query head groups) x (query tiles); a group is one
  // head, or kBM / qrows heads packed into one tile.
  const int Gs = G / (kBM / g.qrows);
  hist[tid] = 0;
  if (tid == 0) {
    n_items[1] = 0;  // work counter of kernels that take items dynamically
    n_items[2] = 0;  // cut tiles
  }
  if (tid == 0) {
    bad = (g.cu_q && nseg >= 0 && (g.cu_q[0] != 0 || g.cu_k[0] != 0)) ? 1 : 0;
    total_steps = 0;
  }
  __syncthreads();
  int carry = 0;
  for (int base = 0; base < nseg; base += kScanThreads) {
    const int s = base + tid;
    int cnt = 0;
    if (s < nseg) {
      const int q0 = cu_q_at(g, s), q1 = cu_q_at(g, s + 1);
      const int k0 = cu_k_at(g, s), k1 = cu_k_at(g, s + 1);
      const int m = q1 - q0, n = k1 - k0;
      bool ok = m >= 0 && n >= 0 && q1 <= Tq && k1 <= Tk && (max_q < 0 || m <= max_q) && (max_k < 0 || n <= max_k);
      if (ok && g.B > 1)
        ok = (m == 0 || q0 / g.Sq == (q1 - 1) / g.Sq) && (n == 0 || k0 / g.Sk == (k1 - 1) / g.Sk);
      if (!ok) bad = 1;
      else cnt = ceil_div(n, kBN);
    }
    int tot;
    const int ex = block_excl_scan(cnt, &tot);
    if (s < nseg) pref[s] = carry + ex;
    carry += tot;
  }
  if (tid == 0) pref[nseg] = carry;
  __syncthreads();
  if (bad) {
    if (tid == 0) {
      record_status(status, kStatusDeviceArgs);
      *n_items = 0;
    }
    return;
  }
  unsigned long long mine = 0;
  for (int x = tid; x < carry; x += kScanThreads) {
    const int s = find_segment(pref, nseg, x);
    mine += (unsigned long long)Gs * tile_cost(g, s, x - pref[s], 1);
  }
  atomicAdd(&total_steps, mine);
  __syncthreads();
  int smax = 0x7fffffff;
  if (split_target > 0) {
    const unsigned long long want = (total_steps * (unsigned long long)Hkv + split_target - 1) / split_target;
    smax = (int)(want < 4 ? 4 : (want > 0x7fffffffull ? 0x7fffffffull : want));
  }
  // The last wave of the largest uncut tiles' units: `extra` of those tiles
  // (a fixed choice: ranked by thread, then by each thread's tiles in order)
  // are cut into four.
  int lmax_mine = 0;
  for (int x = tid; x < carry; x += kScanThreads) {
    const int s = find_segment(pref, nseg, x);
    const int steps = Gs * tile_cost(g, s, x - pref[s], 1);
    if (steps <= smax) lmax_mine = max(lmax_mine, steps);
  }
  const int lmax = block_max(lmax_mine);
  int nmax_mine = 0;
  for (int x = tid; x < carry; x += kScanThreads) {
    const int s = find_segment(pref, nseg, x);
    if (Gs * tile_cost(g, s, x - pref[s], 1) == lmax) ++nmax_mine;
  }
  int nmax;
  const int cand_base = block_excl_scan(nmax_mine, &nmax);
  int extra = 0;
  if (split_target > 0 && nctas > 0 && lmax >= kWaveFillMinSteps) {
    const long long units = (long long)nmax * Hkv;
    if (units >= nctas && 2 * units * lmax >= (long long)(total_steps * (unsigned long long)Hkv)) {
      const long long r = units % nctas;
      if (r > 0 && 2 * r <= nctas) extra = (int)((r + Hkv - 1) / Hkv);
    }
  }
  // Sub-ranges of tile x (steps of it): the cap's cut, or four for the chosen
  // largest tiles; `cand` walks this thread's largest tiles in list order.
  auto sub_ranges = [&](int steps, int& cand) {
    int nsub = steps == 0 ? 1 : (int)(((long long)steps + smax - 1) / smax);
    if (extra > 0 && steps == lmax && nsub == 1) {
      if (cand < extra) nsub = 4;
      ++cand;
    }
    return nsub;
  };
  int nsub_total = 0, slots_mine = 0, cut_mine = 0;
  int cand = cand_base;
  for (int x = tid; x < carry; x += kScanThreads) {
    const int s = find_segment(pref, nseg, x);
    const int steps = Gs * tile_cost(g, s, x - pref[s], 1);
    const int nsub = sub_ranges(steps, cand);
    nsub_total += nsub;
    if (nsub > 1) {
      slots_mine += nsub;
      ++cut_mine;
    }
    for (int i = 0; i < nsub; ++i) {
      const int c = (int)((long long)steps * (i + 1) / nsub - (long long)steps * i / nsub);
      atomicAdd(&hist[min(c, kBuckets - 1)], 1);
    }
  }
  int n_all, slots_all, cut_all;
  block_excl_scan(nsub_total, &n_all);
  int slot_next = block_excl_scan(slots_mine, &slots_all);
  int cut_next = block_excl_scan(cut_mine, &cut_all);
  if (n_all > item_cap || slots_all > slot_cap) {
    if (tid == 0) {
      record_status(status, kStatusDeviceArgs);
      *n_items = 0;
    }
    return;
  }
  int tot;
  const int rb = kBuckets - 1 - tid;
  const int ex = block_excl_scan(hist[rb], &tot);
  start[rb] = ex;
  hist[rb] = 0;
  __syncthreads();
  cand = cand_base;
  for (int x = tid; x < carry; x += kScanThreads) {
    const int s = find_segment(pref, nseg, x);
    const int t = x - pref[s];
    const int steps = Gs * tile_cost(g, s, t, 1);
    const int nsub = sub_ranges(steps, cand);
    if (nsub > 1) {
      const int k0 = cu_k_at(g, s) + t * kBN;
      splits[cut_next++] = make_int4(k0, min(kBN, cu_k_at(g, s + 1) - k0), slot_next, nsub);
    }
    for (int i = 0; i < nsub; ++i) {
      const int a = (int)((long long)steps * i / nsub), e = (int)((long long)steps * (i + 1) / nsub);
      const int b = min(e - a, kBuckets - 1);
      const int at = start[b] + atomicAdd(&hist[b], 1);
      items[at] = make_int4(s, t, a, e);
      item_slot[at] = nsub > 1 ? slot_next + i : -1;
    }
    if (nsub > 1) slot_next += nsub;
  }
  if (tid == 0) {
    *n_items = n_all;
    n_items[2] = cut_all;
  }
}

// out = 0, lse = -inf for query rows at or past cu_q[nseg]; blocks bid of nblk.
__device__ void fwd_tail_body(SegInfo g, uint16_t* out, int64_t o_sb, int64_t o_ss, int64_t o_sh, float* lse,
                              int64_t l_sb, int64_t l_sh, int Hq, int Dv, int bid, int nblk) {
  const int nseg = seg_count(g);
  // Clamped: with invalid segment arrays (which the schedule rejects) this
  // still writes only rows of the tensor.
  const int first = max(cu_q_at(g, nseg), 0);
  const int64_t rows = (int64_t)g.B * g.Sq - first;
  if (rows <= 0) return;
  const int groups = Dv / 8;
  const int64_t total = rows * Hq * groups;
  for (int64_t x = bid * (int64_t)blockDim.x + threadIdx.x; x < total; x += (int64_t)nblk * blockDim.x) {
    const int gidx = (int)(x % groups);
    const int64_t rh = x / groups;
    const int h = (int)(rh % Hq);
    const int f = first + (int)(rh / Hq);
    const int b = f / g.Sq, s = f - b * g.Sq;
    reinterpret_cast<uint4*>(out + b * o_sb + (int64_t)s * o_ss + h * o_sh)[gidx] = make_uint4(0, 0, 0, 0);
    if (gidx == 0) lse[b * l_sb + h * l_sh + s] = -CUDART_INF_F;
  }
}

// Builder: a new piece starts where the id changes, at position 0, and at the
// end of the query shard; each piece is one segment.
constexpr int kBuildPer = 8;
__global__ void __launch_bounds__(kScanThreads) build_segments_kernel(const int32_t* ids, int B, int Sk, int Lq,
                                                                      int q0, int32_t* cu_q, int32_t* cu_k,
                                                                      int capacity, int32_t* meta, uint8_t* is_pad,
                                                                      int skip_pad, int* status) {
  const int tid = threadIdx.x;
  const int q_end = q0 + Lq;
  int offset = 0;
  for (int b = 0; b < B; ++b) {
    const int32_t* row = ids + (size_t)b * Sk;
    for (int base = 0; base < Sk; base += kScanThreads * kBuildPer) {
      const int j0 = base + tid * kBuildPer;
      uint32_t flags = 0;
      int cnt = 0;
#pragma unroll
      for (int e = 0; e < kBuildPer; ++e) {
        const int j = j0 + e;
        if (j < Sk && (j == 0 || j == q_end || row[j] != row[j - 1])) {
          flags |= 1u << e;
          cnt += (skip_pad && row[j] == 0) ? 2 : 1;
        }
      }
      int tot;
      int idx = offset + block_excl_scan(cnt, &tot);
#pragma unroll
      for (int e = 0; e < kBuildPer; ++e) {
        if (flags & (1u << e)) {
          const int j = j0 + e;
          const bool pad = row[j] == 0;
          if (idx < capacity) {
            cu_k[idx] = b * Sk + j;
            cu_q[idx] = b * Lq + min(max(j - q0, 0), Lq);
            if (is_pad) is_pad[idx] = pad ? 1 : 0;
          }
          ++idx;
          // Padding skip: the piece's queries got no keys above; its keys
          // start a second segment with no queries, whose query offset is the
          // next boundary's (filled in below, -1 until then).
          if (skip_pad && pad) {
            if (idx < capacity) {
              cu_k[idx] = b * Sk + j;
              cu_q[idx] = -1;
              if (is_pad) is_pad[idx] = 1;
            }
            ++idx;
          }
        }
      }
      offset += tot;
    }
  }
  const int nseg = offset;
  if (nseg > capacity) {
    if (tid == 0) {
      record_status(status, kStatusDeviceArgs);
      meta[0] = meta[1] = meta[2] = 0;
    }
    return;
  }
  if (tid == 0) {
    cu_q[nseg] = B * Lq;
    cu_k[nseg] = B * Sk;
  }
  __syncthreads();
  if (skip_pad) {
    // A -1 is always followed by a real boundary (or the end), never another -1.
    for (int i = tid; i < nseg; i += kScanThreads)
      if (cu_q[i] < 0) cu_q[i] = cu_q[i + 1];
    __syncthreads();
  }
  int mq = 0, mk = 0;
  for (int i = tid; i < nseg; i += kScanThreads) {
    mq = max(mq, cu_q[i + 1] - cu_q[i]);
    mk = max(mk, cu_k[i + 1] - cu_k[i]);
  }
  mq = block_max(mq);
  mk = block_max(mk);
  if (tid == 0) {
    meta[0] = nseg;
    meta[1] = mq;
    meta[2] = mk;
  }
}

// Dense-kernel eligibility of one ring chunk over all rows (one block):
//   local: the chunk [k0, k0 + Lk) ends where the shard [q0, q0 + Lq) ends and
//     contains it, and in every row the chunk's real tokens are one document
//     forming a prefix (no position p > k0 inside the chunk starts a non-zero
//     run);
//   cross: the chunk lies before the shard, in every row [k0, q0) is one
//     document d > 0 without padding and the shard starts with d and holds no
//     other non-zero run.
// flags[0] = local, flags[1] = cross (1 eligible, 0 not).
__global__ void __launch_bounds__(kScanThreads) chunk_dense_flags_kernel(const int32_t* ids, int B, int S, int q0,
                                                                         int Lq, int k0, int Lk, int32_t* flags) {
  const int tid = threadIdx.x;
  const int q_end = q0 + Lq, k_end = k0 + Lk;
  bool local = Lq > 0 && k0 <= q0 && k_end == q_end;
  bool cross = Lq > 0 && Lk > 0 && k_end <= q0;
  for (int b = 0; b < B && (local || cross); ++b) {
    const int32_t* row = ids + (size_t)b * S;
    int bad_local = 0, bad_cross = 0;
    if (local)
      for (int p = k0 + 1 + tid; p < k_end; p += kScanThreads) {
        const int32_t x = row[p];
        if (x != 0 && x != row[p - 1]) bad_local = 1;
      }
    if (cross) {
      const int32_t d = row[k0];
      if (tid == 0 && (d <= 0 || row[q0] != d)) bad_cross = 1;
      for (int p = k0 + 1 + tid; p < q0; p += kScanThreads)
        if (row[p] != d) bad_cross = 1;
      for (int p = q0 + 1 + tid; p < q_end; p += kScanThreads) {
        const int32_t x = row[p];
        if (x != 0 && x != row[p - 1]) bad_cross = 1;
      }
    }
    if (__syncthreads_or(bad_local)) local = false;
    if (__syncthreads_or(bad_cross)) cross = false;
  }
  if (tid == 0) {
    flags[0] = local ? 1 : 0;
    flags[1] = cross ? 1 : 0;
  }
}

// One warp per query row: a padding row (id 0) gets out = 0 on every head and
// lse = -inf; other rows cost one id read.
__global__ void pad_fixup_kernel(uint16_t* out, float* lse, const int32_t* qids, int B, int Lq, int Hq, int Dv,
                                 int64_t o_sb, int64_t o_ss, int64_t o_sh, int64_t l_sb, int64_t l_sh) {
  const int lane = threadIdx.x & 31;
  const int64_t rows = (int64_t)B * Lq;
  const int64_t nwarps = (int64_t)gridDim.x * (blockDim.x / 32);
  const int groups = Dv / 8;
  for (int64_t f = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) / 32; f < rows; f += nwarps) {
    if (qids[f] != 0) continue;
    const int b = (int)(f / Lq), s = (int)(f - (int64_t)b * Lq);
    for (int x = lane; x < Hq * groups; x += 32) {
      const int h = x / groups, gidx = x - h * groups;
      reinterpret_cast<uint4*>(out + b * o_sb + (int64_t)s * o_ss + h * o_sh)[gidx] = make_uint4(0, 0, 0, 0);
    }
    for (int h = lane; h < Hq; h += 32) lse[b * l_sb + h * l_sh + s] = -CUDART_INF_F;
  }
}

template <typename E>
__global__ void lse_merge_kernel(const E* o1, const float* l1, const E* o2, const float* l2, float* of, E* ob,
                                 float* l, int T, int H, int D) {
  const int groups = D / 8;
  const int64_t total = (int64_t)T * H * groups;
  for (int64_t x = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; x < total; x += (int64_t)gridDim.x * blockDim.x) {
    const int gidx = (int)(x % groups);
    const int64_t th = x / groups;
    const int h = (int)(th % H);
    const int t = (int)(th / H);
    const float a = l1[(int64_t)h * T + t], c = l2[(int64_t)h * T + t];
    const float mx = fmaxf(a, c);
    const float lm = mx == -CUDART_INF_F ? -CUDART_INF_F : mx + logf(expf(a - mx) + expf(c - mx));
    const float wa = lm == -CUDART_INF_F ? 0.f : expf(a - lm);
    const float wc = lm == -CUDART_INF_F ? 0.f : expf(c - lm);
    const int64_t off = th * D + gidx * 8;
    uint4 ua = *reinterpret_cast<const uint4*>(o1 + off);
    uint4 uc = *reinterpret_cast<const uint4*>(o2 + off);
    const uint32_t* pa = reinterpret_cast<const uint32_t*>(&ua);
    const uint32_t* pc = reinterpret_cast<const uint32_t*>(&uc);
    float r[8];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float2 fa = unpack2<E>(pa[j]), fc = unpack2<E>(pc[j]);
      r[2 * j] = wa * fa.x + wc * fc.x;
      r[2 * j + 1] = wa * fa.y + wc * fc.y;
    }
    if (of) {
      reinterpret_cast<float4*>(of + off)[0] = make_float4(r[0], r[1], r[2], r[3]);
      reinterpret_cast<float4*>(of + off)[1] = make_float4(r[4], r[5], r[6], r[7]);
    }
    if (ob)
      *reinterpret_cast<uint4*>(ob + off) =
          make_uint4(pack2<E>(r[0], r[1]), pack2<E>(r[2], r[3]), pack2<E>(r[4], r[5]), pack2<E>(r[6], r[7]));
    if (gidx == 0) l[(int64_t)h * T + t] = lm;
  }
}

// Delta = sum_d dO * O in fp32, by groups of min(32, Dv/8) lanes per
// (row, head), with the grid-stride zeroing of the fp32 dQ accumulator spread
// over the Delta passes; then the zeroed dK / dV rows past the last segment.
// Blocks bid of nblk.
constexpr int kDeltaUnroll = 2;
template <typename E>
__device__ void bwd_pre_body(SegInfo g, const E* dout, int64_t d_sb, int64_t d_ss, int64_t d_sh, const E* out,
                             int64_t o_sb, int64_t o_ss, int64_t o_sh, float* delta, float* dq_acc, int Hq, int Dqk, int Dv,
                             uint16_t* dk, uint16_t* dv, int64_t k_sb,
                             int64_t k_ss, int64_t k_sh, int64_t v_sb, int64_t v_ss, int64_t v_sh, int Hkv, int bid,
                             int nblk) {
  const int64_t rows = (int64_t)g.B * g.Sq;
  const int lanes = min(32, Dv / 8);
  const int lane = threadIdx.x & 31;
  const int sub = lane % lanes, grp = lane / lanes, per_warp = 32 / lanes;
  const int64_t nwarps = (int64_t)nblk * (blockDim.x / 32);
  const int64_t n = rows * Hq, stride = nwarps * per_warp;
  // kDeltaUnroll (row, head) pairs per lane group and pass, all loads issued together.
  constexpr int U = kDeltaUnroll;
  // The dQ accumulator's zero stores go out a few per pass, between the
  // passes' loads, so the writes overlap the reads' latency.
  const int64_t tid = bid * (int64_t)blockDim.x + threadIdx.x;
  const int64_t nthr = (int64_t)nblk * blockDim.x;
  const float4 z4 = make_float4(0.f, 0.f, 0.f, 0.f);
  const int64_t n4 = rows * Hq * Dqk / 4;
  int64_t zx = tid;
  for (int64_t base = (bid * (int64_t)blockDim.x + threadIdx.x) / 32 * per_warp; base < n; base += stride * U) {
#pragma unroll
    for (int i = 0; i < 4; ++i)
      if (zx < n4) {
        reinterpret_cast<float4*>(dq_acc)[zx] = z4;
        zx += nthr;
      }
    float acc[U];
    int64_t off[U], doff[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      acc[u] = 0.f;
      const int64_t wrk = base + u * stride + grp;
      const int64_t f = wrk / Hq;
      const int h = (int)(wrk - f * Hq);
      const int b = (int)(f / g.Sq), s = (int)(f - (int64_t)b * g.Sq);
      const bool live = wrk < n && grp < per_warp;
      off[u] = live ? b * o_sb + (int64_t)s * o_ss + h * o_sh : -1;
      doff[u] = live ? b * d_sb + (int64_t)s * d_ss + h * d_sh : -1;
    }
    for (int d = sub * 8; d < Dv; d += lanes * 8) {
      uint4 ug[U], uo[U];
#pragma unroll
      for (int u = 0; u < U; ++u)
        if (off[u] >= 0) {
          ug[u] = *reinterpret_cast<const uint4*>(dout + doff[u] + d);
          uo[u] = *reinterpret_cast<const uint4*>(out + off[u] + d);
        }
#pragma unroll
      for (int u = 0; u < U; ++u)
        if (off[u] >= 0) {
          const uint32_t* pg = reinterpret_cast<const uint32_t*>(&ug[u]);
          const uint32_t* po = reinterpret_cast<const uint32_t*>(&uo[u]);
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const float2 x = unpack2<E>(pg[j]), y = unpack2<E>(po[j]);
            acc[u] = fmaf(x.x, y.x, acc[u]);
            acc[u] = fmaf(x.y, y.y, acc[u]);
          }
        }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      for (int o = lanes / 2; o > 0; o >>= 1) acc[u] += __shfl_xor_sync(0xffffffffu, acc[u], o);
      const int64_t wrk = base + u * stride + grp;
      if (sub == 0 && off[u] >= 0) {
        const int64_t f = wrk / Hq;
        delta[(int64_t)(wrk - f * Hq) * rows + f] = acc[u];
      }
    }
  }
  for (; zx < n4; zx += nthr) reinterpret_cast<float4*>(dq_acc)[zx] = z4;
  // dK / dV rows inside segments are written by the attention kernel (or the
  // convert, for cut key tiles); rows past the last segment are zero.
  const int64_t krows_all = (int64_t)g.B * g.Sk;
  const int first = max(cu_k_at(g, seg_count(g)), 0);  // clamped as in fwd_tail_body
  const int64_t krows = krows_all - first;
  if (krows > 0) {
    const int gk = Dqk / 8, gv = Dv / 8;
    const int64_t nk = krows * Hkv * (gk + gv);
    for (int64_t x = tid; x < nk; x += nthr) {
      int64_t rh = x / (gk + gv);
      int gidx = (int)(x - rh * (gk + gv));
      const int h = (int)(rh % Hkv);
      const int f = first + (int)(rh / Hkv);
      const int b = f / g.Sk, s = f - b * g.Sk;
      if (gidx < gk)
        reinterpret_cast<uint4*>(dk + b * k_sb + (int64_t)s * k_ss + h * k_sh)[gidx] = make_uint4(0, 0, 0, 0);
      else
        reinterpret_cast<uint4*>(dv + b * v_sb + (int64_t)s * v_ss + h * v_sh)[gidx - gk] = make_uint4(0, 0, 0, 0);
    }
  }
}

// E out = scale * fp32 accumulator ([rows][H][D], packed) in the tensor's own
// layout, for packed row f of a warp: the row's H*D/8 pieces, four per lane in
// flight.
template <typename E>
__device__ __forceinline__ void convert_row(const float* __restrict__ acc, E* __restrict__ dst, int64_t f, int Sr,
                                            int H, int D, int64_t sb, int64_t ss, int64_t sh, float scale) {
  const int G = D / 8, n = H * G, lane = threadIdx.x & 31;
  const int b = (int)(f / Sr), s = (int)(f - (int64_t)b * Sr);
  const float4* src = reinterpret_cast<const float4*>(acc + f * H * D);
  E* row = dst + b * sb + (int64_t)s * ss;
  for (int i0 = lane; i0 < n; i0 += 128) {
    float4 a[4], c[4];
#pragma unroll
    for (int u = 0; u < 4; ++u)
      if (i0 + 32 * u < n) {
        a[u] = src[2 * (i0 + 32 * u)];
        c[u] = src[2 * (i0 + 32 * u) + 1];
      }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int i = i0 + 32 * u;
      if (i >= n) continue;
      const int h = i / G, gi = i - h * G;
      reinterpret_cast<uint4*>(row + h * sh)[gi] =
          make_uint4(pack2<E>(a[u].x * scale, a[u].y * scale), pack2<E>(a[u].z * scale, a[u].w * scale),
                     pack2<E>(c[u].x * scale, c[u].y * scale), pack2<E>(c[u].z * scale, c[u].w * scale));
    }
  }
}

// dQ = scale * dQacc, a warp per packed row; then dK = scale * (sum of the
// partial-sum slots) and dV = (sum of its slots) for the key rows of every
// cut key tile, a warp per (tile, KV head, key row). The dQ rows come first,
// so they need neither the cut-tile count nor the list. A slot holds
// [Hkv][128][D] fp32 rows.
template <typename E>
__global__ void __launch_bounds__(256, 4) bwd_convert_kernel(const float* dq_acc, E* dq, int64_t nq, int Sq, int Hq, int Dqk,
                                   int64_t q_sb, int64_t q_ss, int64_t q_sh, SegInfo g, const int4* splits,
                                   const int* n_split, const float* pk, const float* pv, E* dk, E* dv, int Hkv, int Dv,
                                   int64_t k_sb, int64_t k_ss, int64_t k_sh, int64_t v_sb, int64_t v_ss, int64_t v_sh,
                                   float scale) {
  const int64_t nw = (int64_t)gridDim.x * (blockDim.x / 32);
  const int lane = threadIdx.x & 31;
  const int64_t per_tile = (int64_t)Hkv * kBN;
  const int64_t w0 = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) / 32;
  int64_t x = w0;
  for (; x < nq; x += nw) convert_row(dq_acc, dq, x, Sq, Hq, Dqk, q_sb, q_ss, q_sh, scale);
  if (!splits) return;
  const int64_t ncut = (int64_t)(*n_split) * per_tile;
  for (x -= nq; x < ncut; x += nw) {
    const int e = (int)(x / per_tile);
    const int rem = (int)(x - e * per_tile), hk = rem / kBN, r = rem % kBN;
    const int4 sp = splits[e];  // (first key row, key rows, first slot, slot count)
    if (r >= sp.y) continue;
    const int f = sp.x + r, b = f / g.Sk, sr = f - b * g.Sk;
    // Lane l holds elements [4l, 4l + 4) of the dK row and of the dV row; the
    // slots' loads go out four at a time.
    const bool on_k = lane * 4 < Dqk, on_v = lane * 4 < Dv;
    const float* srck = pk + (((int64_t)sp.z * Hkv + hk) * kBN + r) * Dqk + lane * 4;
    const float* srcv = pv + (((int64_t)sp.z * Hkv + hk) * kBN + r) * Dv + lane * 4;
    const int64_t stk = (int64_t)Hkv * kBN * Dqk, stv = (int64_t)Hkv * kBN * Dv;
    float4 ak = make_float4(0.f, 0.f, 0.f, 0.f), av = ak;
    for (int i0 = 0; i0 < sp.w; i0 += 4) {
      float4 lk[4], lv[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const bool in = i0 + u < sp.w;
        lk[u] = in && on_k ? *reinterpret_cast<const float4*>(srck + (i0 + u) * stk) : make_float4(0.f, 0.f, 0.f, 0.f);
        lv[u] = in && on_v ? *reinterpret_cast<const float4*>(srcv + (i0 + u) * stv) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        ak.x += lk[u].x;
        ak.y += lk[u].y;
        ak.z += lk[u].z;
        ak.w += lk[u].w;
        av.x += lv[u].x;
        av.y += lv[u].y;
        av.z += lv[u].z;
        av.w += lv[u].w;
      }
    }
    if (on_k)
      *reinterpret_cast<uint2*>(dk + b * k_sb + (int64_t)sr * k_ss + hk * k_sh + lane * 4) =
          make_uint2(pack2<E>(ak.x * scale, ak.y * scale), pack2<E>(ak.z * scale, ak.w * scale));
    if (on_v)
      *reinterpret_cast<uint2*>(dv + b * v_sb + (int64_t)sr * v_ss + hk * v_sh + lane * 4) =
          make_uint2(pack2<E>(av.x, av.y), pack2<E>(av.z, av.w));
  }
}

// Cross-chunk segments of a query shard [q0, q0 + Lq) against an earlier key
// chunk [k0, k0 + Lk) of every row: block b handles row b. Runs are contiguous,
// so only the run holding position q0 can reach back into the chunk; the block
// finds where that run starts inside the chunk (the last position in [k0, q0)
// with another id, plus one) and where it ends inside the shard.
// dev_meta must hold zeros on entry (the launcher clears it).
__global__ void __launch_bounds__(kScanThreads) cross_segments_kernel(const int32_t* ids, int B, int S, int q0, int Lq,
                                                                      int k0, int Lk, int32_t* cu_q, int32_t* cu_k,
                                                                      int32_t* dev_meta) {
  const int b = blockIdx.x, tid = threadIdx.x;
  const int32_t* row = ids + (size_t)b * S;
  int nq = 0, ks = k0 + Lk;  // shared run: shard queries [q0, q0 + nq), chunk keys [ks, k0 + Lk)
  if (Lq > 0 && Lk > 0) {
    const int d = row[q0];
    if (d != 0) {
      // Eight loads in flight per thread and pass.
      int last = k0 - 1;
      for (int p0 = k0 + tid; p0 < q0; p0 += 8 * blockDim.x) {
        int v[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int p = p0 + u * blockDim.x;
          v[u] = p < q0 ? row[p] : d;
        }
#pragma unroll
        for (int u = 0; u < 8; ++u)
          if (v[u] != d) last = max(last, p0 + u * (int)blockDim.x);
      }
      last = block_max(last);
      if (last + 1 < k0 + Lk) {
        ks = last + 1;
        int first = -(q0 + Lq);  // block_max of the negated first position with another id
        for (int p0 = q0 + tid; p0 < q0 + Lq; p0 += 8 * blockDim.x) {
          int v[8];
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const int p = p0 + u * blockDim.x;
            v[u] = p < q0 + Lq ? row[p] : d;
          }
#pragma unroll
          for (int u = 0; u < 8; ++u)
            if (v[u] != d) first = max(first, -(p0 + u * (int)blockDim.x));
        }
        nq = -block_max(first) - q0;
      }
    }
  }
  if (tid == 0) {
    const int qb = b * Lq, kb = b * Lk;
    cu_q[3 * b + 1] = qb;
    cu_q[3 * b + 2] = qb + nq;
    cu_q[3 * b + 3] = qb + Lq;
    cu_k[3 * b + 1] = kb + (ks - k0);
    cu_k[3 * b + 2] = kb + Lk;
    cu_k[3 * b + 3] = kb + Lk;
    if (b == 0) {
      cu_q[0] = 0;
      cu_k[0] = 0;
      dev_meta[0] = 3 * B;
    }
    atomicMax(&dev_meta[1], max(nq, Lq - nq));
    atomicMax(&dev_meta[2], max(ks - k0, k0 + Lk - ks));
  }
}

// Segment holding row t (cu_q[s] <= t < cu_q[s + 1]) if it has keys, else -1.
__device__ __forceinline__ int live_segment(const int32_t* cu_q, const int32_t* cu_k, int nseg, int t) {
  int lo = 0, hi = nseg - 1;  // largest s in [0, nseg) with cu_q[s] <= t
  if (nseg <= 0 || __ldg(cu_q) > t) return -1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (__ldg(cu_q + mid) <= t)
      lo = mid;
    else
      hi = mid - 1;
  }
  if (t >= __ldg(cu_q + lo + 1)) return -1;
  return __ldg(cu_k + lo + 1) > __ldg(cu_k + lo) ? lo : -1;
}

// In-place merge of one chunk's (o_new, l_new) into the running result on the
// query rows of the chunk's segments with keys. A warp takes one row at a time
// (one segment lookup per row) and its heads 32 at a time: lane i merges the
// lse of head hb + i, which only it reads and writes, then the warp streams the
// heads' 8-element pieces, four (two with kAcc) per lane in flight, each
// taking its weights from the head's lane by shuffle. kAcc: the running output is read from o_acc
// (fp32) and written to it and to o_run when given; otherwise it is read from
// and written to o_run (E).
template <typename E, bool kAcc>
__global__ void __launch_bounds__(256, 4)
    lse_merge_live_kernel(float* __restrict__ o_acc, E* __restrict__ o_run, float* __restrict__ l_acc,
                          const E* __restrict__ o_new, const float* __restrict__ l_new, const int32_t* cu_q,
                          const int32_t* cu_k, const int32_t* dev_meta, int nseg_cap, int T, int H, int D) {
  constexpr int U = kAcc ? 2 : 4;
  const int nseg = dev_meta ? min(dev_meta[0], nseg_cap) : nseg_cap;
  const int G = D / 8;  // pieces per head
  const int lane = threadIdx.x & 31;
  const int nw = gridDim.x * (blockDim.x / 32);
  for (int t = (blockIdx.x * blockDim.x + threadIdx.x) / 32; t < T; t += nw) {
    if (live_segment(cu_q, cu_k, nseg, t) < 0) continue;
    for (int hb = 0; hb < H; hb += 32) {
      const int h = hb + lane;
      float wa = 0.f, wc = 0.f;
      if (h < H) {
        const float a = l_acc[(int64_t)h * T + t], c = l_new[(int64_t)h * T + t];
        const float m = fmaxf(a, c);
        const float l = m == -CUDART_INF_F ? -CUDART_INF_F : m + logf(expf(a - m) + expf(c - m));
        if (l != -CUDART_INF_F) {
          wa = expf(a - l);
          wc = expf(c - l);
        }
        l_acc[(int64_t)h * T + t] = l;
      }
      const int n = min(32, H - hb) * G;
      const int64_t base = ((int64_t)t * H + hb) * D;
      for (int k0 = 0; k0 < n; k0 += 32 * U) {  // the same trip count on every lane
        const int i0 = k0 + lane;
        uint4 un[U], ur[U];
        float4 fa[U][2];
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int i = i0 + 32 * u;
          if (i >= n) continue;
          const int64_t off = base + (int64_t)i * 8;
          if constexpr (kAcc) {
            fa[u][0] = reinterpret_cast<const float4*>(o_acc + off)[0];
            fa[u][1] = reinterpret_cast<const float4*>(o_acc + off)[1];
          } else {
            ur[u] = *reinterpret_cast<const uint4*>(o_run + off);
          }
          un[u] = *reinterpret_cast<const uint4*>(o_new + off);
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int i = i0 + 32 * u;
          const int src = min(i, n - 1) / G;  // every lane takes part in the shuffles
          const float w_a = __shfl_sync(0xffffffffu, wa, src), w_c = __shfl_sync(0xffffffffu, wc, src);
          if (i >= n) continue;
          const int64_t off = base + (int64_t)i * 8;
          float x8[8];
          if constexpr (kAcc) {
            x8[0] = fa[u][0].x; x8[1] = fa[u][0].y; x8[2] = fa[u][0].z; x8[3] = fa[u][0].w;
            x8[4] = fa[u][1].x; x8[5] = fa[u][1].y; x8[6] = fa[u][1].z; x8[7] = fa[u][1].w;
          } else {
            const uint32_t* pr = reinterpret_cast<const uint32_t*>(&ur[u]);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const float2 f = unpack2<E>(pr[j]);
              x8[2 * j] = f.x;
              x8[2 * j + 1] = f.y;
            }
          }
          const uint32_t* pn = reinterpret_cast<const uint32_t*>(&un[u]);
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const float2 f = unpack2<E>(pn[j]);
            x8[2 * j] = w_a * x8[2 * j] + w_c * f.x;
            x8[2 * j + 1] = w_a * x8[2 * j + 1] + w_c * f.y;
          }
          if constexpr (kAcc) {
            reinterpret_cast<float4*>(o_acc + off)[0] = make_float4(x8[0], x8[1], x8[2], x8[3]);
            reinterpret_cast<float4*>(o_acc + off)[1] = make_float4(x8[4], x8[5], x8[6], x8[7]);
          }
          if (!kAcc || o_run)
            *reinterpret_cast<uint4*>(o_run + off) =
                make_uint4(pack2<E>(x8[0], x8[1]), pack2<E>(x8[2], x8[3]), pack2<E>(x8[4], x8[5]), pack2<E>(x8[6], x8[7]));
        }
      }
    }
  }
}

// dst += src (E, added in fp32, rounded once) on the query rows of the
// segments with keys. A warp takes one row at a time (one segment lookup per
// row) and walks its H*D/8 16-byte pieces with four pieces per lane in flight.
template <typename E>
__global__ void grad_add_live_kernel(E* __restrict__ dst, const E* __restrict__ src, const int32_t* cu_q,
                                     const int32_t* cu_k, const int32_t* dev_meta, int nseg_cap, int T, int H, int D) {
  const int nseg = dev_meta ? min(dev_meta[0], nseg_cap) : nseg_cap;
  const int per_row = H * (D / 8);
  const int lane = threadIdx.x & 31;
  const int nw = gridDim.x * (blockDim.x / 32);
  for (int t = (blockIdx.x * blockDim.x + threadIdx.x) / 32; t < T; t += nw) {
    if (live_segment(cu_q, cu_k, nseg, t) < 0) continue;
    uint4* a = reinterpret_cast<uint4*>(dst) + (int64_t)t * per_row;
    const uint4* b = reinterpret_cast<const uint4*>(src) + (int64_t)t * per_row;
    for (int i0 = lane; i0 < per_row; i0 += 128) {
      uint4 ua[4], ub[4];
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if (i0 + 32 * u < per_row) {
          ua[u] = a[i0 + 32 * u];
          ub[u] = b[i0 + 32 * u];
        }
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if (i0 + 32 * u < per_row) {
          const uint32_t* pa = reinterpret_cast<const uint32_t*>(&ua[u]);
          const uint32_t* pb = reinterpret_cast<const uint32_t*>(&ub[u]);
          uint4 r;
          uint32_t* rp = reinterpret_cast<uint32_t*>(&r);
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const float2 fa = unpack2<E>(pa[j]), fb = unpack2<E>(pb[j]);
            rp[j] = pack2<E>(fa.x + fb.x, fa.y + fb.y);
          }
          a[i0 + 32 * u] = r;
        }
    }
  }
}

// Forward preparation: block 0 builds the heaviest-first tile list while the
// other blocks fill uncovered query rows, so the list's latency-bound build
// overlaps the fill and costs no launch of its own.
__global__ void __launch_bounds__(kScanThreads) fwd_prep_kernel(SegInfo g, int2* items, int* n_items, int* seg_prefix,
                                                                int item_cap, int* status, uint16_t* out,
                                                                int64_t o_sb, int64_t o_ss, int64_t o_sh, float* lse,
                                                                int64_t l_sb, int64_t l_sh, int Hq, int Dv) {
  if (blockIdx.x == 0)
    schedule_body(g, 0, items, n_items, seg_prefix, item_cap, status);
  else
    fwd_tail_body(g, out, o_sb, o_ss, o_sh, lse, l_sb, l_sh, Hq, Dv, blockIdx.x - 1, gridDim.x - 1);
}

// Backward preparation: block 0 builds the work list while the other blocks
// compute Delta and zero the accumulators (HBM-bound), hiding the list's
// latency behind that traffic.
template <typename E>
__global__ void __launch_bounds__(kScanThreads) bwd_prep_kernel(
    SegInfo g, int G, int Hkv, int split_target, int nctas, int4* items, int* item_slot, int4* splits,
    int slot_cap, int* n_items, int* seg_prefix, int item_cap, int* status, const E* dout, int64_t d_sb, int64_t d_ss,
    int64_t d_sh,
    const E* out, int64_t o_sb, int64_t o_ss, int64_t o_sh, float* delta, float* dq_acc, int Hq, int Dqk, int Dv,
    uint16_t* dk, uint16_t* dv, int64_t k_sb, int64_t k_ss, int64_t k_sh, int64_t v_sb, int64_t v_ss, int64_t v_sh) {
  if (blockIdx.x == 0)
    bwd_schedule_body(g, G, Hkv, split_target, nctas, items, item_slot, splits, slot_cap, n_items, seg_prefix,
                      item_cap, status);
  else
    bwd_pre_body(g, dout, d_sb, d_ss, d_sh, out, o_sb, o_ss, o_sh, delta, dq_acc, Hq, Dqk, Dv, dk, dv, k_sb, k_ss,
                 k_sh, v_sb, v_ss, v_sh, Hkv, blockIdx.x - 1, gridDim.x - 1);
}

int grid_for(int64_t work, int threads) {
  int64_t g = (work + threads - 1) / threads;
  if (g < 1) g = 1;
  if (g > 152 * 16) g = 152 * 16;
  return (int)g;
}

}  // namespace

cudaError_t launch_fwd_prep(const SegInfo& g, int2* items, int* n_items, int* seg_prefix, int item_cap, int* status,
                            void* out, int64_t o_sb, int64_t o_ss, int64_t o_sh, float* lse, int64_t l_sb,
                            int64_t l_sh, int Hq, int Dv, cudaStream_t st) {
  // The fill usually has no rows at all (the builder covers every token); a
  // few blocks with a grid-stride loop cover the rest.
  const int fill = min(grid_for((int64_t)g.B * g.Sq * Hq * (Dv / 8), kScanThreads), 2 * 152);
  fwd_prep_kernel<<<1 + fill, kScanThreads, 0, st>>>(g, items, n_items, seg_prefix, item_cap, status,
                                                     static_cast<uint16_t*>(out), o_sb, o_ss, o_sh, lse, l_sb, l_sh,
                                                     Hq, Dv);
  return cudaGetLastError();
}
cudaError_t launch_build_segments(const int32_t* ids, int B, int Sk, int Lq, int q0, int32_t* cu_q, int32_t* cu_k,
                                  int capacity, int32_t* meta, uint8_t* seg_is_pad, int skip_pad, int* status,
                                  cudaStream_t st) {
  build_segments_kernel<<<1, kScanThreads, 0, st>>>(ids, B, Sk, Lq, q0, cu_q, cu_k, capacity, meta, seg_is_pad,
                                                    skip_pad, status);
  return cudaGetLastError();
}

cudaError_t launch_chunk_dense_flags(const int32_t* ids, int B, int S, int q0, int Lq, int k0, int Lk, int32_t* flags,
                                     cudaStream_t st) {
  chunk_dense_flags_kernel<<<1, kScanThreads, 0, st>>>(ids, B, S, q0, Lq, k0, Lk, flags);
  return cudaGetLastError();
}
cudaError_t launch_pad_fixup(void* out, float* lse, const int32_t* qids, int B, int Lq, int Hq, int Dv,
                             int64_t o_sb, int64_t o_ss, int64_t o_sh, int64_t l_sb, int64_t l_sh, cudaStream_t st) {
  pad_fixup_kernel<<<grid_for((int64_t)B * Lq * 32, 256), 256, 0, st>>>(static_cast<uint16_t*>(out), lse, qids, B, Lq, Hq, Dv, o_sb, o_ss,
                                                                        o_sh, l_sb, l_sh);
  return cudaGetLastError();
}

cudaError_t launch_lse_merge(const void* o1, const float* l1, const void* o2, const float* l2, float* of, void* ob,
                             float* l, int T, int H, int D, int f16, cudaStream_t st) {
  const int grid = grid_for((int64_t)T * H * (D / 8), 256);
  if (f16)
    lse_merge_kernel<__half><<<grid, 256, 0, st>>>(static_cast<const __half*>(o1), l1, static_cast<const __half*>(o2),
                                                   l2, of, static_cast<__half*>(ob), l, T, H, D);
  else
    lse_merge_kernel<__nv_bfloat16><<<grid, 256, 0, st>>>(static_cast<const __nv_bfloat16*>(o1), l1,
                                                          static_cast<const __nv_bfloat16*>(o2), l2, of,
                                                          static_cast<__nv_bfloat16*>(ob), l, T, H, D);
  return cudaGetLastError();
}

cudaError_t launch_bwd_prep(const SegInfo& g, int G, int Hkv, int split_target, const BwdSchedule& sc, int* status,
                            const void* dout, int64_t d_sb, int64_t d_ss, int64_t d_sh, const void* out, int64_t o_sb,
                            int64_t o_ss, int64_t o_sh, float* delta, float* dq_acc, int Hq, int Dqk, int Dv, void* dk,
                            void* dv, int64_t k_sb, int64_t k_ss, int64_t k_sh, int64_t v_sb, int64_t v_ss,
                            int64_t v_sh, int f16, cudaStream_t st) {
  // One 1024-thread block per SM fits (the schedule block's registers and
  // shared memory), so the fill takes one wave beside it.
  const int64_t work = (int64_t)g.B * g.Sq * Hq * (Dqk + Dv) / 4;
  const int fill = min(grid_for(work, kScanThreads), 152 - 1);
  uint16_t* dk16 = static_cast<uint16_t*>(dk);
  uint16_t* dv16 = static_cast<uint16_t*>(dv);
  if (f16)
    bwd_prep_kernel<__half><<<1 + fill, kScanThreads, 0, st>>>(
        g, G, Hkv, split_target, sc.nctas, sc.items, sc.item_slot, sc.splits, sc.slot_cap, sc.n_items, sc.seg_prefix,
        sc.item_cap, status, static_cast<const __half*>(dout), d_sb, d_ss, d_sh, static_cast<const __half*>(out), o_sb,
        o_ss, o_sh, delta, dq_acc, Hq, Dqk, Dv, dk16, dv16, k_sb, k_ss, k_sh, v_sb, v_ss, v_sh);
  else
    bwd_prep_kernel<__nv_bfloat16><<<1 + fill, kScanThreads, 0, st>>>(
        g, G, Hkv, split_target, sc.nctas, sc.items, sc.item_slot, sc.splits, sc.slot_cap, sc.n_items, sc.seg_prefix,
        sc.item_cap, status, static_cast<const __nv_bfloat16*>(dout), d_sb, d_ss, d_sh,
        static_cast<const __nv_bfloat16*>(out), o_sb, o_ss, o_sh, delta, dq_acc, Hq, Dqk, Dv, dk16, dv16, k_sb, k_ss,
        k_sh, v_sb, v_ss, v_sh);
  return cudaGetLastError();
}
cudaError_t launch_cross_segments(const int32_t* ids, int B, int S, int q0, int Lq, int k0, int Lk, int32_t* cu_q,
                                  int32_t* cu_k, int32_t* dev_meta, cudaStream_t st) {
  cudaError_t e = cudaMemsetAsync(dev_meta, 0, 3 * sizeof(int32_t), st);
  if (e != cudaSuccess) return e;
  cross_segments_kernel<<<B, kScanThreads, 0, st>>>(ids, B, S, q0, Lq, k0, Lk, cu_q, cu_k, dev_meta);
  return cudaGetLastError();
}
cudaError_t launch_lse_merge_live(float* o_acc, void* o_run, float* l_acc, const void* o_new, const float* l_new,
                                  const int32_t* cu_q, const int32_t* cu_k, const int32_t* dev_meta, int nseg, int T,
                                  int H, int D, int f16, cudaStream_t st) {
  const int grid = grid_for((int64_t)T * 32, 256);
  auto go = [&](auto kern, auto* run, auto* onew) {
    kern<<<grid, 256, 0, st>>>(o_acc, run, l_acc, onew, l_new, cu_q, cu_k, dev_meta, nseg, T, H, D);
  };
  if (f16) {
    __half* run = static_cast<__half*>(o_run);
    const __half* onew = static_cast<const __half*>(o_new);
    if (o_acc) go(lse_merge_live_kernel<__half, true>, run, onew);
    else go(lse_merge_live_kernel<__half, false>, run, onew);
  } else {
    __nv_bfloat16* run = static_cast<__nv_bfloat16*>(o_run);
    const __nv_bfloat16* onew = static_cast<const __nv_bfloat16*>(o_new);
    if (o_acc) go(lse_merge_live_kernel<__nv_bfloat16, true>, run, onew);
    else go(lse_merge_live_kernel<__nv_bfloat16, false>, run, onew);
  }
  return cudaGetLastError();
}
cudaError_t launch_grad_add_live(void* dst, const void* src, const int32_t* cu_q, const int32_t* cu_k,
                                 const int32_t* dev_meta, int nseg, int T, int H, int D, int f16, cudaStream_t st) {
  const int grid = grid_for((int64_t)T * 32, 256);
  if (f16)
    grad_add_live_kernel<__half><<<grid, 256, 0, st>>>(static_cast<__half*>(dst), static_cast<const __half*>(src), cu_q,
                                                       cu_k, dev_meta, nseg, T, H, D);
  else
    grad_add_live_kernel<__nv_bfloat16><<<grid, 256, 0, st>>>(static_cast<__nv_bfloat16*>(dst),
                                                              static_cast<const __nv_bfloat16*>(src), cu_q, cu_k,
                                                              dev_meta, nseg, T, H, D);
  return cudaGetLastError();
}
cudaError_t launch_bwd_convert(const float* dq_acc, void* dq, bool have_q, int B, int Sq, int Hq, int Dqk,
                               int64_t q_sb, int64_t q_ss, int64_t q_sh, const SegInfo& g, const BwdSchedule* sc,
                               const float* pk, const float* pv, void* dk, void* dv, int Hkv, int Dv, int64_t k_sb,
                               int64_t k_ss, int64_t k_sh, int64_t v_sb, int64_t v_ss, int64_t v_sh, float scale,
                               int f16, cudaStream_t st) {
  const int64_t nq = have_q ? (int64_t)B * Sq : 0;
  // Cut tiles: at most slot_cap / 2 of them (each has two slots or more).
  const int64_t split_rows = sc ? (int64_t)(sc->slot_cap / 2) * Hkv * kBN : 0;
  const int64_t rows = nq + split_rows;
  if (rows == 0) return cudaSuccess;
  const int64_t work = rows * 32;  // a warp per row
  const int4* splits = sc ? sc->splits : nullptr;
  const int* n_split = sc ? sc->n_items + 2 : nullptr;
  if (f16)
    bwd_convert_kernel<__half><<<grid_for(work, 256), 256, 0, st>>>(
        dq_acc, static_cast<__half*>(dq), nq, Sq, Hq, Dqk, q_sb, q_ss, q_sh, g, splits, n_split, pk, pv,
        static_cast<__half*>(dk), static_cast<__half*>(dv), Hkv, Dv, k_sb, k_ss, k_sh, v_sb, v_ss, v_sh, scale);
  else
    bwd_convert_kernel<__nv_bfloat16><<<grid_for(work, 256), 256, 0, st>>>(
        dq_acc, static_cast<__nv_bfloat16*>(dq), nq, Sq, Hq, Dqk, q_sb, q_ss, q_sh, g, splits, n_split, pk, pv,
        static_cast<__nv_bfloat16*>(dk), static_cast<__nv_bfloat16*>(dv), Hkv, Dv, k_sb, k_ss, k_sh, v_sb, v_ss,
        v_sh, scale);
  return cudaGetLastError();
}

namespace {

// Check of the bounded pipeline wait: warp 0 waits on an mbarrier that expects
// one arrival, which warp 1 makes only when `arrive` is set. Without it the
// wait runs out after limit_ns, records kStatusTimeout in the status word and
// the kernel returns, as every pipeline wait in the attention kernels does.
__global__ void __launch_bounds__(64, 1) wait_check_kernel(int arrive, uint64_t limit_ns, int* status) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x >= 32) {
    if (arrive && threadIdx.x == 32) mbar_arrive(&bar);
    return;
  }
  const Ctl c{status, limit_ns, &abort_flag};
  wait_bar(&bar, 0, c);
}

}  // namespace

cudaError_t launch_wait_check(int arrive, uint64_t limit_ns, int* status, cudaStream_t st) {
  wait_check_kernel<<<1, 64, 0, st>>>(arrive, limit_ns, status);
  return cudaGetLastError();
}

}  // namespace psf

// common.cuh -- parameter blocks, bounded pipeline waits and segment/tile
// arithmetic shared by the attention kernels.
#pragma once

#include <math_constants.h>
#include <stdint.h>

#include "ptx.cuh"

namespace psf {

constexpr int kBM = 128;  // query rows per tile (TMEM lanes)
constexpr int kBN = 128;  // key rows per tile
constexpr int kChunkBytes = 16384;  // one TMA box: 128 rows x 64 bf16, 128-byte swizzled

// Status codes mirrored from the public header.
constexpr int kStatusDeviceArgs = -4;
constexpr int kStatusTimeout = -5;

// Segment description as the kernels see it. Rows are flattened (b * S + s);
// a null cu array means "one segment per batch row" (dense attention).
struct SegInfo {
  const int32_t* cu_q;
  const int32_t* cu_k;
  const int32_t* dev_meta;  // nullable {nseg, max_q, max_k}
  int nseg;                 // count, or the capacity when dev_meta is given
  int max_q, max_k;
  int B, Sq, Sk;            // batches and rows per batch of the q / k tensors
  int causal;
  int window;               // > 0: left window counting the current token
  int qrows = kBM;          // query rows per forward tile (fewer when query heads are packed into one tile)
};

__device__ __forceinline__ int seg_count(const SegInfo& g) {
  if (!g.dev_meta) return g.nseg;
  int n = g.dev_meta[0];
  return n < 0 ? 0 : (n > g.nseg ? g.nseg : n);
}
__device__ __forceinline__ int cu_q_at(const SegInfo& g, int s) { return g.cu_q ? g.cu_q[s] : s * g.Sq; }
__device__ __forceinline__ int cu_k_at(const SegInfo& g, int s) { return g.cu_k ? g.cu_k[s] : s * g.Sk; }

// Keys [lo, hi) (segment-local) that some query of rows [i0, i0 + rows) can see.
__device__ __forceinline__ void kv_range_for_q_tile(int m, int n, int i0, int causal, int window, int& lo, int& hi,
                                                    int rows = kBM) {
  int i1 = min(i0 + rows, m);
  int delta = n - m;
  hi = causal ? min(n, i1 + delta) : n;
  lo = window > 0 ? max(0, i0 + delta - window + 1) : 0;
  if (hi < lo) hi = lo;
}
// Queries [lo, hi) (segment-local) that some key of rows [j0, j0 + kBN) is seen by.
__device__ __forceinline__ void q_range_for_kv_tile(int m, int n, int j0, int causal, int window, int& lo, int& hi) {
  int j1 = min(j0 + kBN, n);
  int delta = n - m;
  lo = causal ? max(0, j0 - delta) : 0;
  hi = window > 0 ? min(m, j1 - 1 - delta + window) : m;
  if (hi < lo) hi = lo;
}
__device__ __forceinline__ int ceil_div(int a, int b) { return (a + b - 1) / b; }

// Softcapped logit in log2 units, c * log2(e) * tanh(scale * s / c), for a raw
// score s = q . k, from tanh(u) = 1 - 2 / (e^(2u) + 1) with k1 = 2 * scale *
// log2(e) / c and c2 = c * log2(e) (the saturated ends come out as +-c2 exactly).
// A masked score (-inf) stays -inf.
__device__ __forceinline__ float softcap_log2(float s, float k1, float c2) {
  const float e = ex2_approx(s * k1);
  const float y = fmaf(rcp_approx(e + 1.f), -2.f * c2, c2);
  return s == -CUDART_INF_F ? -CUDART_INF_F : y;
}

// Static work assignment over a heaviest-first list: in round i CTA b takes
// item i * G + b when i is even and i * G + (G - 1 - b) when i is odd (G CTAs),
// so each CTA's heavy and light items pair up and the CTAs' sums stay close.
__device__ __forceinline__ int snake_item(int i) {
  const int g = (int)gridDim.x, b = (int)blockIdx.x;
  return i * g + ((i & 1) ? g - 1 - b : b);
}

// Compile-time flag for element passes that exist in a masked and an unmasked
// form (mask arithmetic inside the common, unmasked loop costs throughput even
// when it never fires).
template <bool B>
struct MaskTag {
  static constexpr bool value = B;
};

// Pipeline control: every wait is bounded. A wait that runs out records
// kStatusTimeout, raises the CTA-wide abort flag and returns false; the other
// roles notice the flag at their next wait and wind down, so the CTA always
// reaches its final barrier, drains its own asynchronous work and frees TMEM.
struct Ctl {
  int* status;
  uint64_t limit_ns;
  volatile int* abort_flag;  // shared memory
};

__device__ __forceinline__ bool wait_bar(uint64_t* bar, uint32_t parity, const Ctl& c) {
  if (mbar_test(bar, parity)) return true;
  uint64_t t0 = globaltimer_ns();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 16; ++i)
      if (mbar_test_sleep(bar, parity, 20000)) return true;
    if (*c.abort_flag) return false;
    if (globaltimer_ns() - t0 > c.limit_ns) {
      atomicCAS(c.status, 0, kStatusTimeout);
      *c.abort_flag = 1;
      return false;
    }
  }
}
// Drain-only wait used while winding down after an abort: bounded, no flag.
__device__ __forceinline__ void wait_bar_drain(uint64_t* bar, uint32_t parity, uint64_t limit_ns) {
  uint64_t t0 = globaltimer_ns();
  while (!mbar_test(bar, parity))
    if (globaltimer_ns() - t0 > limit_ns) return;
}

__device__ __forceinline__ void record_status(int* status, int code) { atomicCAS(status, 0, code); }

// Byte offset of 16-byte granule g (0..7) of row r inside a 128-byte-swizzled
// chunk of 128-byte rows (the layout TMA writes with CU_TENSOR_MAP_SWIZZLE_128B).
__device__ __forceinline__ uint32_t sw128_offset(int r, int g) { return (uint32_t)(r * 128 + ((g ^ (r & 7)) << 4)); }

}  // namespace psf

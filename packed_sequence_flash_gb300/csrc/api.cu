// api.cu -- the C ABI declared in include/psf.h: argument validation, workspace
// carving, tensor-map construction and kernel launches. Nothing here computes
// attention; every step runs in the kernels of fwd.cu, bwd.cu and aux.cu.
#include <math.h>
#include <stdarg.h>
#include <stdio.h>
#include <stdlib.h>

#include <mutex>
#include <string>
#include <vector>

#include "psf.h"
#include "bwd.cuh"
#include "fwd.cuh"
#include "launch.h"
#include "tmap.h"

using namespace psf;

namespace {

thread_local std::string g_last_error = "no error";

int fail(int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return code;
}

int cuda_fail(cudaError_t e, const char* where) {
  return fail(PSF_ECUDA, "%s: %s", where, cudaGetErrorString(e));
}

uint64_t initial_wait_limit() {
  const char* s = getenv("PSF_WAIT_LIMIT_NS");
  if (s && *s) {
    unsigned long long v = strtoull(s, nullptr, 10);
    if (v > 0) return v;
  }
  return 2000000000ull;
}
uint64_t g_wait_limit_ns = initial_wait_limit();

// Per-device status word the kernels record faults in (first fault wins).
__device__ int g_psf_status;

constexpr int kMaxDevices = 64;
struct DeviceInfo {
  bool ready = false;
  int sms = 0;
  int major = 0, minor = 0;
  int* status = nullptr;
};
DeviceInfo g_dev[kMaxDevices];
std::mutex g_dev_mu;

int device_info(DeviceInfo** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return fail(PSF_EUNSUPPORTED, "device index %d out of range", dev);
  std::lock_guard<std::mutex> lk(g_dev_mu);
  DeviceInfo& d = g_dev[dev];
  if (!d.ready) {
    if ((e = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&d.major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&d.minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess)
      return cuda_fail(e, "cudaDeviceGetAttribute");
    void* p = nullptr;
    if ((e = cudaGetSymbolAddress(&p, g_psf_status)) != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress");
    d.status = static_cast<int*>(p);
    d.ready = true;
  }
  if (!(d.major == 10 && d.minor == 3))
    return fail(PSF_EUNSUPPORTED, "device compute capability %d.%d; the library is compiled for sm_103a", d.major, d.minor);
  *out = &d;
  return PSF_OK;
}

// Optional event pairs around the main kernels (profiling only).
struct TimedLaunch {
  int kind;
  cudaEvent_t start, stop;
};
std::mutex g_timing_mu;
bool g_timing_on = false;
std::vector<TimedLaunch> g_timed;

// Inside a stream capture the record becomes an event-record node of the
// graph (external flag), so every replay of the graph re-records the pair and
// the kernel's time can be read after each replay.
void record_timing_event(cudaEvent_t ev, cudaStream_t st) {
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(st, &cs) == cudaSuccess && cs == cudaStreamCaptureStatusActive)
    cudaEventRecordWithFlags(ev, st, cudaEventRecordExternal);
  else
    cudaEventRecord(ev, st);
}

bool timing_begin(int kind, cudaStream_t st, TimedLaunch* t) {
  std::lock_guard<std::mutex> lk(g_timing_mu);
  if (!g_timing_on) return false;
  t->kind = kind;
  if (cudaEventCreate(&t->start) != cudaSuccess) return false;
  if (cudaEventCreate(&t->stop) != cudaSuccess) {
    cudaEventDestroy(t->start);
    return false;
  }
  record_timing_event(t->start, st);
  return true;
}
void timing_end(TimedLaunch* t, cudaStream_t st) {
  record_timing_event(t->stop, st);
  std::lock_guard<std::mutex> lk(g_timing_mu);
  g_timed.push_back(*t);
}
void timing_clear_locked() {
  for (auto& t : g_timed) {
    cudaEventDestroy(t.start);
    cudaEventDestroy(t.stop);
  }
  g_timed.clear();
}

constexpr size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

bool supported_dims(int dqk, int dv) {
  return (dqk == 64 && dv == 64) || (dqk == 128 && dv == 128) || (dqk == 192 && dv == 128) ||
         (dqk == 512 && dv == 512);
}

// Element strides (batch, row, head) of a [rows, H, D] (THD) or [B, H, S, D]
// (BHSD) tensor, and of the matching lse ([H, rows] or [B, H, S]).
struct View {
  int64_t sb, ss, sh;
};
View tensor_view(int layout, int S, int H, int D) {
  if (layout == PSF_LAYOUT_THD) return View{(int64_t)S * H * D, (int64_t)H * D, (int64_t)D};
  return View{(int64_t)H * S * D, (int64_t)D, (int64_t)S * D};
}
View lse_view(int layout, int S, int H) {
  if (layout == PSF_LAYOUT_THD) return View{(int64_t)H * S, 1, (int64_t)S};
  return View{(int64_t)H * S, 1, (int64_t)S};
}

// Tensor idx of a call: its element strides from the caller's (batch, head,
// row) triple strides[3 idx .. 3 idx + 2], or the layout's contiguous strides
// when strides is NULL. A dimension of extent 1 is never stepped over and keeps
// its packed stride. Other strides must be positive multiples of 8 elements
// (16 bytes: the TMA global-stride rule, and the kernels' 16-byte vector
// accesses) below 2^38; an output's view must not overlap itself.
int strided_view(const int64_t* strides, int idx, const char* name, int layout, int B, int S, int H, int D,
                 bool output, View* v) {
  *v = tensor_view(layout, S, H, D);
  if (!strides) return PSF_OK;
  const int64_t* t = strides + 3 * idx;
  const int64_t ext[3] = {layout == PSF_LAYOUT_THD ? 1 : B, H, S};
  int64_t st[3] = {v->sb, v->sh, v->ss};
  static const char* dim_name[3] = {"batch", "head", "row"};
  for (int i = 0; i < 3; ++i) {
    if (ext[i] <= 1) continue;
    if (t[i] <= 0 || t[i] % 8 != 0 || t[i] >= ((int64_t)1 << 38))
      return fail(PSF_EINVAL, "%s: %s stride %lld must be a positive multiple of 8 elements below 2^38", name,
                  dim_name[i], (long long)t[i]);
    st[i] = t[i];
  }
  if (output) {
    // Dimensions by increasing stride: each must step past everything the
    // smaller ones (and the contiguous head dim) cover.
    int ord[3] = {0, 1, 2};
    for (int a = 0; a < 3; ++a)
      for (int b = a + 1; b < 3; ++b)
        if (st[ord[b]] < st[ord[a]]) {
          const int x = ord[a];
          ord[a] = ord[b];
          ord[b] = x;
        }
    int64_t span = D;
    for (int i = 0; i < 3; ++i) {
      const int d = ord[i];
      if (ext[d] <= 1) continue;
      if (st[d] < span) return fail(PSF_EINVAL, "%s: the strided view overlaps itself (an output must not)", name);
      span += st[d] * (ext[d] - 1);
    }
  }
  v->sb = st[0];
  v->sh = st[1];
  v->ss = st[2];
  return PSF_OK;
}

struct FwdWorkspace {
  int* n_items;
  int* seg_prefix;
  int2* items;
  int item_cap;
};
// Bytes of the forward workspace: the 256-byte header (item count, work
// counter), the per-segment tile prefix and the (segment, tile) item list;
// qrows: query rows per tile (kBM, or fewer when query heads share a tile).
constexpr int64_t fwd_item_cap(int64_t rows, int nseg, int qrows) { return (rows + qrows - 1) / qrows + nseg + 1; }
constexpr size_t fwd_ws_bytes(int64_t rows, int nseg, int qrows) {
  return 256 + align256(sizeof(int) * (size_t)(nseg + 2)) +
         align256(sizeof(int2) * (size_t)fwd_item_cap(rows, nseg, qrows));
}
size_t fwd_ws_layout(int64_t rows, int nseg, FwdWorkspace* w, void* base, int qrows = kBM) {
  const int64_t cap = fwd_item_cap(rows, nseg, qrows);
  size_t off = 256;
  size_t prefix_off = off;
  off += align256(sizeof(int) * (size_t)(nseg + 2));
  size_t items_off = off;
  off += align256(sizeof(int2) * (size_t)cap);
  if (w && base) {
    char* b = static_cast<char*>(base);
    w->n_items = reinterpret_cast<int*>(b);
    w->seg_prefix = reinterpret_cast<int*>(b + prefix_off);
    w->items = reinterpret_cast<int2*>(b + items_off);
    w->item_cap = (int)cap;
  }
  return off;
}

struct BwdWorkspace {
  BwdSchedule sc;
  float* delta;
  float* dq_acc;
  float* pk;  // dK partial-sum slots [slot][Hkv][128][Dqk] (head dims <= 128)
  float* pv;  // dV partial-sum slots [slot][Hkv][128][Dv]
};
// Heavy key tiles are split into at most this many sub-ranges' worth of work
// per SM (see bwd_schedule_body); the item capacity follows from it.
constexpr int kSplitPerSm = 2;
// Partial-sum slots: a cut tile has more steps than the cap per sub-range,
// steps * Hkv / (kSplitPerSm * sms) or more, and fewer than twice its steps
// over that cap in sub-ranges, so all cut tiles' sub-ranges of one KV head
// number fewer than 2 * kSplitPerSm * sms / Hkv. The last-wave fill cuts at
// most ceil(sms / (2 Hkv)) more tiles, into four each.
constexpr int bwd_wave_fill_tiles(int sms, int Hkv) { return sms / (2 * Hkv) + 1; }
constexpr int bwd_slot_cap(int sms, int Hkv) {
  return 2 * kSplitPerSm * sms / Hkv + 2 + 4 * bwd_wave_fill_tiles(sms, Hkv);
}
size_t bwd_ws_layout(int64_t q_rows, int64_t k_rows, int nseg, int Hq, int Hkv, int Dqk, int Dv, int sms,
                     BwdWorkspace* w, void* base) {
  const int64_t cap = (k_rows + kBN - 1) / kBN + nseg + (int64_t)kSplitPerSm * sms + 2 +
                      3 * (int64_t)bwd_wave_fill_tiles(sms, Hkv);
  // Only the head-dim <= 128 kernel cuts key tiles.
  const int slot_cap = (Dqk <= 128 && Dv <= 128) ? bwd_slot_cap(sms, Hkv) : 0;
  size_t off = 256;
  const size_t prefix_off = off;
  off += align256(sizeof(int) * (size_t)(nseg + 2));
  const size_t items_off = off;
  off += align256(sizeof(int4) * (size_t)cap);
  const size_t slot_off = off;
  off += align256(sizeof(int) * (size_t)cap);
  const size_t splits_off = off;
  off += align256(sizeof(int4) * (size_t)(slot_cap / 2 + 1));
  const size_t delta_off = off;
  off += align256(sizeof(float) * (size_t)Hq * (size_t)q_rows);
  const size_t dq_off = off;
  off += align256(sizeof(float) * (size_t)q_rows * Hq * Dqk);
  const size_t pk_off = off;
  off += align256(sizeof(float) * (size_t)slot_cap * Hkv * kBN * Dqk);
  const size_t pv_off = off;
  off += align256(sizeof(float) * (size_t)slot_cap * Hkv * kBN * Dv);
  if (w && base) {
    char* b = static_cast<char*>(base);
    w->sc.n_items = reinterpret_cast<int*>(b);
    w->sc.seg_prefix = reinterpret_cast<int*>(b + prefix_off);
    w->sc.items = reinterpret_cast<int4*>(b + items_off);
    w->sc.item_slot = reinterpret_cast<int*>(b + slot_off);
    w->sc.splits = reinterpret_cast<int4*>(b + splits_off);
    w->sc.item_cap = (int)cap;
    w->sc.slot_cap = slot_cap;
    w->sc.nctas = sms;
    w->delta = reinterpret_cast<float*>(b + delta_off);
    w->dq_acc = reinterpret_cast<float*>(b + dq_off);
    w->pk = reinterpret_cast<float*>(b + pk_off);
    w->pv = reinterpret_cast<float*>(b + pv_off);
  }
  return off;
}
// The workspace size query must not depend on the device; size it for the
// largest SM count this library targets.
constexpr int kMinPackedRows = kBM / 16;  // tile rows with 16 query heads packed into one tile
constexpr int kMaxSms = 160;

int check_common(int layout, int B, int Sq, int Sk, int Hq, int Hkv, int Dqk, int Dv, float scale, int32_t window,
                 int nseg) {
  if (layout != PSF_LAYOUT_THD && layout != PSF_LAYOUT_BHSD) return fail(PSF_EINVAL, "unknown layout %d", layout);
  if (B < 1 || Sq < 0 || Sk < 0) return fail(PSF_EINVAL, "bad sizes B=%d Sq=%d Sk=%d", B, Sq, Sk);
  if (layout == PSF_LAYOUT_THD && B != 1) return fail(PSF_EINVAL, "packed THD layout takes B = 1 (got %d)", B);
  if ((int64_t)B * Sq > 0x7fffffff || (int64_t)B * Sk > 0x7fffffff)
    return fail(PSF_EINVAL, "more than 2^31 - 1 rows");
  if (Hq < 1 || Hkv < 1 || Hq % Hkv != 0) return fail(PSF_EINVAL, "Hq=%d must be a positive multiple of Hkv=%d", Hq, Hkv);
  if (!supported_dims(Dqk, Dv))
    return fail(PSF_EUNSUPPORTED, "head dims (Dqk=%d, Dv=%d) not in {(64,64),(128,128),(192,128),(512,512)}", Dqk, Dv);
  if (window == 0) return fail(PSF_EINVAL, "window_left == 0 is undefined (use > 0, or < 0 for none)");
  if (!(scale > 0.f) || !isfinite(scale)) return fail(PSF_EINVAL, "scale must be finite and > 0 (got %g)", (double)scale);
  if (nseg < 0) return fail(PSF_EINVAL, "nseg < 0");
  return PSF_OK;
}

int check_softcap(float softcap) {
  if (!(softcap >= 0.f) || !isfinite(softcap)) return fail(PSF_EINVAL, "softcap must be finite and >= 0 (got %g)", (double)softcap);
  return PSF_OK;
}

int check_dtype(int dtype) {
  if (dtype != PSF_DTYPE_BF16 && dtype != PSF_DTYPE_F16) return fail(PSF_EINVAL, "unknown dtype %d", dtype);
  return PSF_OK;
}

// TMA view of a 16-bit (bf16 or fp16) tensor; a box is box_d x box_s rows x box_h heads.
int make_map16(CUtensorMap* m, const void* base, int D, int S, int H, int B, const View& v, int box_d, int dtype,
               int box_s = kBM, int box_h = 1, CUtensorMapSwizzle swz = CU_TENSOR_MAP_SWIZZLE_128B) {
  int rc = make_tmap_4d(m, dtype == PSF_DTYPE_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                        2, base, D, S, H, B, v.ss, v.sh, v.sb, box_d, box_s, swz, box_h);
  if (rc) return fail(PSF_ECUDA, "cuTensorMapEncodeTiled failed (%d) for a [%d,%d,%d,%d] view", rc, B, H, S, D);
  return PSF_OK;
}

int attn_fwd_impl(const void* q, const void* k, const void* v, void* out, float* lse, const int32_t* cu_q,
                  const int32_t* cu_k, const int32_t* dev_meta, int nseg, int max_q, int max_k, int layout, int dtype,
                  int B,
                  int Sq, int Sk, int Hq, int Hkv, int Dqk, int Dv, float scale, int causal, int32_t window, void* ws,
                  size_t ws_bytes, void* stream, int flags = 0, float softcap = 0.f, const int64_t* strides = nullptr) {
  int rc = check_common(layout, B, Sq, Sk, Hq, Hkv, Dqk, Dv, scale, window, nseg);
  if (rc) return rc;
  View vq, vk, vv, vo;
  if ((rc = strided_view(strides, 0, "q", layout, B, Sq, Hq, Dqk, false, &vq)) ||
      (rc = strided_view(strides, 1, "k", layout, B, Sk, Hkv, Dqk, false, &vk)) ||
      (rc = strided_view(strides, 2, "v", layout, B, Sk, Hkv, Dv, false, &vv)) ||
      (rc = strided_view(strides, 3, "out", layout, B, Sq, Hq, Dv, true, &vo)))
    return rc;
  if ((rc = check_softcap(softcap))) return rc;
  if ((rc = check_dtype(dtype))) return rc;
  if (flags & ~PSF_FWD_PACK_GQA) return fail(PSF_EINVAL, "unknown forward flags 0x%x", flags);
  // Packed query heads: the G = Hq / Hkv heads of a KV head share one tile of
  // 128 / G rows each (the two-CTA kernel, head dims 64 and 128, G in 2..16
  // dividing 128); other shapes run one head per tile, with the same result.
  const int G = Hq / Hkv;
  const int pack = ((flags & PSF_FWD_PACK_GQA) && G > 1 && G <= 16 && kBM % G == 0 && Dqk == Dv &&
                    (Dqk == 64 || Dqk == 128))
                       ? G
                       : 1;
  // Dqk = 192, Dv = 128 runs two 128-row halves of a 256-row item side by side
  // (attn_fwd_pair_kernel); the schedule then lists 256-row tiles.
  const bool pair = Dqk == 192 && Dv == 128;
  const int qrows = pair ? 2 * kBM : kBM / pack;
  const int64_t q_rows = (int64_t)B * Sq, k_rows = (int64_t)B * Sk;
  if (q_rows == 0) return PSF_OK;
  if (!q || !out || !lse || (k_rows > 0 && (!k || !v))) return fail(PSF_EINVAL, "null tensor pointer");
  if (!aligned16(q) || !aligned16(out) || (k_rows > 0 && (!aligned16(k) || !aligned16(v))))
    return fail(PSF_EINVAL, "tensor base pointers must be 16-byte aligned");
  if ((cu_q == nullptr) != (cu_k == nullptr)) return fail(PSF_EINVAL, "cu_q and cu_k must both be given");
  const size_t need = fwd_ws_layout(q_rows, nseg, nullptr, nullptr, qrows);
  if (!ws || ws_bytes < need) return fail(PSF_EWORKSPACE, "forward workspace needs %zu bytes (got %zu)", need, ws_bytes);
  DeviceInfo* dev = nullptr;
  if ((rc = device_info(&dev))) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);

  FwdWorkspace w;
  fwd_ws_layout(q_rows, nseg, &w, ws, qrows);
  SegInfo g{cu_q, cu_k, dev_meta, nseg, max_q, max_k, B, Sq, Sk, causal ? 1 : 0, window > 0 ? (int)window : 0, qrows};
  const View vl = lse_view(layout, Sq, Hq);
  if (k_rows == 0) {
    // No keys at all: every query row sees none, so out = 0 and lse = -inf
    // everywhere. The preparation kernel writes exactly that for the rows past
    // the last segment; run it with no segments and launch no attention kernel
    // (which would hold key-side tensor maps over no memory).
    SegInfo none = g;
    none.cu_q = none.cu_k = nullptr;
    none.dev_meta = nullptr;
    none.nseg = 0;
    cudaError_t e0 = launch_fwd_prep(none, w.items, w.n_items, w.seg_prefix, w.item_cap, dev->status, out, vo.sb,
                                     vo.ss, vo.sh, lse, vl.sb, vl.sh, Hq, Dv, st);
    return e0 == cudaSuccess ? PSF_OK : cuda_fail(e0, "forward preparation launch");
  }
  cudaError_t e = launch_fwd_prep(g, w.items, w.n_items, w.seg_prefix, w.item_cap, dev->status,
                                  out, vo.sb, vo.ss, vo.sh, lse, vl.sb, vl.sh, Hq, Dv, st);
  if (e != cudaSuccess) return cuda_fail(e, "forward preparation launch");

  FwdParams p;
  memset(&p, 0, sizeof(p));
  if ((rc = make_map16(&p.tm_q, q, Dqk, Sq, Hq, B, vq, 64, dtype, pair ? kBM : qrows, pack))) return rc;
  // The two-CTA kernel (head dims 64, 128) stores out in 32 x 32 boxes.
  if (Dqk == Dv && (Dv == 64 || Dv == 128) &&
      (rc = make_map16(&p.tm_o, out, Dv, Sq, Hq, B, vo, 32, dtype, 32, 1, CU_TENSOR_MAP_SWIZZLE_64B)))
    return rc;
  if (k_rows > 0) {
    if ((rc = make_map16(&p.tm_k, k, Dqk, Sk, Hkv, B, vk, 64, dtype))) return rc;
    if ((rc = make_map16(&p.tm_v, v, Dv, Sk, Hkv, B, vv, 64, dtype))) return rc;
  }
  p.seg = g;
  p.out = out;
  p.o_sb = vo.sb;
  p.o_ss = vo.ss;
  p.o_sh = vo.sh;
  p.lse = lse;
  p.l_sb = vl.sb;
  p.l_sh = vl.sh;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.pack = pack;
  p.dv_parts = Dv == 512 ? 2 : 1;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.softcap = softcap;
  p.items = w.items;
  p.n_items = w.n_items;
  p.work_next = w.n_items + 1;
  p.status = dev->status;
  p.limit_ns = g_wait_limit_ns;
  const int64_t max_work = (int64_t)w.item_cap * (Hq / pack) * p.dv_parts;
  TimedLaunch tl;
  const bool timed = timing_begin(0, st, &tl);
  e = launch_fwd(p, Dqk, Dv / p.dv_parts, dev->sms, max_work, dtype == PSF_DTYPE_F16, st);
  if (timed) timing_end(&tl, st);
  if (e != cudaSuccess) return cuda_fail(e, "forward launch");
  return PSF_OK;
}

int attn_bwd_impl(const void* dout, const void* q, const void* k, const void* v, const void* out, const float* lse,
                  void* dq, void* dk, void* dv, const int32_t* cu_q, const int32_t* cu_k, const int32_t* dev_meta,
                  int nseg, int max_q, int max_k, int layout, int dtype, int B, int Sq, int Sk, int Hq, int Hkv,
                  int Dqk, int Dv, float scale, int causal, int32_t window, void* ws, size_t ws_bytes, void* stream,
                  float softcap = 0.f, int flags = 0, const int64_t* strides = nullptr) {
  int rc = check_common(layout, B, Sq, Sk, Hq, Hkv, Dqk, Dv, scale, window, nseg);
  if (rc) return rc;
  // Tensor order of the strides array: q, k, v, out, dout, dq, dk, dv.
  View vq, vk, vv, vo, vdo, vdq, vdk, vdv;
  if ((rc = strided_view(strides, 0, "q", layout, B, Sq, Hq, Dqk, false, &vq)) ||
      (rc = strided_view(strides, 1, "k", layout, B, Sk, Hkv, Dqk, false, &vk)) ||
      (rc = strided_view(strides, 2, "v", layout, B, Sk, Hkv, Dv, false, &vv)) ||
      (rc = strided_view(strides, 3, "out", layout, B, Sq, Hq, Dv, false, &vo)) ||
      (rc = strided_view(strides, 4, "dout", layout, B, Sq, Hq, Dv, false, &vdo)) ||
      (rc = strided_view(strides, 5, "dq", layout, B, Sq, Hq, Dqk, true, &vdq)) ||
      (rc = strided_view(strides, 6, "dk", layout, B, Sk, Hkv, Dqk, true, &vdk)) ||
      (rc = strided_view(strides, 7, "dv", layout, B, Sk, Hkv, Dv, true, &vdv)))
    return rc;
  if ((rc = check_softcap(softcap))) return rc;
  if (flags & ~PSF_BWD_PACK_GQA) return fail(PSF_EINVAL, "unknown backward flags 0x%x", flags);
  if ((rc = check_dtype(dtype))) return rc;
  const int f16 = dtype == PSF_DTYPE_F16;
  if (bwd_smem_bytes(Dqk, Dv) < 0)
    return fail(PSF_EUNSUPPORTED, "backward for (Dqk=%d, Dv=%d) is not built", Dqk, Dv);
  const int64_t q_rows = (int64_t)B * Sq, k_rows = (int64_t)B * Sk;
  if (q_rows == 0 && k_rows == 0) return PSF_OK;
  const void* ptrs[] = {dout, q, out, dq};
  for (const void* x : ptrs)
    if (q_rows > 0 && (!x || !aligned16(x))) return fail(PSF_EINVAL, "null or unaligned query-side tensor");
  const void* kptrs[] = {k, v, dk, dv};
  for (const void* x : kptrs)
    if (k_rows > 0 && (!x || !aligned16(x))) return fail(PSF_EINVAL, "null or unaligned key-side tensor");
  if (q_rows > 0 && !lse) return fail(PSF_EINVAL, "null lse");
  if ((cu_q == nullptr) != (cu_k == nullptr)) return fail(PSF_EINVAL, "cu_q and cu_k must both be given");
  const size_t need = bwd_ws_layout(q_rows, k_rows, nseg, Hq, Hkv, Dqk, Dv, kMaxSms, nullptr, nullptr);
  if (!ws || ws_bytes < need) return fail(PSF_EWORKSPACE, "backward workspace needs %zu bytes (got %zu)", need, ws_bytes);
  DeviceInfo* dev = nullptr;
  if ((rc = device_info(&dev))) return rc;
  if (dev->sms > kMaxSms) return fail(PSF_EUNSUPPORTED, "more than %d SMs", kMaxSms);
  cudaStream_t st = static_cast<cudaStream_t>(stream);

  // Head dims up to 128 run the kernel that can cut heavy key tiles across
  // SMs, their sub-ranges' dK/dV partial sums added up by the convert.
  const bool accumulate = Dqk <= 128 && Dv <= 128;
  // Packed query heads: a step of the head-dim-<=-128 kernel takes the G = Hq / Hkv
  // query heads of its KV head, 128 / G rows each (G in {2, 4}, so that a dQ
  // read-out box of 32 rows stays inside one head; no softcap); other calls
  // take one head per step, with the same results.
  const int G = Hq / Hkv;
  const int pack = ((flags & PSF_BWD_PACK_GQA) && accumulate && (G == 2 || G == 4) && softcap == 0.f) ? G : 1;
  const int qrows = kBM / pack;
  BwdWorkspace w;
  bwd_ws_layout(q_rows, k_rows, nseg, Hq, Hkv, Dqk, Dv, dev->sms, &w, ws);
  SegInfo g{cu_q, cu_k, dev_meta, nseg, max_q, max_k, B, Sq, Sk, causal ? 1 : 0, window > 0 ? (int)window : 0, qrows};
  const View vl = lse_view(layout, Sq, Hq);
  if (q_rows == 0) {
    // No queries: every gradient is zero. The preparation kernel zeroes dK and
    // dV rows past the last segment; run it with no segments and without the
    // accumulators, and launch no attention kernel (which would hold
    // query-side tensor maps over no memory).
    SegInfo none = g;
    none.cu_q = none.cu_k = nullptr;
    none.dev_meta = nullptr;
    none.nseg = 0;
    cudaError_t e0 = launch_bwd_prep(none, Hq / Hkv, Hkv, 0, w.sc, dev->status, dout, vdo.sb, vdo.ss, vdo.sh, out,
                                     vo.sb, vo.ss, vo.sh, w.delta, w.dq_acc, Hq, Dqk, Dv, dk, dv, vdk.sb, vdk.ss,
                                     vdk.sh, vdv.sb, vdv.ss, vdv.sh, f16, st);
    return e0 == cudaSuccess ? PSF_OK : cuda_fail(e0, "backward preparation launch");
  }
  cudaError_t e = launch_bwd_prep(g, Hq / Hkv, Hkv, accumulate ? kSplitPerSm * dev->sms : 0, w.sc, dev->status, dout,
                                  vdo.sb, vdo.ss, vdo.sh, out, vo.sb, vo.ss, vo.sh, w.delta, w.dq_acc, Hq, Dqk, Dv, dk,
                                  dv, vdk.sb, vdk.ss, vdk.sh, vdv.sb, vdv.ss, vdv.sh, f16, st);
  if (e != cudaSuccess) return cuda_fail(e, "backward preparation launch");

  if (k_rows > 0) {
    BwdParams p;
    memset(&p, 0, sizeof(p));
    if (q_rows > 0) {
      if ((rc = make_map16(&p.tm_q, q, Dqk, Sq, Hq, B, vq, 64, dtype, qrows, pack))) return rc;
      if ((rc = make_map16(&p.tm_do, dout, Dv, Sq, Hq, B, vdo, 64, dtype, qrows, pack))) return rc;
      int r2 = make_tmap_4d(&p.tm_dq, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, w.dq_acc, Dqk, Sq, Hq, B, (int64_t)Hq * Dqk,
                            Dqk, (int64_t)Sq * Hq * Dqk, 32, 32, CU_TENSOR_MAP_SWIZZLE_128B);
      if (r2) return fail(PSF_ECUDA, "cuTensorMapEncodeTiled failed (%d) for the dQ accumulator", r2);
    }
    if (accumulate) {
      const int ns = w.sc.slot_cap;
      int r2 = make_tmap_4d(&p.tm_dk, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, w.pk, Dqk, kBN, Hkv, ns, Dqk,
                            (int64_t)kBN * Dqk, (int64_t)Hkv * kBN * Dqk, 32, 32, CU_TENSOR_MAP_SWIZZLE_128B);
      r2 |= make_tmap_4d(&p.tm_dv, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, w.pv, Dv, kBN, Hkv, ns, Dv,
                         (int64_t)kBN * Dv, (int64_t)Hkv * kBN * Dv, 32, 32, CU_TENSOR_MAP_SWIZZLE_128B);
      if (r2) return fail(PSF_ECUDA, "cuTensorMapEncodeTiled failed for the dK/dV partial-sum slots");
    }
    if ((rc = make_map16(&p.tm_k, k, Dqk, Sk, Hkv, B, vk, 64, dtype))) return rc;
    if ((rc = make_map16(&p.tm_v, v, Dv, Sk, Hkv, B, vv, 64, dtype))) return rc;
    p.seg = g;
    p.lse = lse;
    p.l_sb = vl.sb;
    p.l_sh = vl.sh;
    p.delta = w.delta;
    p.q_rows = (int)q_rows;
    p.dk = dk;
    p.k_sb = vdk.sb;
    p.k_ss = vdk.ss;
    p.k_sh = vdk.sh;
    p.dv = dv;
    p.v_sb = vdv.sb;
    p.v_ss = vdv.ss;
    p.v_sh = vdv.sh;
    p.Hq = Hq;
    p.Hkv = Hkv;
    p.scale = scale;
    p.scale_log2 = scale * 1.4426950408889634f;
    p.softcap = softcap;
    p.pack = pack;
    p.items = w.sc.items;
    p.item_slot = w.sc.item_slot;
    p.n_items = w.sc.n_items;
    p.work_next = w.sc.n_items + 1;
    p.status = dev->status;
    p.limit_ns = g_wait_limit_ns;
    TimedLaunch tl;
    const bool timed = timing_begin(1, st, &tl);
    e = launch_bwd(p, Dqk, Dv, dev->sms, w.sc.item_cap, f16, st);
    if (timed) timing_end(&tl, st);
    if (e != cudaSuccess) return cuda_fail(e, "backward launch");
  }
  e = launch_bwd_convert(w.dq_acc, dq, q_rows > 0, B, Sq, Hq, Dqk, vdq.sb, vdq.ss, vdq.sh, g,
                         accumulate && k_rows > 0 ? &w.sc : nullptr, w.pk, w.pv, dk, dv, Hkv, Dv, vdk.sb, vdk.ss,
                         vdk.sh, vdv.sb, vdv.ss, vdv.sh, scale, f16, st);
  if (e != cudaSuccess) return cuda_fail(e, "convert launch");
  return PSF_OK;
}

// Fixed scratch of psf_attn_varlen_fwd_noalloc: the forward's tile schedule
// (item count, per-segment tile prefix, (segment, tile) list) for up to
// PSF_NOALLOC_MAX_Q_ROWS query rows and PSF_NOALLOC_MAX_SEGMENTS segments.
constexpr size_t kNoAllocScratchBytes = fwd_ws_bytes(PSF_NOALLOC_MAX_Q_ROWS, PSF_NOALLOC_MAX_SEGMENTS, kBM);
static_assert(kNoAllocScratchBytes == 852736, "the header documents the scratch array's size");
static __device__ __align__(256) unsigned char g_noalloc_fwd_scratch[kNoAllocScratchBytes];

// Device address of the scratch array, looked up once per device with that
// device current (the host-side symbol is only a stand-in, never a device
// address).
void* g_noalloc_ptr[kMaxDevices];
std::mutex g_noalloc_mu;

int noalloc_scratch(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return fail(PSF_EUNSUPPORTED, "device index %d out of range", dev);
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  if (!g_noalloc_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress((void**)&p, g_noalloc_fwd_scratch);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(scratch)");
    g_noalloc_ptr[dev] = p;
  }
  *out = g_noalloc_ptr[dev];
  return PSF_OK;
}

}  // namespace

extern "C" {

const char* psf_last_error(void) { return g_last_error.c_str(); }

int psf_device_supported(void) {
  DeviceInfo* d = nullptr;
  return device_info(&d) == PSF_OK ? 1 : 0;
}

int psf_device_status(int clear) {
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceSynchronize");
  int v = 0;
  if ((e = cudaMemcpyFromSymbol(&v, g_psf_status, sizeof(int))) != cudaSuccess) return cuda_fail(e, "status read");
  if (clear) {
    int z = 0;
    if ((e = cudaMemcpyToSymbol(g_psf_status, &z, sizeof(int))) != cudaSuccess) return cuda_fail(e, "status clear");
  }
  if (v == PSF_EDEVICE_ARGS) return fail(v, "kernel-side validation rejected the segment arrays");
  if (v == PSF_ETIMEOUT) return fail(v, "a pipeline wait inside a kernel exceeded its limit");
  return v;
}

void psf_set_wait_limit_ns(uint64_t ns) { g_wait_limit_ns = ns > 0 ? ns : 1; }

int psf_check_pipeline_wait(int arrive, void* stream) {
  DeviceInfo* dev = nullptr;
  int rc = device_info(&dev);
  if (rc) return rc;
  cudaError_t e = launch_wait_check(arrive != 0, g_wait_limit_ns, dev->status, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PSF_OK : cuda_fail(e, "wait-check launch");
}

int psf_kernel_timing(int enable) {
  std::lock_guard<std::mutex> lk(g_timing_mu);
  if (enable) timing_clear_locked();
  g_timing_on = enable != 0;
  return PSF_OK;
}

int psf_kernel_times_ms(int kind, double* total_ms, int* launches) {
  if (!total_ms || !launches) return fail(PSF_EINVAL, "null output pointer");
  std::lock_guard<std::mutex> lk(g_timing_mu);
  double sum = 0.0;
  int n = 0;
  for (auto& t : g_timed) {
    if (t.kind != kind) continue;
    cudaError_t e = cudaEventSynchronize(t.stop);
    if (e != cudaSuccess) return cuda_fail(e, "cudaEventSynchronize");
    float ms = 0.f;
    if ((e = cudaEventElapsedTime(&ms, t.start, t.stop)) != cudaSuccess) return cuda_fail(e, "cudaEventElapsedTime");
    sum += ms;
    ++n;
  }
  *total_ms = sum;
  *launches = n;
  return PSF_OK;
}

size_t psf_attn_fwd_workspace_size(int64_t total_q_rows, int nseg) {
  if (total_q_rows < 0 || nseg < 0) return 0;
  // Large enough for the shortest tiles (packed query heads, up to kBM / 8 = 16 heads).
  return fwd_ws_layout(total_q_rows, nseg, nullptr, nullptr, kMinPackedRows);
}

size_t psf_attn_bwd_workspace_size(int64_t total_q_rows, int64_t total_k_rows, int nseg, int Hq, int Hkv, int Dqk,
                                   int Dv) {
  if (total_q_rows < 0 || total_k_rows < 0 || nseg < 0 || Hq < 1 || Hkv < 1 || Dqk < 1 || Dv < 1) return 0;
  return bwd_ws_layout(total_q_rows, total_k_rows, nseg, Hq, Hkv, Dqk, Dv, kMaxSms, nullptr, nullptr);
}

int psf_attn_varlen_fwd(const void* q, const void* k, const void* v, void* out, float* lse, const int32_t* cu_q,
                        const int32_t* cu_k, const int32_t* dev_meta, int nseg, int max_q, int max_k, int layout,
                        int dtype, int B, int Sq, int Sk, int Hq, int Hkv, int Dqk, int Dv, const int64_t* strides,
                        float scale, int causal, int32_t window_left, float softcap, int flags, void* workspace,
                        size_t ws_bytes, void* stream) {
  if (!cu_q || !cu_k) return fail(PSF_EINVAL, "varlen calls need cu_q and cu_k");
  return attn_fwd_impl(q, k, v, out, lse, cu_q, cu_k, dev_meta, nseg, max_q, max_k, layout, dtype, B, Sq, Sk, Hq, Hkv,
                       Dqk, Dv, scale, causal, window_left, workspace, ws_bytes, stream, flags, softcap, strides);
}

int psf_attn_varlen_fwd_noalloc(const void* q, const void* k, const void* v, void* out, float* lse,
                                const int32_t* cu_q, const int32_t* cu_k, const int32_t* dev_meta, int nseg,
                                int max_q, int max_k, int layout, int dtype, int B, int Sq, int Sk, int Hq, int Hkv,
                                int Dqk, int Dv, float scale, int causal, int32_t window_left, void* stream) {
  if (!cu_q || !cu_k) return fail(PSF_EINVAL, "varlen calls need cu_q and cu_k");
  if (B < 1 || Sq < 0 || nseg < 0) return fail(PSF_EINVAL, "bad sizes B=%d Sq=%d nseg=%d", B, Sq, nseg);
  if ((int64_t)B * Sq > PSF_NOALLOC_MAX_Q_ROWS)
    return fail(PSF_EINVAL, "no-allocation forward handles at most %d query rows (got %lld)", PSF_NOALLOC_MAX_Q_ROWS,
                (long long)B * Sq);
  if (nseg > PSF_NOALLOC_MAX_SEGMENTS)
    return fail(PSF_EINVAL, "no-allocation forward handles at most %d segments (got %d)", PSF_NOALLOC_MAX_SEGMENTS,
                nseg);
  void* scratch = nullptr;
  int rc = noalloc_scratch(&scratch);
  if (rc) return rc;
  return attn_fwd_impl(q, k, v, out, lse, cu_q, cu_k, dev_meta, nseg, max_q, max_k, layout, dtype, B, Sq, Sk, Hq, Hkv,
                       Dqk, Dv, scale, causal, window_left, scratch, kNoAllocScratchBytes, stream);
}

int psf_attn_varlen_bwd(const void* dout, const void* q, const void* k, const void* v, const void* out,
                        const float* lse, void* dq, void* dk, void* dv, const int32_t* cu_q, const int32_t* cu_k,
                        const int32_t* dev_meta, int nseg, int max_q, int max_k, int layout, int dtype, int B, int Sq,
                        int Sk, int Hq, int Hkv, int Dqk, int Dv, const int64_t* strides, float scale, int causal,
                        int32_t window_left, float softcap, int flags, void* workspace, size_t ws_bytes,
                        void* stream) {
  if (!cu_q || !cu_k) return fail(PSF_EINVAL, "varlen calls need cu_q and cu_k");
  return attn_bwd_impl(dout, q, k, v, out, lse, dq, dk, dv, cu_q, cu_k, dev_meta, nseg, max_q, max_k, layout, dtype, B,
                       Sq, Sk, Hq, Hkv, Dqk, Dv, scale, causal, window_left, workspace, ws_bytes, stream, softcap,
                       flags, strides);
}

int psf_attn_dense_fwd(const void* q, const void* k, const void* v, void* out, float* lse, int B, int Hq, int Hkv,
                       int Nq, int Nk, int Dqk, int Dv, const int64_t* strides, int dtype, float scale, int causal,
                       int32_t window_left, float softcap, int flags, void* workspace, size_t ws_bytes,
                       void* stream) {
  return attn_fwd_impl(q, k, v, out, lse, nullptr, nullptr, nullptr, B, Nq, Nk, PSF_LAYOUT_BHSD, dtype, B, Nq, Nk, Hq,
                       Hkv, Dqk, Dv, scale, causal, window_left, workspace, ws_bytes, stream, flags, softcap, strides);
}

int psf_attn_dense_bwd(const void* dout, const void* q, const void* k, const void* v, const void* out,
                       const float* lse, void* dq, void* dk, void* dv, int B, int Hq, int Hkv, int Nq, int Nk,
                       int Dqk, int Dv, const int64_t* strides, int dtype, float scale, int causal,
                       int32_t window_left, float softcap, int flags, void* workspace, size_t ws_bytes,
                       void* stream) {
  return attn_bwd_impl(dout, q, k, v, out, lse, dq, dk, dv, nullptr, nullptr, nullptr, B, Nq, Nk, PSF_LAYOUT_BHSD,
                       dtype, B, Nq, Nk, Hq, Hkv, Dqk, Dv, scale, causal, window_left, workspace, ws_bytes, stream,
                       softcap, flags, strides);
}

int psf_build_doc_segments(const int32_t* kv_doc_ids, int B, int Sk, int q_length, int q_global_start,
                           int32_t* cu_q, int32_t* cu_k, int capacity, int32_t* dev_meta, uint8_t* seg_is_pad,
                           int flags, void* stream) {
  if (flags & ~PSF_SEGMENTS_SKIP_PAD) return fail(PSF_EINVAL, "unknown builder flags 0x%x", flags);
  if (B < 1 || Sk < 0 || q_length < 0 || q_global_start < 0 || (int64_t)q_global_start + q_length > Sk)
    return fail(PSF_EINVAL, "need B >= 1 and 0 <= q_global_start <= q_global_start + q_length <= Sk");
  if ((int64_t)B * (Sk + 1) > 0x7fffffff) return fail(PSF_EINVAL, "too many rows");
  if (!cu_q || !cu_k || !dev_meta || (Sk > 0 && !kv_doc_ids)) return fail(PSF_EINVAL, "null pointer");
  if (capacity < 0) return fail(PSF_EINVAL, "capacity < 0");
  DeviceInfo* dev = nullptr;
  int rc = device_info(&dev);
  if (rc) return rc;
  cudaError_t e = launch_build_segments(kv_doc_ids, B, Sk, q_length, q_global_start, cu_q, cu_k, capacity, dev_meta,
                                        seg_is_pad, (flags & PSF_SEGMENTS_SKIP_PAD) ? 1 : 0, dev->status,
                                        static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PSF_OK : cuda_fail(e, "builder launch");
}

int psf_chunk_dense_flags(const int32_t* kv_doc_ids, int B, int S, int q_start, int q_length, int k_start,
                          int k_length, int32_t* flags, void* stream) {
  if (B < 1 || S < 1 || q_start < 0 || q_length < 0 || k_start < 0 || k_length < 0 ||
      (int64_t)q_start + q_length > S || (int64_t)k_start + k_length > S)
    return fail(PSF_EINVAL, "shard and chunk must lie inside the row");
  if (!kv_doc_ids || !flags) return fail(PSF_EINVAL, "null pointer");
  DeviceInfo* dev = nullptr;
  int rc = device_info(&dev);
  if (rc) return rc;
  cudaError_t e = launch_chunk_dense_flags(kv_doc_ids, B, S, q_start, q_length, k_start, k_length, flags,
                                           static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PSF_OK : cuda_fail(e, "dense-eligibility launch");
}

int psf_pad_fixup(void* out, float* lse, const int32_t* q_doc_ids, int layout, int B, int Lq, int Hq, int Dv,
                  void* stream) {
  if (layout != PSF_LAYOUT_THD && layout != PSF_LAYOUT_BHSD) return fail(PSF_EINVAL, "unknown layout");
  if (B < 1 || Lq < 0 || Hq < 1 || Dv < 8 || Dv % 8) return fail(PSF_EINVAL, "bad sizes");
  if (layout == PSF_LAYOUT_THD && B != 1) return fail(PSF_EINVAL, "packed THD layout takes B = 1");
  if (Lq == 0) return PSF_OK;
  if (!out || !lse || !q_doc_ids || !aligned16(out)) return fail(PSF_EINVAL, "null or unaligned pointer");
  DeviceInfo* dev = nullptr;
  int rc = device_info(&dev);
  if (rc) return rc;
  const View vo = tensor_view(layout, Lq, Hq, Dv), vl = lse_view(layout, Lq, Hq);
  cudaError_t e = launch_pad_fixup(out, lse, q_doc_ids, B, Lq, Hq, Dv, vo.sb, vo.ss,
                                   vo.sh, vl.sb, vl.sh, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PSF_OK : cuda_fail(e, "pad fixup launch");
}

int psf_lse_merge(const void* o1, const float* l1, const void* o2, const float* l2, float* o_f32, void* o_bf16,
                  float* l, int T, int H, int D, int dtype, void* stream) {
  if (T < 0 || H < 1 || D < 8 || D % 8) return fail(PSF_EINVAL, "bad sizes");
  if (int rc0 = check_dtype(dtype)) return rc0;
  if (T == 0) return PSF_OK;
  if (!o1 || !o2 || !l1 || !l2 || !l || (!o_f32 && !o_bf16)) return fail(PSF_EINVAL, "null pointer");
  if (!aligned16(o1) || !aligned16(o2) || (o_f32 && !aligned16(o_f32)) || (o_bf16 && !aligned16(o_bf16)))
    return fail(PSF_EINVAL, "unaligned pointer");
  DeviceInfo* dev = nullptr;
  int rc = device_info(&dev);
  if (rc) return rc;
  cudaError_t e = launch_lse_merge(o1, l1, o2, l2, o_f32, o_bf16, l, T, H, D, dtype == PSF_DTYPE_F16,
                                   static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PSF_OK : cuda_fail(e, "merge launch");
}

int psf_build_cross_segments(const int32_t* kv_doc_ids, int B, int S, int q_start, int q_length, int k_start,
                             int k_length, int32_t* cu_q, int32_t* cu_k, int32_t* dev_meta, void* stream) {
  if (B < 1 || S < 0 || q_start < 0 || q_length < 0 || k_start < 0 || k_length < 0 ||
      (int64_t)q_start + q_length > S || (int64_t)k_start + k_length > q_start)
    return fail(PSF_EINVAL, "need 0 <= k_start <= k_start + k_length <= q_start <= q_start + q_length <= S");
  if ((int64_t)B * 3 + 1 > 0x7fffffff || (int64_t)B * (S + 1) > 0x7fffffff) return fail(PSF_EINVAL, "too many rows");
  if (!cu_q || !cu_k || !dev_meta || (S > 0 && !kv_doc_ids)) return fail(PSF_EINVAL, "null pointer");
  DeviceInfo* dev = nullptr;
  int rc = device_info(&dev);
  if (rc) return rc;
  cudaError_t e = launch_cross_segments(kv_doc_ids, B, S, q_start, q_length, k_start, k_length, cu_q, cu_k, dev_meta,
                                        static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PSF_OK : cuda_fail(e, "cross builder launch");
}

int psf_lse_merge_live_rows(float* o_acc, void* o_run, float* l_acc, const void* o_new, const float* l_new,
                            const int32_t* cu_q, const int32_t* cu_k, const int32_t* dev_meta, int nseg, int T, int H,
                            int D, int dtype, void* stream) {
  if (T < 0 || H < 1 || D < 8 || D % 8 || nseg < 0) return fail(PSF_EINVAL, "bad sizes");
  if (int rc0 = check_dtype(dtype)) return rc0;
  if (T == 0 || nseg == 0) return PSF_OK;
  if ((!o_acc && !o_run) || !l_acc || !o_new || !l_new || !cu_q || !cu_k) return fail(PSF_EINVAL, "null pointer");
  if ((o_acc && !aligned16(o_acc)) || (o_run && !aligned16(o_run)) || !aligned16(o_new))
    return fail(PSF_EINVAL, "unaligned pointer");
  DeviceInfo* dev = nullptr;
  int rc = device_info(&dev);
  if (rc) return rc;
  cudaError_t e = launch_lse_merge_live(o_acc, o_run, l_acc, o_new, l_new, cu_q, cu_k, dev_meta, nseg, T, H, D,
                                        dtype == PSF_DTYPE_F16, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PSF_OK : cuda_fail(e, "live-row merge launch");
}

int psf_grad_add_live_rows(void* dst, const void* src, const int32_t* cu_q, const int32_t* cu_k,
                           const int32_t* dev_meta, int nseg, int T, int H, int D, int dtype, void* stream) {
  if (T < 0 || H < 1 || D < 8 || D % 8 || nseg < 0) return fail(PSF_EINVAL, "bad sizes");
  if (int rc0 = check_dtype(dtype)) return rc0;
  if (T == 0 || nseg == 0) return PSF_OK;
  if (!dst || !src || !cu_q || !cu_k) return fail(PSF_EINVAL, "null pointer");
  if (!aligned16(dst) || !aligned16(src)) return fail(PSF_EINVAL, "unaligned pointer");
  DeviceInfo* dev = nullptr;
  int rc = device_info(&dev);
  if (rc) return rc;
  cudaError_t e = launch_grad_add_live(dst, src, cu_q, cu_k, dev_meta, nseg, T, H, D, dtype == PSF_DTYPE_F16,
                                       static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PSF_OK : cuda_fail(e, "live-row gradient add launch");
}

}  // extern "C"

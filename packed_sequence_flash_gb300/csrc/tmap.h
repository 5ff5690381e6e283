// tmap.h -- host-side construction of TMA tensor maps (cuTensorMapEncodeTiled),
// resolved through the runtime's driver entry-point query so the library needs
// no link-time dependency on libcuda.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace psf {

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

inline EncodeTiledFn encode_tiled_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

// A 4-D view (d, s, h, b) of a tensor whose innermost dimension d is contiguous:
// element (d, s, h, b) sits at base + d + s*stride_s + h*stride_h + b*stride_b
// (strides in elements). The box is (box_d, box_s, 1, 1), 128-byte swizzled.
// Returns 0 on success.
inline int make_tmap_4d(CUtensorMap* map, CUtensorMapDataType dtype, int elem_bytes, const void* base,
                        int64_t D, int64_t S, int64_t H, int64_t B, int64_t stride_s, int64_t stride_h,
                        int64_t stride_b, int box_d, int box_s, CUtensorMapSwizzle swz, int box_h = 1) {
  EncodeTiledFn fn = encode_tiled_fn();
  if (!fn) return -1;
  cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)(S > 0 ? S : 1), (cuuint64_t)(H > 0 ? H : 1),
                        (cuuint64_t)(B > 0 ? B : 1)};
  cuuint64_t strides[3] = {(cuuint64_t)(stride_s * elem_bytes), (cuuint64_t)(stride_h * elem_bytes),
                           (cuuint64_t)(stride_b * elem_bytes)};
  // A degenerate dimension of extent 1 is never stepped over; give it the packed
  // stride so that the map stays legal (16-byte multiples) whatever the caller passed.
  for (int i = 0; i < 3; ++i) {
    if (dims[i + 1] == 1) {
      cuuint64_t inner = (i == 0) ? (cuuint64_t)D * elem_bytes : strides[i - 1] * dims[i];
      strides[i] = (inner + 15) / 16 * 16;
    }
    if (strides[i] == 0 || (strides[i] % 16) != 0) return -2;
  }
  cuuint32_t box[4] = {(cuuint32_t)box_d, (cuuint32_t)box_s, (cuuint32_t)box_h, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = fn(map, dtype, 4, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? 0 : -3;
}

}  // namespace psf

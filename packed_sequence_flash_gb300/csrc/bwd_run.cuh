// bwd_run.cuh -- launch helpers of the attention backward kernels, templated on
// the softcap and packed-heads flags; bwd.cu instantiates them with neither,
// bwd_cap.cu with the cap, bwd_pack.cu with packed query heads.
#pragma once

#include "bwd_dual.cuh"
#include "bwd_wide.cuh"

namespace psf {
namespace bwd_run {

template <typename T, int DQK, int DV, bool CAP, bool PACK>
cudaError_t run_dual(const BwdParams& p, int grid, cudaStream_t st) {
  const int smem = BwdDualCfg<DQK, DV>::SMEM_BYTES;
  cudaError_t e = cudaFuncSetAttribute(attn_bwd_dual_kernel<T, DQK, DV, CAP, PACK>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  attn_bwd_dual_kernel<T, DQK, DV, CAP, PACK><<<grid, 512, smem, st>>>(p);
  return cudaGetLastError();
}
template <typename T, int D, bool CAP>
cudaError_t run_wide(const BwdParams& p, int grid, cudaStream_t st) {
  const int smem = BwdWideCfg<D>::SMEM_BYTES;
  cudaError_t e =
      cudaFuncSetAttribute(attn_bwd_wide_kernel<T, D, CAP>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  attn_bwd_wide_kernel<T, D, CAP><<<grid, 384, smem, st>>>(p);
  return cudaGetLastError();
}
template <typename T, int DQK, int DV, bool CAP>
cudaError_t run_single(const BwdParams& p, int grid, cudaStream_t st) {
  const int smem = BwdCfg<DQK, DV>::SMEM_BYTES;
  cudaError_t e =
      cudaFuncSetAttribute(attn_bwd_kernel<T, DQK, DV, CAP>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  attn_bwd_kernel<T, DQK, DV, CAP><<<grid, 512, smem, st>>>(p);
  return cudaGetLastError();
}
template <typename T, bool CAP>
cudaError_t run_any(const BwdParams& p, int dqk, int dv, int grid, cudaStream_t st) {
  if (dqk == 512 && dv == 512) return run_wide<T, 512, CAP>(p, grid, st);
  if (dqk == 64 && dv == 64) return run_dual<T, 64, 64, CAP, false>(p, grid, st);
  if (dqk == 128 && dv == 128) return run_dual<T, 128, 128, CAP, false>(p, grid, st);
  if (dqk == 192 && dv == 128) return run_single<T, 192, 128, CAP>(p, grid, st);
  return cudaErrorInvalidValue;
}
template <bool CAP>
cudaError_t launch_grid(const BwdParams& p, int dqk, int dv, int grid, int f16, cudaStream_t st) {
  return f16 ? run_any<__half, CAP>(p, dqk, dv, grid, st) : run_any<__nv_bfloat16, CAP>(p, dqk, dv, grid, st);
}
// Packed query heads (head dims up to 128, no cap).
template <typename T>
cudaError_t run_packed(const BwdParams& p, int dqk, int dv, int grid, cudaStream_t st) {
  if (dqk == 64 && dv == 64) return run_dual<T, 64, 64, false, true>(p, grid, st);
  if (dqk == 128 && dv == 128) return run_dual<T, 128, 128, false, true>(p, grid, st);
  return cudaErrorInvalidValue;
}

}  // namespace bwd_run
}  // namespace psf

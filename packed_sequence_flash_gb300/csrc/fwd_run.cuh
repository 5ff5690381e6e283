// fwd_run.cuh -- launch helpers of the attention forward kernels, templated on
// the softcap flag; fwd.cu instantiates them without a cap, fwd_cap.cu with.
#pragma once

#include "fwd512.cuh"
#include "fwd_duo.cuh"
#include "fwd_pair.cuh"

namespace psf {
namespace fwd_run {

template <typename T, int DQK, int DVC, bool CAP>
cudaError_t run(const FwdParams& p, int grid, cudaStream_t st) {
  const int smem = FwdCfg<DQK, DVC>::SMEM_BYTES;
  cudaError_t e =
      cudaFuncSetAttribute(attn_fwd_kernel<T, DQK, DVC, CAP>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  attn_fwd_kernel<T, DQK, DVC, CAP><<<grid, 256, smem, st>>>(p);
  return cudaGetLastError();
}
template <typename T, int D, bool CAP>
cudaError_t run_duo(const FwdParams& p, int grid, cudaStream_t st) {
  const int smem = FwdDuoCfg<D>::SMEM_BYTES;
  cudaError_t e =
      cudaFuncSetAttribute(attn_fwd_duo_kernel<T, D, CAP>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  attn_fwd_duo_kernel<T, D, CAP><<<grid, 192, smem, st>>>(p);
  return cudaGetLastError();
}
template <typename T, int DQK, int DV, bool CAP>
cudaError_t run_pair(const FwdParams& p, int grid, cudaStream_t st) {
  const int smem = FwdPairCfg<DQK, DV>::SMEM_BYTES;
  cudaError_t e =
      cudaFuncSetAttribute(attn_fwd_pair_kernel<T, DQK, DV, CAP>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  attn_fwd_pair_kernel<T, DQK, DV, CAP><<<grid, 352, smem, st>>>(p);
  return cudaGetLastError();
}
template <typename T, bool CAP>
cudaError_t run_any(const FwdParams& p, int dqk, int dvc, int grid, cudaStream_t st) {
  if (dqk == 64 && dvc == 64) return run_duo<T, 64, CAP>(p, grid, st);
  if (dqk == 128 && dvc == 128) return run_duo<T, 128, CAP>(p, grid, st);
  if (dqk == 192 && dvc == 128) return run_pair<T, 192, 128, CAP>(p, grid, st);
  if (dqk == 512 && dvc == 256) return run<T, 512, 256, CAP>(p, grid, st);
  return cudaErrorInvalidValue;
}
template <bool CAP>
cudaError_t launch_grid(const FwdParams& p, int dqk, int dvc, int grid, int f16, cudaStream_t st) {
  return f16 ? run_any<__half, CAP>(p, dqk, dvc, grid, st) : run_any<__nv_bfloat16, CAP>(p, dqk, dvc, grid, st);
}

}  // namespace fwd_run
}  // namespace psf

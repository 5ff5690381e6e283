// bwd_run.cuh -- launch helpers of the attention backward kernels, templated on
// the softcap and packed-heads flags; bwd.cu instantiates them with neither,
// bwd_cap.cu with the cap, bwd_pack.cu with packed query heads.
#pragma once

#include "bwd192.cuh"
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
// The 512 kernel runs as four-CTA clusters; `grid` CTAs is rounded down to
// whole clusters and capped at the clusters that can be resident at once
// (the clusters take their units statically, so a cluster that had to wait
// for a free GPC would add a whole pass of units at the end).
template <typename T, int D, bool CAP>
cudaError_t run_wide(const BwdParams& p, int grid, cudaStream_t st) {
  const int smem = BwdWideCfg<D>::SMEM_BYTES;
  auto kern = attn_bwd_wide_kernel<T, D, CAP>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  static int resident[64] = {};  // per device: clusters resident at once (0: not yet asked)
  int dev = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (resident[dev] == 0) {
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = BwdWideCfg<D>::NP;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3(BwdWideCfg<D>::NP * 64);
    cfg.blockDim = dim3(384);
    cfg.dynamicSmemBytes = smem;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if ((e = cudaOccupancyMaxActiveClusters(&n, kern, &cfg)) != cudaSuccess) return e;
    if (n <= 0) return cudaErrorInvalidConfiguration;
    resident[dev] = n;
  }
  int clusters = grid / BwdWideCfg<D>::NP;
  if (clusters > resident[dev]) clusters = resident[dev];
  if (clusters < 1) clusters = 1;
  kern<<<clusters * BwdWideCfg<D>::NP, 384, smem, st>>>(p);
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

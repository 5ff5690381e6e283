// bwd.cu -- instantiations and launcher of the attention backward kernels:
// attn_bwd_dual_kernel for head dims up to 128, attn_bwd_kernel (single TMEM
// region) for Dqk = 192.
#include "bwd_dual.cuh"
#include "launch.h"

namespace psf {

namespace {
template <int DQK, int DV>
cudaError_t run_dual(const BwdParams& p, int grid, cudaStream_t st) {
  const int smem = BwdDualCfg<DQK, DV>::SMEM_BYTES;
  cudaError_t e =
      cudaFuncSetAttribute(attn_bwd_dual_kernel<DQK, DV>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  attn_bwd_dual_kernel<DQK, DV><<<grid, 384, smem, st>>>(p);
  return cudaGetLastError();
}
template <int DQK, int DV>
cudaError_t run_single(const BwdParams& p, int grid, cudaStream_t st) {
  const int smem = BwdCfg<DQK, DV>::SMEM_BYTES;
  cudaError_t e = cudaFuncSetAttribute(attn_bwd_kernel<DQK, DV>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  attn_bwd_kernel<DQK, DV><<<grid, 384, smem, st>>>(p);
  return cudaGetLastError();
}
}  // namespace

int bwd_smem_bytes(int dqk, int dv) {
  if (dqk == 64 && dv == 64) return BwdDualCfg<64, 64>::SMEM_BYTES;
  if (dqk == 128 && dv == 128) return BwdDualCfg<128, 128>::SMEM_BYTES;
  if (dqk == 192 && dv == 128) return BwdCfg<192, 128>::SMEM_BYTES;
  return -1;
}

cudaError_t launch_bwd(const BwdParams& p, int dqk, int dv, int grid, cudaStream_t st) {
  if (dqk == 64 && dv == 64) return run_dual<64, 64>(p, grid, st);
  if (dqk == 128 && dv == 128) return run_dual<128, 128>(p, grid, st);
  if (dqk == 192 && dv == 128) return run_single<192, 128>(p, grid, st);
  return cudaErrorInvalidValue;
}

}  // namespace psf

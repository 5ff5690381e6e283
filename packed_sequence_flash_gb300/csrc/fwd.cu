// fwd.cu -- instantiations and launcher of the attention forward kernel.
#include "fwd.cuh"
#include "launch.h"

namespace psf {

namespace {
template <int DQK, int DVC>
cudaError_t run(const FwdParams& p, int grid, cudaStream_t st) {
  const int smem = FwdCfg<DQK, DVC>::SMEM_BYTES;
  cudaError_t e = cudaFuncSetAttribute(attn_fwd_kernel<DQK, DVC>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  attn_fwd_kernel<DQK, DVC><<<grid, 256, smem, st>>>(p);
  return cudaGetLastError();
}
}  // namespace

int fwd_smem_bytes(int dqk, int dvc) {
  if (dqk == 64 && dvc == 64) return FwdCfg<64, 64>::SMEM_BYTES;
  if (dqk == 128 && dvc == 128) return FwdCfg<128, 128>::SMEM_BYTES;
  if (dqk == 192 && dvc == 128) return FwdCfg<192, 128>::SMEM_BYTES;
  if (dqk == 512 && dvc == 256) return FwdCfg<512, 256>::SMEM_BYTES;
  return -1;
}

cudaError_t launch_fwd(const FwdParams& p, int dqk, int dvc, int grid, cudaStream_t st) {
  if (dqk == 64 && dvc == 64) return run<64, 64>(p, grid, st);
  if (dqk == 128 && dvc == 128) return run<128, 128>(p, grid, st);
  if (dqk == 192 && dvc == 128) return run<192, 128>(p, grid, st);
  if (dqk == 512 && dvc == 256) return run<512, 256>(p, grid, st);
  return cudaErrorInvalidValue;
}

}  // namespace psf

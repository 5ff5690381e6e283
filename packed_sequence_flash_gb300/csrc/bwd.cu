// bwd.cu -- instantiations and launcher of the attention backward kernel.
#include "bwd.cuh"
#include "launch.h"

namespace psf {

namespace {
template <int DQK, int DV>
cudaError_t run(const BwdParams& p, int grid, cudaStream_t st) {
  const int smem = BwdCfg<DQK, DV>::SMEM_BYTES;
  cudaError_t e = cudaFuncSetAttribute(attn_bwd_kernel<DQK, DV>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  attn_bwd_kernel<DQK, DV><<<grid, 384, smem, st>>>(p);
  return cudaGetLastError();
}
}  // namespace

int bwd_smem_bytes(int dqk, int dv) {
  if (dqk == 64 && dv == 64) return BwdCfg<64, 64>::SMEM_BYTES;
  if (dqk == 128 && dv == 128) return BwdCfg<128, 128>::SMEM_BYTES;
  if (dqk == 192 && dv == 128) return BwdCfg<192, 128>::SMEM_BYTES;
  return -1;
}

cudaError_t launch_bwd(const BwdParams& p, int dqk, int dv, int grid, cudaStream_t st) {
  if (dqk == 64 && dv == 64) return run<64, 64>(p, grid, st);
  if (dqk == 128 && dv == 128) return run<128, 128>(p, grid, st);
  if (dqk == 192 && dv == 128) return run<192, 128>(p, grid, st);
  return cudaErrorInvalidValue;
}

}  // namespace psf

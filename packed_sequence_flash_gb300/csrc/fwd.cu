// fwd.cu -- instantiations and launcher of the attention forward kernels.
#include "fwd.cuh"
#include "fwd_duo.cuh"
#include "launch.h"

namespace psf {

namespace {
template <typename T, int DQK, int DVC>
cudaError_t run(const FwdParams& p, int grid, cudaStream_t st) {
  const int smem = FwdCfg<DQK, DVC>::SMEM_BYTES;
  cudaError_t e =
      cudaFuncSetAttribute(attn_fwd_kernel<T, DQK, DVC>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  attn_fwd_kernel<T, DQK, DVC><<<grid, 256, smem, st>>>(p);
  return cudaGetLastError();
}
template <typename T, int D>
cudaError_t run_duo(const FwdParams& p, int grid, cudaStream_t st) {
  const int smem = FwdDuoCfg<D>::SMEM_BYTES;
  cudaError_t e =
      cudaFuncSetAttribute(attn_fwd_duo_kernel<T, D>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  attn_fwd_duo_kernel<T, D><<<grid, 192, smem, st>>>(p);
  return cudaGetLastError();
}
template <typename T>
cudaError_t run_any(const FwdParams& p, int dqk, int dvc, int grid, cudaStream_t st) {
  if (dqk == 64 && dvc == 64) return run_duo<T, 64>(p, grid, st);
  if (dqk == 128 && dvc == 128) return run_duo<T, 128>(p, grid, st);
  if (dqk == 192 && dvc == 128) return run<T, 192, 128>(p, grid, st);
  if (dqk == 512 && dvc == 256) return run<T, 512, 256>(p, grid, st);
  return cudaErrorInvalidValue;
}
}  // namespace

int fwd_smem_bytes(int dqk, int dvc) {
  if (dqk == 64 && dvc == 64) return FwdDuoCfg<64>::SMEM_BYTES;
  if (dqk == 128 && dvc == 128) return FwdDuoCfg<128>::SMEM_BYTES;
  if (dqk == 192 && dvc == 128) return FwdCfg<192, 128>::SMEM_BYTES;
  if (dqk == 512 && dvc == 256) return FwdCfg<512, 256>::SMEM_BYTES;
  return -1;
}

// Head dims 64 and 128 run two CTAs per SM (attn_fwd_duo_kernel); the wider
// ones one CTA per SM.
cudaError_t launch_fwd(const FwdParams& p, int dqk, int dvc, int sms, int64_t max_work, int f16, cudaStream_t st) {
  const bool duo = (dqk == 64 && dvc == 64) || (dqk == 128 && dvc == 128);
  const int64_t cap = (int64_t)sms * (duo ? 2 : 1);
  const int grid = (int)(max_work < cap ? max_work : cap);
  if (grid <= 0) return cudaSuccess;
  return f16 ? run_any<__half>(p, dqk, dvc, grid, st) : run_any<__nv_bfloat16>(p, dqk, dvc, grid, st);
}

}  // namespace psf

// bwd.cu -- instantiations and launcher of the attention backward kernels:
// attn_bwd_dual_kernel for head dims up to 128, attn_bwd_kernel (single TMEM
// region) for Dqk = 192, attn_bwd_wide_kernel (column parts) for 512.
#include "bwd_dual.cuh"
#include "bwd_wide.cuh"
#include "launch.h"

namespace psf {

namespace {
template <typename T, int DQK, int DV>
cudaError_t run_dual(const BwdParams& p, int grid, cudaStream_t st) {
  const int smem = BwdDualCfg<DQK, DV>::SMEM_BYTES;
  cudaError_t e =
      cudaFuncSetAttribute(attn_bwd_dual_kernel<T, DQK, DV>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  attn_bwd_dual_kernel<T, DQK, DV><<<grid, 512, smem, st>>>(p);
  return cudaGetLastError();
}
template <typename T, int D>
cudaError_t run_wide(const BwdParams& p, int grid, cudaStream_t st) {
  const int smem = BwdWideCfg<D>::SMEM_BYTES;
  cudaError_t e =
      cudaFuncSetAttribute(attn_bwd_wide_kernel<T, D>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  attn_bwd_wide_kernel<T, D><<<grid, 384, smem, st>>>(p);
  return cudaGetLastError();
}
template <typename T, int DQK, int DV>
cudaError_t run_single(const BwdParams& p, int grid, cudaStream_t st) {
  const int smem = BwdCfg<DQK, DV>::SMEM_BYTES;
  cudaError_t e =
      cudaFuncSetAttribute(attn_bwd_kernel<T, DQK, DV>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  attn_bwd_kernel<T, DQK, DV><<<grid, 384, smem, st>>>(p);
  return cudaGetLastError();
}
template <typename T>
cudaError_t run_any(const BwdParams& p, int dqk, int dv, int grid, cudaStream_t st) {
  if (dqk == 512 && dv == 512) return run_wide<T, 512>(p, grid, st);
  if (dqk == 64 && dv == 64) return run_dual<T, 64, 64>(p, grid, st);
  if (dqk == 128 && dv == 128) return run_dual<T, 128, 128>(p, grid, st);
  if (dqk == 192 && dv == 128) return run_single<T, 192, 128>(p, grid, st);
  return cudaErrorInvalidValue;
}
}  // namespace

int bwd_smem_bytes(int dqk, int dv) {
  if (dqk == 64 && dv == 64) return BwdDualCfg<64, 64>::SMEM_BYTES;
  if (dqk == 128 && dv == 128) return BwdDualCfg<128, 128>::SMEM_BYTES;
  if (dqk == 192 && dv == 128) return BwdCfg<192, 128>::SMEM_BYTES;
  if (dqk == 512 && dv == 512) return BwdWideCfg<512>::SMEM_BYTES;
  return -1;
}

cudaError_t launch_bwd(const BwdParams& p, int dqk, int dv, int sms, int item_cap, int f16, cudaStream_t st) {
  const int64_t units = (int64_t)item_cap * p.Hkv * (dqk == 512 ? BwdWideCfg<512>::NP : 1);
  const int grid = (int)(units < sms ? units : sms);
  return f16 ? run_any<__half>(p, dqk, dv, grid, st) : run_any<__nv_bfloat16>(p, dqk, dv, grid, st);
}

}  // namespace psf

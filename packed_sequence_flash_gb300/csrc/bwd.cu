// bwd.cu -- instantiations and launcher of the attention backward kernels:
// attn_bwd_dual_kernel for head dims up to 128, attn_bwd_kernel (single TMEM
// region) for Dqk = 192, attn_bwd_wide_kernel (column parts) for 512.
#include "bwd_dual.cuh"
#include "bwd_wide.cuh"
#include "launch.h"

namespace psf {

namespace {
template <int DQK, int DV>
cudaError_t run_dual(const BwdParams& p, int grid, cudaStream_t st) {
  const int smem = BwdDualCfg<DQK, DV>::SMEM_BYTES;
  cudaError_t e =
      cudaFuncSetAttribute(attn_bwd_dual_kernel<DQK, DV>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  attn_bwd_dual_kernel<DQK, DV><<<grid, 512, smem, st>>>(p);
  return cudaGetLastError();
}
template <int D>
cudaError_t run_wide(const BwdParams& p, int grid, cudaStream_t st) {
  const int smem = BwdWideCfg<D>::SMEM_BYTES;
  cudaError_t e = cudaFuncSetAttribute(attn_bwd_wide_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  attn_bwd_wide_kernel<D><<<grid, 384, smem, st>>>(p);
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
  if (dqk == 512 && dv == 512) return BwdWideCfg<512>::SMEM_BYTES;
  return -1;
}

cudaError_t launch_bwd(const BwdParams& p, int dqk, int dv, int sms, int item_cap, cudaStream_t st) {
  const int64_t units = (int64_t)item_cap * p.Hkv * (dqk == 512 ? BwdWideCfg<512>::NP : 1);
  const int grid = (int)(units < sms ? units : sms);
  if (dqk == 512 && dv == 512) return run_wide<512>(p, grid, st);
  if (dqk == 64 && dv == 64) return run_dual<64, 64>(p, grid, st);
  if (dqk == 128 && dv == 128) return run_dual<128, 128>(p, grid, st);
  if (dqk == 192 && dv == 128) return run_single<192, 128>(p, grid, st);
  return cudaErrorInvalidValue;
}

}  // namespace psf

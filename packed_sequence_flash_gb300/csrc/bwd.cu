// bwd.cu -- instantiations and launcher of the attention backward kernels:
// attn_bwd_dual_kernel for head dims up to 128, attn_bwd_kernel (single TMEM
// region) for Dqk = 192, attn_bwd_wide_kernel (column parts) for 512.
#include "bwd_run.cuh"
#include "launch.h"

namespace psf {

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
  if (grid <= 0) return cudaSuccess;
  if (p.pack > 1) return launch_bwd_packed(p, dqk, dv, grid, f16, st);
  if (p.softcap > 0.f) return launch_bwd_capped(p, dqk, dv, grid, f16, st);
  return bwd_run::launch_grid<false>(p, dqk, dv, grid, f16, st);
}

}  // namespace psf

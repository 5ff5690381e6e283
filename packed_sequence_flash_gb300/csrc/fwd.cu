// fwd.cu -- instantiations and launcher of the attention forward kernels.
#include "fwd_run.cuh"
#include "launch.h"

namespace psf {

int fwd_smem_bytes(int dqk, int dvc) {
  if (dqk == 64 && dvc == 64) return FwdDuoCfg<64>::SMEM_BYTES;
  if (dqk == 128 && dvc == 128) return FwdDuoCfg<128>::SMEM_BYTES;
  if (dqk == 192 && dvc == 128) return FwdPairCfg<192, 128>::SMEM_BYTES;
  if (dqk == 512 && dvc == 256) return FwdCfg<512, 256>::SMEM_BYTES;
  return -1;
}

// Head dims 64 and 128 run two CTAs per SM (attn_fwd_duo_kernel); 192/128 one
// CTA per SM over 256-row items (attn_fwd_pair_kernel), 512 one CTA per SM.
cudaError_t launch_fwd(const FwdParams& p, int dqk, int dvc, int sms, int64_t max_work, int f16, cudaStream_t st) {
  const bool duo = (dqk == 64 && dvc == 64) || (dqk == 128 && dvc == 128);
  const int64_t cap = (int64_t)sms * (duo ? 2 : 1);
  const int grid = (int)(max_work < cap ? max_work : cap);
  if (grid <= 0) return cudaSuccess;
  if (p.softcap > 0.f) return launch_fwd_capped(p, dqk, dvc, grid, f16, st);
  return fwd_run::launch_grid<false>(p, dqk, dvc, grid, f16, st);
}

}  // namespace psf

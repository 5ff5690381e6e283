// fwd_cap.cu -- the attention forward kernels with a logit softcap.
#include "fwd_run.cuh"
#include "launch.h"

namespace psf {

cudaError_t launch_fwd_capped(const FwdParams& p, int dqk, int dvc, int grid, int f16, cudaStream_t st) {
  return fwd_run::launch_grid<true>(p, dqk, dvc, grid, f16, st);
}

}  // namespace psf

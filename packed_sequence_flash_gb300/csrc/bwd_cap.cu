// bwd_cap.cu -- the attention backward kernels with a logit softcap.
#include "bwd_run.cuh"
#include "launch.h"

namespace psf {

cudaError_t launch_bwd_capped(const BwdParams& p, int dqk, int dv, int grid, int f16, cudaStream_t st) {
  return bwd_run::launch_grid<true>(p, dqk, dv, grid, f16, st);
}

}  // namespace psf

// bwd_pack.cu -- the head-dim-<=-128 attention backward with a KV head's query
// heads packed into each step.
#include "bwd_run.cuh"
#include "launch.h"

namespace psf {

cudaError_t launch_bwd_packed(const BwdParams& p, int dqk, int dv, int grid, int f16, cudaStream_t st) {
  return f16 ? bwd_run::run_packed<__half>(p, dqk, dv, grid, st)
             : bwd_run::run_packed<__nv_bfloat16>(p, dqk, dv, grid, st);
}

}  // namespace psf

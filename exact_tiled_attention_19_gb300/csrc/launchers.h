// Internal declarations of the per-variant kernel launchers (one per head dim
// and element type), implemented in attn_fwd_inst.cu.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

namespace etattn {

struct FwdParams;

#define ETATTN_DECLARE_LAUNCHER(name)                                                                     \
  cudaError_t name(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v, const FwdParams& p, \
                   dim3 grid, int nsub, bool general, cudaStream_t stream);

ETATTN_DECLARE_LAUNCHER(launch_fwd_d32_0)
ETATTN_DECLARE_LAUNCHER(launch_fwd_d32_1)
ETATTN_DECLARE_LAUNCHER(launch_fwd_d64_0)
ETATTN_DECLARE_LAUNCHER(launch_fwd_d64_1)
ETATTN_DECLARE_LAUNCHER(launch_fwd_d128_0)
ETATTN_DECLARE_LAUNCHER(launch_fwd_d128_1)

#undef ETATTN_DECLARE_LAUNCHER

}  // namespace etattn

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

// Merge of split-KV partial states (attn_combine.cu).  Row r is the lse
// index of an output row; its slice-s state is part_o[(s * rows + r) * D ..]
// and part_lse[s * rows + r].
struct CombineParams {
  const float* part_o;
  const float* part_lse;
  int64_t rows;                  // rows per slice (the size of lse)
  int num_splits;
  void* o;                       // output in the input type
  float* lse;                    // or nullptr
  int64_t o_sb, o_sh, o_sn;      // element strides of o (batch, head, token)
  int Hq, Nq;                    // batched layout: row = (b * Hq + h) * Nq + t
  int packed;                    // packed layout: row = h * total + t
  int64_t total;                 // packed: query tokens
};

cudaError_t launch_combine(int D, bool bf16, const CombineParams& c, cudaStream_t stream);

}  // namespace etattn

// Internal declarations of the per-variant kernel launchers (one per head dim
// and element type), implemented in attn_fwd_inst.cu.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

namespace etattn {

struct FwdParams;

#define ETATTN_DECLARE_LAUNCHER(name)                                                                     \
  cudaError_t name(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v, const FwdParams& p, \
                   dim3 grid, int nsub, bool general, bool ksplit, bool split, cudaStream_t stream);

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

// Backward pass (attn_bwd_aux.cu, attn_bwd_inst.cu).
struct BwdParams;

// Before the backward kernel: one row per (batch, query head, query) of
// [B * Hq][Nq_pad].
struct BwdPreParams {
  const void* o;                 // forward output, input type
  const void* dout;              // upstream gradient, input type
  const float* lse;              // [B, Hq, Nq] contiguous
  int64_t o_sb, o_sh, o_sn;      // element strides (batch, head, token); d-stride 1
  int64_t do_sb, do_sh, do_sn;
  int64_t rows;                  // B * Hq * Nq_pad
  int Hq, Nq, Nq_pad;
  float scale;
  float* nsd;                    // out: [B * Hq][Nq_pad], -scale * <dO, O>
  float* nlse2;                  // out: [B * Hq][Nq_pad], -lse * log2(e)
  float* dq_acc;                 // out: [B, Hq, Nq, D] zeroed
};

// After: FP32 dQ to the input type.
struct BwdConvertParams {
  const float* dq_acc;           // [B, Hq, Nq, D]
  void* dq;
  int64_t dq_sb, dq_sh, dq_sn;
  int64_t rows;                  // B * Hq * Nq
  int Hq, Nq;
};

cudaError_t launch_bwd_pre(int D, bool bf16, const BwdPreParams& c, cudaStream_t stream);
cudaError_t launch_bwd_convert(int D, bool bf16, const BwdConvertParams& c, cudaStream_t stream);

#define ETATTN_DECLARE_BWD_LAUNCHER(name)                                                                  \
  cudaError_t name(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v, const CUtensorMap& dout, \
                   const CUtensorMap& dq_acc, const BwdParams& p, dim3 grid, cudaStream_t stream);

ETATTN_DECLARE_BWD_LAUNCHER(launch_bwd_d32_0)
ETATTN_DECLARE_BWD_LAUNCHER(launch_bwd_d32_1)
ETATTN_DECLARE_BWD_LAUNCHER(launch_bwd_d64_0)
ETATTN_DECLARE_BWD_LAUNCHER(launch_bwd_d64_1)
ETATTN_DECLARE_BWD_LAUNCHER(launch_bwd_d128_0)
ETATTN_DECLARE_BWD_LAUNCHER(launch_bwd_d128_1)

#undef ETATTN_DECLARE_BWD_LAUNCHER

}  // namespace etattn

// One (head dim, element type) instantiation of the backward kernel and its
// launcher, compiled once per variant with -DETATTN_INST_D=<32|64|128>
// -DETATTN_INST_BF16=<0|1> (like attn_fwd_inst.cu).
#include <atomic>
#include <cuda_runtime.h>

#include "attn_bwd_kernel.cuh"
#include "launchers.h"

#ifndef ETATTN_INST_D
#error "ETATTN_INST_D must be defined"
#endif
#ifndef ETATTN_INST_BF16
#error "ETATTN_INST_BF16 must be defined"
#endif

#define ETATTN_BCAT2(a, b, c) a##b##_##c
#define ETATTN_BCAT(a, b, c) ETATTN_BCAT2(a, b, c)
#define ETATTN_BWD_LAUNCHER ETATTN_BCAT(launch_bwd_d, ETATTN_INST_D, ETATTN_INST_BF16)

namespace etattn {

cudaError_t ETATTN_BWD_LAUNCHER(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                                const CUtensorMap& dout, const CUtensorMap& dq_acc, const BwdParams& p, dim3 grid,
                                cudaStream_t stream) {
  using C = BwdCfg<ETATTN_INST_D>;
  auto kern = attn_bwd_kernel<ETATTN_INST_D, ETATTN_INST_BF16 != 0>;
  // The dynamic shared-memory opt-in is per device; set it once per device.
  static std::atomic<unsigned long long> configured{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = 1ull << (dev & 63);
  if (!(configured.load() & bit)) {
    // The kernel re-splits its registers between warpgroups (setmaxnreg);
    // the split is only valid if every thread launches with LAUNCH_REGS.
    cudaFuncAttributes fa;
    e = cudaFuncGetAttributes(&fa, kern);
    if (e != cudaSuccess) return e;
    if (fa.numRegs != C::LAUNCH_REGS) return cudaErrorInvalidConfiguration;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    configured.fetch_or(bit);
  }
  kern<<<grid, C::THREADS, C::SMEM_BYTES, stream>>>(q, k, v, dout, dq_acc, p);
  return cudaGetLastError();
}

}  // namespace etattn

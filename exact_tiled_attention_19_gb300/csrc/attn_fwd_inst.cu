// One (head dim, element type) instantiation of the forward kernel and its
// launcher.  The build compiles this file once per variant with
// -DETATTN_INST_D=<32|64|128> -DETATTN_INST_BF16=<0|1>, so the variants
// compile in parallel.
#include <atomic>
#include <cuda_runtime.h>

#include "attn_fwd_kernel.cuh"
#include "launchers.h"

#ifndef ETATTN_INST_D
#error "ETATTN_INST_D must be defined"
#endif
#ifndef ETATTN_INST_BF16
#error "ETATTN_INST_BF16 must be defined"
#endif

#define ETATTN_CAT2(a, b, c) a##b##_##c
#define ETATTN_CAT(a, b, c) ETATTN_CAT2(a, b, c)
#define ETATTN_LAUNCHER ETATTN_CAT(launch_fwd_d, ETATTN_INST_D, ETATTN_INST_BF16)

namespace etattn {

namespace {

template <int NSUB, bool GEN, bool KS, bool GLB, bool SPL>
cudaError_t launch_one(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v, const FwdParams& p, dim3 grid,
                       cudaStream_t stream) {
  using C = TileCfg<ETATTN_INST_D, NSUB>;
  auto kern = attn_fwd_kernel<ETATTN_INST_D, NSUB, ETATTN_INST_BF16 != 0, GEN, KS, GLB, SPL>;
  // The dynamic shared-memory opt-in is per device; set it once per device.
  static std::atomic<unsigned long long> configured{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = 1ull << (dev & 63);
  if (!(configured.load() & bit)) {
    if (NSUB == 2) {
      // The two-sub-tile kernel re-splits its registers between warpgroups
      // (setmaxnreg); the split is only valid if every thread launches with
      // LAUNCH_REGS registers.
      cudaFuncAttributes fa;
      e = cudaFuncGetAttributes(&fa, kern);
      if (e != cudaSuccess) return e;
      if (fa.numRegs != C::LAUNCH_REGS) return cudaErrorInvalidConfiguration;
    }
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    configured.fetch_or(bit);
  }
  // Programmatic stream serialisation: the launch may be scheduled while the
  // previous grid on the stream finishes; the kernel's griddepcontrol.wait
  // keeps every memory access after that grid's completion.
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(C::THREADS);
  cfg.dynamicSmemBytes = C::SMEM_BYTES;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, q, k, v, p);
}

}  // namespace

// The build with split = true carries the two-part P path for rows with few
// keys (BF16 only; an FP16 call never asks for it).
template <bool SPL>
cudaError_t launch_variant(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v, const FwdParams& p,
                           dim3 grid, int nsub, bool general, bool ksplit, cudaStream_t stream) {
  if (p.num_global > 0)  // global tokens: the general build with the two-phase tile stream
    return nsub == 1 ? launch_one<1, true, false, true, SPL>(q, k, v, p, grid, stream)
                     : launch_one<2, true, false, true, SPL>(q, k, v, p, grid, stream);
  if (ksplit) return launch_one<2, true, true, false, SPL>(q, k, v, p, grid, stream);
  if (general)
    return nsub == 1 ? launch_one<1, true, false, false, SPL>(q, k, v, p, grid, stream)
                     : launch_one<2, true, false, false, SPL>(q, k, v, p, grid, stream);
  return nsub == 1 ? launch_one<1, false, false, false, SPL>(q, k, v, p, grid, stream)
                   : launch_one<2, false, false, false, SPL>(q, k, v, p, grid, stream);
}

cudaError_t ETATTN_LAUNCHER(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v, const FwdParams& p,
                            dim3 grid, int nsub, bool general, bool ksplit, bool split, cudaStream_t stream) {
#if ETATTN_INST_BF16
  if (split) return launch_variant<true>(q, k, v, p, grid, nsub, general, ksplit, stream);
#else
  (void)split;
#endif
  return launch_variant<false>(q, k, v, p, grid, nsub, general, ksplit, stream);
}

}  // namespace etattn

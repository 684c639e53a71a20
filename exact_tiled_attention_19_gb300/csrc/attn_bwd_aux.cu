// The launches before and after the attention backward kernel.
//
// Before ("Attention algorithms and data movement", lesson 03: the saved
// normalisation state): for every query row, -scale * D with D = <dO, O> in
// FP32, the negated saved logsumexp in base 2 (-lse * log2(e); -inf for a row
// that read no key, so that its recomputed probabilities are 0), and a zeroed
// FP32 dQ row.  Rows past Nq up to the next multiple of 128 get 0 and -inf,
// so the backward kernel can copy 128 values per query block without a
// bounds check.
//
// After: dQ, accumulated in FP32 by the backward kernel, in the input type.
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "launchers.h"

namespace etattn {

namespace {

template <bool BF16>
__device__ __forceinline__ float to_f32(uint16_t h) {
  return BF16 ? __uint_as_float((uint32_t)h << 16) : __half2float(__ushort_as_half(h));
}

template <int D, bool BF16>
__global__ void __launch_bounds__(256) bwd_pre_kernel(BwdPreParams c) {
  constexpr int PER = D / 32;
  const int64_t row = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
  if (row >= c.rows) return;
  const int lane = threadIdx.x & 31;
  const int64_t bh = row / c.Nq_pad;
  const int q = (int)(row - bh * c.Nq_pad);
  float d = 0.f, l2 = -INFINITY;
  if (q < c.Nq) {
    const int64_t b = bh / c.Hq, h = bh - b * c.Hq;
    const uint16_t* o = static_cast<const uint16_t*>(c.o) + b * c.o_sb + h * c.o_sh + (int64_t)q * c.o_sn + lane * PER;
    const uint16_t* g = static_cast<const uint16_t*>(c.dout) + b * c.do_sb + h * c.do_sh + (int64_t)q * c.do_sn +
                        lane * PER;
    float acc = 0.f;
#pragma unroll
    for (int i = 0; i < PER; ++i) acc = fmaf(to_f32<BF16>(o[i]), to_f32<BF16>(g[i]), acc);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    d = -c.scale * acc;
    const float lse = c.lse[bh * c.Nq + q];
    l2 = lse == -INFINITY ? -INFINITY : -lse * 1.4426950408889634f;
    float* dq = c.dq_acc + (bh * c.Nq + q) * D + lane * PER;
#pragma unroll
    for (int i = 0; i < PER; ++i) dq[i] = 0.f;
  }
  if (lane == 0) {
    c.nsd[row] = d;
    c.nlse2[row] = l2;
  }
}

template <int D, bool BF16>
__global__ void __launch_bounds__(256) bwd_dq_convert_kernel(BwdConvertParams c) {
  constexpr int PER = D / 32;
  const int64_t row = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
  if (row >= c.rows) return;
  const int lane = threadIdx.x & 31;
  const int64_t bh = row / c.Nq, q = row - bh * c.Nq;
  const int64_t b = bh / c.Hq, h = bh - b * c.Hq;
  const float* src = c.dq_acc + row * D + lane * PER;
  uint16_t* dst = static_cast<uint16_t*>(c.dq) + b * c.dq_sb + h * c.dq_sh + q * c.dq_sn + lane * PER;
#pragma unroll
  for (int i = 0; i < PER; ++i) {
    if constexpr (BF16) {
      dst[i] = __bfloat16_as_ushort(__float2bfloat16_rn(src[i]));
    } else {
      dst[i] = __half_as_ushort(__float2half_rn(src[i]));
    }
  }
}

template <int D, bool BF16>
cudaError_t pre(const BwdPreParams& c, cudaStream_t s) {
  const int64_t blocks = (c.rows + 7) / 8;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  if (blocks > 0) bwd_pre_kernel<D, BF16><<<(unsigned)blocks, 256, 0, s>>>(c);
  return cudaGetLastError();
}

template <int D, bool BF16>
cudaError_t convert(const BwdConvertParams& c, cudaStream_t s) {
  const int64_t blocks = (c.rows + 7) / 8;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  if (blocks > 0) bwd_dq_convert_kernel<D, BF16><<<(unsigned)blocks, 256, 0, s>>>(c);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_pre(int D, bool bf16, const BwdPreParams& c, cudaStream_t s) {
  switch (D) {
    case 32: return bf16 ? pre<32, true>(c, s) : pre<32, false>(c, s);
    case 64: return bf16 ? pre<64, true>(c, s) : pre<64, false>(c, s);
    default: return bf16 ? pre<128, true>(c, s) : pre<128, false>(c, s);
  }
}

cudaError_t launch_bwd_convert(int D, bool bf16, const BwdConvertParams& c, cudaStream_t s) {
  switch (D) {
    case 32: return bf16 ? convert<32, true>(c, s) : convert<32, false>(c, s);
    case 64: return bf16 ? convert<64, true>(c, s) : convert<64, false>(c, s);
    default: return bf16 ? convert<128, true>(c, s) : convert<128, false>(c, s);
  }
}

}  // namespace etattn

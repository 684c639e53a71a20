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
#include <cstring>
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
template <bool BF16>
__device__ __forceinline__ uint16_t from_f32(float x) {
  return BF16 ? __bfloat16_as_ushort(__float2bfloat16_rn(x)) : __half_as_ushort(__float2half_rn(x));
}

// A lane's PER consecutive elements of a row move as one vector access: the
// rows start on 16-byte boundaries (the launcher's stride and alignment
// checks), so lane * PER elements of 2 or 4 bytes are aligned to the access.
template <int BYTES> struct VecOf;
template <> struct VecOf<2> { using T = uint16_t; };
template <> struct VecOf<4> { using T = uint32_t; };
template <> struct VecOf<8> { using T = uint2; };
template <> struct VecOf<16> { using T = uint4; };

template <typename E, int PER>
__device__ __forceinline__ void load_vec(const E* src, E (&dst)[PER]) {
  using V = typename VecOf<sizeof(E) * PER>::T;
  const V v = *reinterpret_cast<const V*>(src);
  memcpy(dst, &v, sizeof v);
}
template <typename E, int PER>
__device__ __forceinline__ void store_vec(E* dst, const E (&src)[PER]) {
  using V = typename VecOf<sizeof(E) * PER>::T;
  V v;
  memcpy(&v, src, sizeof v);
  *reinterpret_cast<V*>(dst) = v;
}

// One warp per query row; each block of 256 threads takes ROWS_PER_WARP rows
// per warp (all loads of a warp's rows go out before the first use).
constexpr int ROWS_PER_WARP = 2;

template <int D, bool BF16>
__global__ void __launch_bounds__(256) bwd_pre_kernel(BwdPreParams c) {
  constexpr int PER = D / 32;
  const int lane = threadIdx.x & 31;
  const int64_t row0 = ((int64_t)blockIdx.x * 8 + (threadIdx.x >> 5)) * ROWS_PER_WARP;
  uint16_t ov[ROWS_PER_WARP][PER], gv[ROWS_PER_WARP][PER];
  bool live[ROWS_PER_WARP];
  int64_t bhs[ROWS_PER_WARP];
  int qs[ROWS_PER_WARP];
#pragma unroll
  for (int r = 0; r < ROWS_PER_WARP; ++r) {
    const int64_t row = row0 + r;
    const int64_t bh = row / c.Nq_pad;
    const int q = (int)(row - bh * c.Nq_pad);
    bhs[r] = bh;
    qs[r] = q;
    live[r] = row < c.rows && q < c.Nq;
    if (live[r]) {
      const int64_t b = bh / c.Hq, h = bh - b * c.Hq;
      load_vec(static_cast<const uint16_t*>(c.o) + b * c.o_sb + h * c.o_sh + (int64_t)q * c.o_sn + lane * PER, ov[r]);
      load_vec(static_cast<const uint16_t*>(c.dout) + b * c.do_sb + h * c.do_sh + (int64_t)q * c.do_sn + lane * PER,
               gv[r]);
    }
  }
#pragma unroll
  for (int r = 0; r < ROWS_PER_WARP; ++r) {
    const int64_t row = row0 + r;
    if (row >= c.rows) break;
    float d = 0.f, l2 = -INFINITY;
    if (live[r]) {
      float acc = 0.f;
#pragma unroll
      for (int i = 0; i < PER; ++i) acc = fmaf(to_f32<BF16>(ov[r][i]), to_f32<BF16>(gv[r][i]), acc);
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
      d = -c.scale * acc;
      const float lse = c.lse[bhs[r] * c.Nq + qs[r]];
      l2 = lse == -INFINITY ? -INFINITY : -lse * 1.4426950408889634f;
      float z[PER];
#pragma unroll
      for (int i = 0; i < PER; ++i) z[i] = 0.f;
      store_vec(c.dq_acc + (bhs[r] * c.Nq + qs[r]) * D + lane * PER, z);
    }
    if (lane == 0) {
      c.nsd[row] = d;
      c.nlse2[row] = l2;
    }
  }
}

template <int D, bool BF16>
__global__ void __launch_bounds__(256) bwd_dq_convert_kernel(BwdConvertParams c) {
  constexpr int PER = D / 32;
  const int lane = threadIdx.x & 31;
  const int64_t row0 = ((int64_t)blockIdx.x * 8 + (threadIdx.x >> 5)) * ROWS_PER_WARP;
  float v[ROWS_PER_WARP][PER];
#pragma unroll
  for (int r = 0; r < ROWS_PER_WARP; ++r)
    if (row0 + r < c.rows) load_vec(c.dq_acc + (row0 + r) * D + lane * PER, v[r]);
#pragma unroll
  for (int r = 0; r < ROWS_PER_WARP; ++r) {
    const int64_t row = row0 + r;
    if (row >= c.rows) break;
    const int64_t bh = row / c.Nq, q = row - bh * c.Nq;
    const int64_t b = bh / c.Hq, h = bh - b * c.Hq;
    uint16_t o[PER];
#pragma unroll
    for (int i = 0; i < PER; ++i) o[i] = from_f32<BF16>(v[r][i]);
    store_vec(static_cast<uint16_t*>(c.dq) + b * c.dq_sb + h * c.dq_sh + q * c.dq_sn + lane * PER, o);
  }
}

template <int D, bool BF16>
cudaError_t pre(const BwdPreParams& c, cudaStream_t s) {
  const int64_t blocks = (c.rows + 8 * ROWS_PER_WARP - 1) / (8 * ROWS_PER_WARP);
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  if (blocks > 0) bwd_pre_kernel<D, BF16><<<(unsigned)blocks, 256, 0, s>>>(c);
  return cudaGetLastError();
}

template <int D, bool BF16>
cudaError_t convert(const BwdConvertParams& c, cudaStream_t s) {
  const int64_t blocks = (c.rows + 8 * ROWS_PER_WARP - 1) / (8 * ROWS_PER_WARP);
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

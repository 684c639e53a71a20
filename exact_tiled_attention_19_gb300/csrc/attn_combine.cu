// Second launch of a split-KV forward pass: merge every row's partial states
// over the key slices and normalise.
//
// Method ("Intermediate and advanced extension", workshop row "Split
// softmax", and "Logic review before implementation": partial denominators
// are rescaled before they are merged, and a kernel boundary on the same
// stream orders the stages, with no cross-block spin barrier).  Slice s of a
// row holds O_s = acc_s / l_s and lse_s = scale * m_s + ln l_s, the
// (maximum, exponential sum, numerator) state of its keys in normalised form.
// With M = max_s lse_s and w_s = exp(lse_s - M):
//     O = sum_s w_s O_s / sum_s w_s,   lse = M + ln sum_s w_s,
// the merge of the slices' states ("Attention algorithms and data movement",
// lesson 01).  A slice with no eligible key has lse_s = -inf and weight 0;
// a row whose slices are all empty gets O = 0 and lse = -inf (the explicit
// empty identity).
#include <cstdint>
#include <cuda_runtime.h>

#include "launchers.h"

namespace etattn {

namespace {

// One warp per row; lane l owns the D/32 consecutive elements at l * D/32.
template <int D, bool BF16>
__global__ void __launch_bounds__(256) attn_combine_kernel(CombineParams c) {
  constexpr int PER = D / 32;
  const int64_t row = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
  if (row >= c.rows) return;
  const int lane = threadIdx.x & 31;

  float mx = -INFINITY;
  for (int s = lane; s < c.num_splits; s += 32) mx = fmaxf(mx, c.part_lse[(int64_t)s * c.rows + row]);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));

  float acc[PER];
#pragma unroll
  for (int i = 0; i < PER; ++i) acc[i] = 0.f;
  float wsum = 0.f;
  if (mx != -INFINITY) {
    for (int s = 0; s < c.num_splits; ++s) {
      const float ls = c.part_lse[(int64_t)s * c.rows + row];  // same address in every lane
      const float w = expf(ls - mx);                            // 0 for an empty slice
      // A slice of weight 0 (no eligible key) adds nothing, and its partial
      // row is not read: after a failed forward launch it may hold anything,
      // and 0 * NaN would poison the merged row.  (w is the same in every lane.)
      if (w == 0.f) continue;
      wsum += w;
      const float* src = c.part_o + ((int64_t)s * c.rows + row) * D + lane * PER;
      if constexpr (PER == 4) {
        const float4 x = *reinterpret_cast<const float4*>(src);
        acc[0] += w * x.x;
        acc[1] += w * x.y;
        acc[2] += w * x.z;
        acc[3] += w * x.w;
      } else if constexpr (PER == 2) {
        const float2 x = *reinterpret_cast<const float2*>(src);
        acc[0] += w * x.x;
        acc[1] += w * x.y;
      } else {
        acc[0] += w * src[0];
      }
    }
  }
  const float inv = wsum > 0.f ? 1.f / wsum : 0.f;

  // Row -> (batch/sequence, head, token) of the output.
  int64_t b, h, t;
  if (c.packed) {  // lse index = h * T + t
    h = row / c.total;
    t = row - h * c.total;
    b = 0;
  } else {         // lse index = (b * Hq + h) * Nq + t
    t = row % c.Nq;
    const int64_t bh = row / c.Nq;
    h = bh % c.Hq;
    b = bh / c.Hq;
  }
  uint16_t* dst = reinterpret_cast<uint16_t*>(static_cast<uint8_t*>(c.o) +
                                              2 * (b * c.o_sb + h * c.o_sh + t * c.o_sn)) + lane * PER;
#pragma unroll
  for (int i = 0; i < PER; i += 2) {
    const float a0 = acc[i] * inv;
    const float a1 = PER > 1 ? acc[i + 1] * inv : 0.f;
    uint32_t packed;
    if constexpr (BF16) {
      asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(packed) : "f"(a1), "f"(a0));
    } else {
      asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(packed) : "f"(a1), "f"(a0));
    }
    if constexpr (PER > 1) {
      *reinterpret_cast<uint32_t*>(dst + i) = packed;
    } else {
      dst[i] = (uint16_t)(packed & 0xffffu);
    }
  }
  if (c.lse != nullptr && lane == 0) c.lse[row] = wsum > 0.f ? mx + logf(wsum) : -INFINITY;
}

template <int D, bool BF16>
cudaError_t launch(const CombineParams& c, cudaStream_t stream) {
  const int64_t blocks = (c.rows + 7) / 8;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  attn_combine_kernel<D, BF16><<<(unsigned)blocks, 256, 0, stream>>>(c);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_combine(int D, bool bf16, const CombineParams& c, cudaStream_t stream) {
  switch (D) {
    case 32: return bf16 ? launch<32, true>(c, stream) : launch<32, false>(c, stream);
    case 64: return bf16 ? launch<64, true>(c, stream) : launch<64, false>(c, stream);
    default: return bf16 ? launch<128, true>(c, stream) : launch<128, false>(c, stream);
  }
}

}  // namespace etattn

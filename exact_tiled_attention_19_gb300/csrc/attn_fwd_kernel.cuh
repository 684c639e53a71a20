// Exact streaming attention forward, one 128-row query tile per CTA, for
// sm_103a: TMA-staged Q/K/V tiles, tcgen05 MMAs accumulating in tensor
// memory, and warp-specialised roles.
//
// Method ("Intermediate and advanced extension", workshop row "Streaming
// attention" and "Logic review before implementation"): S = Q K^T is formed
// one 128-key tile at a time; every query row keeps a running maximum m and a
// rescaled exponential sum l in FP32; P = exp(scale*(S - m)) is rounded to the
// input type and O += P V accumulates in FP32.  When m grows, BOTH l and the
// O accumulator are multiplied by exp(scale*(m_old - m_new)).  The causal
// mask keeps the diagonal; key tiles wholly in a row block's future are never
// visited.  The epilogue writes O / l and lse = scale*m + ln l.
//
// Roles (192 threads):
//   warps 0-3  softmax: thread t owns query row t of the tile (tensor-memory
//              lane t); reads S, updates (m, l), writes P to tensor memory,
//              rescales its O row when needed, and runs the epilogue.
//   warp 4     TMA producer: Q once, then K_j and V_j into two-stage rings.
//   warp 5     tensor-memory allocator and MMA issuer.
//
// Tensor memory (512 columns x 128 lanes, FP32 cells):
//   [  0,128) S buffer 0     [128,256) S buffer 1
//   [256,256+D) O accumulator
//   [384,448) P buffer 0     [448,512) P buffer 1   (two 16-bit values per cell)
//
// Lazy rescaling: m is only moved when the tile maximum exceeds it by more
// than 8 in log2 units; until then P = exp2(scale*log2e*(s - m)) <= 256, which
// FP16/BF16 and the FP32 sums hold exactly enough.  The final O / l and lse
// use the same m as every P, so the result is unchanged.
#pragma once

#include <cstdint>
#include <cuda.h>

#include "sm103_ptx.cuh"

namespace etattn {

struct FwdParams {
  void* o;
  float* lse;
  int64_t o_sb, o_sh, o_sn;      // element strides of o (batch/sequence, head, token); d-stride 1
  int64_t lse_sb, lse_sh;        // element strides of lse (batch, head); token stride 1
  const int* cu_seqlens;         // packed batch offsets, or nullptr for the batched layout
  int N;                         // tokens per sequence (batched)
  int total_tokens;              // packed batch: total tokens T
  int max_seqlen;                // packed batch: bound on every length
  int Hq, group;                 // query heads, Hq / Hkv
  int causal;
  float scale;                   // logit scale
  float scale_log2;              // scale * log2(e)
  int* status;                   // device status word
  int hn_swapped;                // bit 0/1/2: the q/k/v tensor map orders (d, head, token, batch)
                                 // instead of (d, token, head, batch)
};

// TMA load of one box at (d offset, token row, head, batch) for a map whose
// middle axes may be ordered either way.
__device__ __forceinline__ void tma_load_tile(void* dst, const CUtensorMap* map, uint64_t* bar, int d0, int row,
                                              int head, int batch, bool swapped) {
  if (swapped)
    tma_load_4d(dst, map, bar, d0, head, row, batch);
  else
    tma_load_4d(dst, map, bar, d0, row, head, batch);
}

template <int D>
struct TileCfg {
  static constexpr int BM = 128;                       // query rows per tile
  static constexpr int BN = 128;                       // keys per tile
  static constexpr int SW_ELEMS = D >= 64 ? 64 : 32;   // elements per swizzled smem row
  static constexpr int SW_BYTES = SW_ELEMS * 2;        // 128 B (D >= 64) or 64 B (D = 32)
  static constexpr uint32_t SWIZZLE = D >= 64 ? kSw128 : kSw64;
  static constexpr int NCHUNK = D / SW_ELEMS;          // TMA boxes per tile along d
  static constexpr int KSTEPS_PER_CHUNK = SW_ELEMS / 16;
  static constexpr int Q_BYTES = BM * D * 2;
  static constexpr int KV_BYTES = BN * D * 2;
  static constexpr int STAGES = 2;
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = Q_BYTES;
  static constexpr int OFF_V = Q_BYTES + STAGES * KV_BYTES;
  static constexpr int SMEM_BYTES = Q_BYTES + 2 * STAGES * KV_BYTES + 1024;  // + alignment slack
  static constexpr uint32_t SBO = 8 * SW_BYTES;        // stride between 8-row swizzle atoms
  static constexpr uint32_t TM_S0 = 0, TM_O = 256, TM_P0 = 384;
  static constexpr int THREADS = 192;
};

__device__ __forceinline__ void fence_regs32(uint32_t* r) {
  asm volatile("" : ETATTN_RW8(r, 0), ETATTN_RW8(r, 8), ETATTN_RW8(r, 16), ETATTN_RW8(r, 24));
}

template <int D>
struct SmemBarriers {
  uint64_t q_full;
  uint64_t k_full[2], k_empty[2];
  uint64_t v_full[2], v_empty[2];
  uint64_t s_full[2], s_empty[2];
  uint64_t p_full[2], pv_done[2];
  uint32_t tmem_base;
};

// ----------------------------------------------------------------- producer
template <int D>
__device__ __forceinline__ void producer_role(const CUtensorMap* tmQ, const CUtensorMap* tmK,
                                              const CUtensorMap* tmV, SmemBarriers<D>& sb, uint8_t* smem,
                                              int q_row0, int kv_row0, int h, int hk, int bcoord, int n_kv,
                                              int hn_swapped, int* status) {
  using C = TileCfg<D>;
  const int lane = threadIdx.x & 31;
  const bool swq = hn_swapped & 1, swk = (hn_swapped >> 1) & 1, swv = (hn_swapped >> 2) & 1;
  if (lane == 0) {
    mbar_arrive_expect_tx(&sb.q_full, C::Q_BYTES);
#pragma unroll
    for (int c = 0; c < C::NCHUNK; ++c)
      tma_load_tile(smem + C::OFF_Q + c * C::BM * C::SW_BYTES, tmQ, &sb.q_full, c * C::SW_ELEMS, q_row0, h,
                    bcoord, swq);
  }
  for (int j = 0; j < n_kv; ++j) {
    const int st = j & 1;
    const uint32_t ph_prev = ((j - 2) >> 1) & 1;
    if (j >= 2 && !__all_sync(0xffffffffu, mbar_wait(&sb.k_empty[st], ph_prev, status))) return;
    if (lane == 0) {
      mbar_arrive_expect_tx(&sb.k_full[st], C::KV_BYTES);
#pragma unroll
      for (int c = 0; c < C::NCHUNK; ++c)
        tma_load_tile(smem + C::OFF_K + st * C::KV_BYTES + c * C::BN * C::SW_BYTES, tmK, &sb.k_full[st],
                      c * C::SW_ELEMS, kv_row0 + j * C::BN, hk, bcoord, swk);
    }
    if (j >= 2 && !__all_sync(0xffffffffu, mbar_wait(&sb.v_empty[st], ph_prev, status))) return;
    if (lane == 0) {
      mbar_arrive_expect_tx(&sb.v_full[st], C::KV_BYTES);
#pragma unroll
      for (int c = 0; c < C::NCHUNK; ++c)
        tma_load_tile(smem + C::OFF_V + st * C::KV_BYTES + c * C::BN * C::SW_BYTES, tmV, &sb.v_full[st],
                      c * C::SW_ELEMS, kv_row0 + j * C::BN, hk, bcoord, swv);
    }
    __syncwarp();
  }
}

// ----------------------------------------------------------------- MMA issuer
template <int D>
__device__ __forceinline__ bool issue_pv(SmemBarriers<D>& sb, uint8_t* smem, uint32_t tmem, int i,
                                         uint32_t idesc_pv, int* status) {
  using C = TileCfg<D>;
  const int st = i & 1;
  const uint32_t ph = (i >> 1) & 1;
  bool ok = mbar_wait(&sb.v_full[st], ph, status) && mbar_wait(&sb.p_full[st], ph, status);
  if (!__all_sync(0xffffffffu, ok)) return false;
  tc_fence_after();
  if ((threadIdx.x & 31) == 0) {
    const uint32_t v_base = smem_u32(smem + C::OFF_V + st * C::KV_BYTES);
    const uint32_t p_base = tmem + C::TM_P0 + st * 64;
#pragma unroll
    for (int kk = 0; kk < C::BN / 16; ++kk) {
      // V is MN-major (d contiguous): 16 keys per step = 16 swizzled rows;
      // LBO steps between d-chunks, SBO between 8-row groups.
      const uint64_t vdesc = smem_desc(v_base + kk * 16 * C::SW_BYTES, C::BN * C::SW_BYTES, C::SBO, C::SWIZZLE);
      mma_ts(tmem + C::TM_O, p_base + kk * 8, vdesc, idesc_pv, (i > 0 || kk > 0) ? 1u : 0u);
    }
    mma_commit(&sb.pv_done[st]);
    mma_commit(&sb.v_empty[st]);
  }
  __syncwarp();
  return true;
}

template <int D>
__device__ __forceinline__ void mma_role(SmemBarriers<D>& sb, uint8_t* smem, uint32_t tmem, int n_kv,
                                         uint32_t idesc_s, uint32_t idesc_pv, int* status) {
  using C = TileCfg<D>;
  if (!__all_sync(0xffffffffu, mbar_wait(&sb.q_full, 0, status))) return;
  const uint32_t q_base = smem_u32(smem + C::OFF_Q);
  for (int j = 0; j < n_kv; ++j) {
    const int st = j & 1;
    bool ok = mbar_wait(&sb.k_full[st], (j >> 1) & 1, status);
    if (j >= 2) ok = ok && mbar_wait(&sb.s_empty[st], ((j - 2) >> 1) & 1, status);
    if (!__all_sync(0xffffffffu, ok)) return;
    tc_fence_after();
    if ((threadIdx.x & 31) == 0) {
      const uint32_t k_base = smem_u32(smem + C::OFF_K + st * C::KV_BYTES);
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        // Q and K are K-major (d contiguous): a 16-element step moves 32 bytes
        // inside a swizzled row, and a new d-chunk starts a new box.
        const int c = kk / C::KSTEPS_PER_CHUNK, w = kk % C::KSTEPS_PER_CHUNK;
        const uint64_t qdesc = smem_desc(q_base + c * C::BM * C::SW_BYTES + w * 32, 16, C::SBO, C::SWIZZLE);
        const uint64_t kdesc = smem_desc(k_base + c * C::BN * C::SW_BYTES + w * 32, 16, C::SBO, C::SWIZZLE);
        mma_ss(tmem + C::TM_S0 + st * 128, qdesc, kdesc, idesc_s, kk > 0 ? 1u : 0u);
      }
      mma_commit(&sb.s_full[st]);
      mma_commit(&sb.k_empty[st]);
    }
    __syncwarp();
    if (j >= 1 && !issue_pv<D>(sb, smem, tmem, j - 1, idesc_pv, status)) return;
  }
  if (!issue_pv<D>(sb, smem, tmem, n_kv - 1, idesc_pv, status)) return;
  // Drain: wait for the commit arrivals nobody else consumes (the last two
  // iterations' stage releases and PV completions) so that no arrival can
  // land in shared memory after the CTA exits.
  for (int i = n_kv >= 2 ? n_kv - 2 : 0; i < n_kv; ++i) {
    const uint32_t ph = (i >> 1) & 1;
    const bool ok = mbar_wait(&sb.k_empty[i & 1], ph, status) && mbar_wait(&sb.v_empty[i & 1], ph, status) &&
                    mbar_wait(&sb.pv_done[i & 1], ph, status);
    if (!__all_sync(0xffffffffu, ok)) return;
  }
}

// ----------------------------------------------------------------- softmax / correction / epilogue
template <bool BF16>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  return BF16 ? pack_bf16x2(lo, hi) : pack_f16x2(lo, hi);
}

template <int D, bool BF16>
__device__ __forceinline__ void softmax_role(SmemBarriers<D>& sb, uint32_t tmem, const FwdParams& p, int q_tile,
                                             int n_kv, int L, int tok0, int b, int h) {
  using C = TileCfg<D>;
  constexpr uint32_t FULL = 0xffffffffu;
  const int t = threadIdx.x;  // query row inside the tile = tensor-memory lane
  const uint32_t lane_off = (uint32_t)((t >> 5) * 32) << 16;
  const int row_pos = q_tile * C::BM + t;  // logical position inside the sequence
  const float c2 = p.scale_log2;
  int* status = p.status;
  // Last eligible key position of this row: the diagonal under the causal
  // mask, and never past the end of the sequence.
  const int last_key = p.causal ? min(row_pos, L - 1) : L - 1;
  float m_run = -INFINITY;  // running maximum of the raw scores (scale > 0)
  float l_run = 0.f;        // sum of exp2(c2 * (s - m_run)) over the keys seen

  for (int j = 0; j < n_kv; ++j) {
    const int st = j & 1;
    if (!__all_sync(FULL, mbar_wait(&sb.s_full[st], (j >> 1) & 1, status))) return;
    tc_fence_after();
    uint32_t sr[C::BN];
    const uint32_t s_addr = tmem + C::TM_S0 + st * 128 + lane_off;
    tmem_ld_x32(s_addr + 0, sr + 0);
    tmem_ld_x32(s_addr + 32, sr + 32);
    tmem_ld_x32(s_addr + 64, sr + 64);
    tmem_ld_x32(s_addr + 96, sr + 96);
    tmem_ld_wait32(sr);
    fence_regs32(sr + 32);
    fence_regs32(sr + 64);
    fence_regs32(sr + 96);
    tc_fence_before();
    mbar_arrive(&sb.s_empty[st]);  // S buffer may be overwritten by S_{j+2}

    float s[C::BN];
#pragma unroll
    for (int i = 0; i < C::BN; ++i) s[i] = __uint_as_float(sr[i]);
    // Mask keys past the diagonal (causal) or past the sequence end.
    const int lim = last_key - j * C::BN;
    if (lim < C::BN - 1) {
#pragma unroll
      for (int i = 0; i < C::BN; ++i) s[i] = (i > lim) ? -INFINITY : s[i];
    }
    float mx0 = s[0], mx1 = s[1], mx2 = s[2], mx3 = s[3];
#pragma unroll
    for (int i = 4; i < C::BN; i += 4) {
      mx0 = fmaxf(mx0, s[i]);
      mx1 = fmaxf(mx1, s[i + 1]);
      mx2 = fmaxf(mx2, s[i + 2]);
      mx3 = fmaxf(mx3, s[i + 3]);
    }
    const float m_tile = fmaxf(fmaxf(mx0, mx1), fmaxf(mx2, mx3));
    const float m_new = fmaxf(m_run, m_tile);
    // Lazy rescale: move the reference maximum only when it grows by more
    // than 8 in log2 units (always on the first tile).
    const bool rescale = (j == 0) || (m_new - m_run) * c2 > 8.f;
    float alpha = 1.f;
    if (rescale) {
      alpha = (j == 0) ? 0.f : ex2_approx((m_run - m_new) * c2);
      m_run = m_new;
    }
    const float neg_mc = -m_run * c2;
    uint32_t pk[C::BN / 2];
    float rs0 = 0.f, rs1 = 0.f;
#pragma unroll
    for (int i = 0; i < C::BN / 2; ++i) {
      const float p0 = ex2_approx(fmaf(s[2 * i], c2, neg_mc));
      const float p1 = ex2_approx(fmaf(s[2 * i + 1], c2, neg_mc));
      rs0 += p0;
      rs1 += p1;
      pk[i] = pack2<BF16>(p0, p1);
    }
    l_run = l_run * alpha + (rs0 + rs1);

    // P buffer st was last read by PV_{j-2}.
    if (j >= 2) {
      if (!__all_sync(FULL, mbar_wait(&sb.pv_done[st], ((j - 2) >> 1) & 1, status))) return;
      tc_fence_after();
    }
    const uint32_t p_addr = tmem + C::TM_P0 + st * 64 + lane_off;
    tmem_st_x32(p_addr, pk);
    tmem_st_x32(p_addr + 32, pk + 32);

    // Correction: O_acc *= alpha for rows whose maximum moved, after PV_{j-1}
    // has landed and before PV_j is issued.
    if (j > 0 && __any_sync(FULL, rescale)) {
      if (!__all_sync(FULL, mbar_wait(&sb.pv_done[(j - 1) & 1], ((j - 1) >> 1) & 1, status))) return;
      tc_fence_after();
#pragma unroll
      for (int c = 0; c < D; c += 32) {
        uint32_t o[32];
        tmem_ld_x32(tmem + C::TM_O + lane_off + c, o);
        tmem_ld_wait32(o);
#pragma unroll
        for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
        tmem_st_x32(tmem + C::TM_O + lane_off + c, o);
      }
    }
    tmem_st_wait();
    tc_fence_before();
    mbar_arrive(&sb.p_full[st]);
  }

  // Epilogue: O = O_acc / l in the input type, lse = scale * m + ln l.
  const int last = n_kv - 1;
  if (!__all_sync(FULL, mbar_wait(&sb.pv_done[last & 1], (last >> 1) & 1, status))) return;
  tc_fence_after();
  const bool valid = row_pos < L;
  const float inv_l = 1.f / l_run;
  uint8_t* orow = reinterpret_cast<uint8_t*>(p.o) +
                  2 * ((int64_t)b * p.o_sb + (int64_t)h * p.o_sh + (int64_t)(tok0 + row_pos) * p.o_sn);
#pragma unroll
  for (int c = 0; c < D; c += 32) {
    uint32_t o[32];
    tmem_ld_x32(tmem + C::TM_O + lane_off + c, o);
    tmem_ld_wait32(o);
    uint32_t w[16];
#pragma unroll
    for (int i = 0; i < 16; ++i)
      w[i] = pack2<BF16>(__uint_as_float(o[2 * i]) * inv_l, __uint_as_float(o[2 * i + 1]) * inv_l);
    if (valid) {
      uint4* dst = reinterpret_cast<uint4*>(orow + c * 2);
      dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
      dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
      dst[2] = make_uint4(w[8], w[9], w[10], w[11]);
      dst[3] = make_uint4(w[12], w[13], w[14], w[15]);
    }
  }
  if (valid && p.lse != nullptr)
    p.lse[(int64_t)b * p.lse_sb + (int64_t)h * p.lse_sh + tok0 + row_pos] = m_run * p.scale + __logf(l_run);
}

// ----------------------------------------------------------------- kernel
// Grid: x = (batch or sequence) * Hq + head, y = query tile counted from the
// last one, so that the longest causal rows are dispatched first.
template <int D, bool BF16>
__global__ void __launch_bounds__(192, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const FwdParams p) {
  using C = TileCfg<D>;
  __shared__ SmemBarriers<D> sb;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

  const int bh = blockIdx.x;
  const int h = bh % p.Hq, b = bh / p.Hq;
  const int q_tile = (int)gridDim.y - 1 - (int)blockIdx.y;
  int L = p.N, tok0 = 0, bcoord = b;
  if (p.cu_seqlens != nullptr) {
    const int s0 = p.cu_seqlens[b], s1 = p.cu_seqlens[b + 1];
    if (s0 < 0 || s1 < s0 || s1 > p.total_tokens || s1 - s0 > p.max_seqlen) {
      if (threadIdx.x == 0) atomicCAS(p.status, 0, (int)kDevBadSeqlens);
      return;
    }
    L = s1 - s0;
    tok0 = s0;
    bcoord = 0;
  }
  if (q_tile * C::BM >= L) return;  // uniform across the CTA
  const int n_kv = p.causal ? q_tile + 1 : (L + C::BN - 1) / C::BN;
  const int warp = threadIdx.x >> 5;

  if (threadIdx.x == 0) {
    mbar_init(&sb.q_full, 1);
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sb.k_full[i], 1);
      mbar_init(&sb.k_empty[i], 1);
      mbar_init(&sb.v_full[i], 1);
      mbar_init(&sb.v_empty[i], 1);
      mbar_init(&sb.s_full[i], 1);
      mbar_init(&sb.s_empty[i], 128);
      mbar_init(&sb.p_full[i], 128);
      mbar_init(&sb.pv_done[i], 1);
    }
    fence_mbar_init();
  }
  if (warp == 4 && (threadIdx.x & 31) == 0) {
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
  }
  if (warp == 5) {
    tmem_alloc(&sb.tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sb.tmem_base;

  if (warp < 4) {
    softmax_role<D, BF16>(sb, tmem, p, q_tile, n_kv, L, tok0, b, h);
  } else if (warp == 4) {
    producer_role<D>(&tmQ, &tmK, &tmV, sb, smem, tok0 + q_tile * C::BM, tok0, h, h / p.group, bcoord, n_kv,
                     p.hn_swapped, p.status);
  } else {
    constexpr uint32_t ab = BF16 ? 1u : 0u;
    constexpr uint32_t idesc_s = instr_desc_f16(128, C::BN, ab, false, false);
    constexpr uint32_t idesc_pv = instr_desc_f16(128, D, ab, false, true);
    mma_role<D>(sb, smem, tmem, n_kv, idesc_s, idesc_pv, p.status);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace etattn

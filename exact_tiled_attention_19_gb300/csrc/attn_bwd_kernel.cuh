// Attention backward for sm_103a: dQ, dK, dV of sum(dO * O), recomputing the
// probabilities from the logsumexp the forward pass saved.
//
// Method ("Attention algorithms and data movement", lesson 03: recompute the
// probabilities and differentiate the normalised row from the saved
// normalisation state; the forward's masks, unequal lengths, windows and GQA
// map of lessons 04, 05 and 07):
//   P_ij  = exp(scale * <q_i, k_j> - lse_i) on eligible pairs, else 0
//   dV_j += sum_i P_ij dO_i            dP_ij = <dO_i, v_j>
//   dS_ij = scale * P_ij (dP_ij - D_i),  D_i = <dO_i, O_i>  (one launch before)
//   dK_j += sum_i dS_ij q_i            dQ_i += sum_j dS_ij k_j
//
// A CTA owns 128 keys of one (batch, key/value head) and walks every query
// head of the group and every query block of 128 rows that can read one of
// its keys.  dK and dV accumulate in tensor memory for the whole walk and are
// written once; each step's dQ contribution is added to an FP32 buffer with
// TMA reduce-adds (a later launch converts it to the input type).
//
// The scores are formed transposed (keys as rows), so that one thread owns
// one key for P and dS and the dK / dV products take P^T and dS^T straight
// from tensor memory:
//   S^T   = K Q^T      (A = K, B = Q, both K-major in shared memory)
//   dP^T  = V dO^T     (A = V, B = dO, both K-major)
//   dV   += P^T dO     (A = P^T in tensor memory, B = dO MN-major)
//   dK   += dS^T Q     (A = dS^T in tensor memory, B = Q MN-major)
//   dQ_i  = dS K       (A = dS in shared memory, MN-major; B = K MN-major)
//
// Roles (512 threads, 4 warpgroups):
//   warpgroups 0, 1  thread t owns key row t; warpgroup c takes the query
//                    columns [64c, 64c + 64) of each step: P^T from S^T, then
//                    dS^T from dP^T (into tensor memory and, transposed, into
//                    shared memory for dQ).  Epilogue: dK (0) and dV (1).
//   warpgroup 2      thread t owns query row t of dQ_i: reads it from tensor
//                    memory; each warp stages its 32 rows in shared memory
//                    32 columns at a time and its lane 0 adds each staged box
//                    to the FP32 buffer, the four warps independently.
//   warp 12          TMA: K and V once; per step Q with its lse and dO with
//                    its D, two stages each.  At D = 128 the dS tile of a step
//                    takes the place of its dO tile once dV has read it.
//   warp 13          tensor-memory allocation and MMA issue (one thread).
//
// Tensor memory (512 columns): dK [0, D), dV [128, 128 + D), S^T [256, 384)
// (P^T of query columns [64c, 64c + 64) packed into [256 + 64c, 256 + 64c +
// 32)), dP^T [384, 512) (dS^T packed likewise at 384 + 64c; dQ_i over it once
// dK has read dS^T).  The dS phase reads P^T back first, so the next step's
// S^T is issued right after dV_i and that step's P phase finds its scores
// ready as soon as this dS phase ends; only the next dP^T, which overwrites
// dQ_i, waits for the dQ read-out.  Per step the tensor core runs
// dP_i, dV_i, S_(i+1), dK_i, dQ_i.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_fp16.h>

#include "sm103_ptx.cuh"

namespace etattn {

struct BwdParams {
  void* dk;
  void* dv;
  int64_t dk_sb, dk_sh, dk_sn;   // element strides of dk (batch, head, token); d-stride 1
  int64_t dv_sb, dv_sh, dv_sn;
  const float* nlse2;            // [B * Hq][Nq_pad]: -lse * log2(e); -inf where a row reads no key
  const float* nsd;              // [B * Hq][Nq_pad]: -scale * <dO, O>; 0 on padding rows
  int Nq, Nk, Nq_pad;            // Nq_pad: Nq rounded up to 128
  int Hq, group;
  int win_left, win_right;       // as in the forward pass (causal: win_right = 0)
  float scale, scale_log2;
  int* status;
  int hn_swapped;                // bit 0/1/2/3: the q/k/v/dO tensor map orders (d, head, token, batch)
  int grid_x, grid_y;            // key blocks, KV heads (the logical grid's x and y extents)
  int sched_q, sched_rem;        // > 0: 1-D launch in grouped longest-first order (bwd_cta_coords)
};

// The logical (key block, KV head, batch) of this CTA.  With sched_q > 0 the
// grid is launched 1-D and the (KV head, batch) pairs (head fastest) are cut
// into contiguous groups of near-equal size (sched_rem groups of sched_q + 1
// pairs, then groups of sched_q); a group's CTAs come one after another,
// ordered by key block and then by pair.  Key block 0 is read by the most
// query blocks, so every group's longest CTAs start first and the last CTAs
// to start are the shortest ones of the last group, while the CTAs running at
// any time read the Q, dO and dQ rows of one group.  (Plain divisions: a
// backward CTA runs for many steps, and the map is a few hundred cycles.)
__device__ __forceinline__ int3 bwd_cta_coords(const BwdParams& p) {
  if (p.sched_q <= 0) return make_int3((int)blockIdx.x, (int)blockIdx.y, (int)blockIdx.z);
  const uint32_t lin = blockIdx.x, gx = (uint32_t)p.grid_x, gy = (uint32_t)p.grid_y;
  const uint32_t q = (uint32_t)p.sched_q, big = (uint32_t)p.sched_rem * (q + 1);  // pairs in the larger groups
  const uint32_t pi = lin / gx;  // CTA lin lies in the group holding the pi-th pair
  const bool large = pi < big;
  const uint32_t size = large ? q + 1 : q;
  const uint32_t first = large ? pi / size * size : big + (pi - big) / q * q;
  const uint32_t r = lin - first * gx;
  const uint32_t x = r / size;
  const uint32_t pair = first + (r - x * size);
  const uint32_t z = pair / gy;
  return make_int3((int)x, (int)(pair - z * gy), (int)z);
}

template <int D>
struct BwdCfg {
  static constexpr int BN = 128;                       // keys per CTA
  static constexpr int BM = 128;                       // query rows per step
  static constexpr int SW_ELEMS = D >= 64 ? 64 : 32;   // elements per swizzled row of a Q/K/V/dO tile
  static constexpr int SW_BYTES = SW_ELEMS * 2;
  static constexpr uint32_t SWIZZLE = D >= 64 ? kSw128 : kSw64;
  static constexpr int NCHUNK = D / SW_ELEMS;
  static constexpr int KSTEPS_PER_CHUNK = SW_ELEMS / 16;
  static constexpr int TILE = 128 * D * 2;             // one 128-row tile
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = TILE;
  static constexpr int OFF_Q = 2 * TILE;               // two stages
  static constexpr int OFF_DO = 4 * TILE;              // two stages
  static constexpr int DS_BYTES = 128 * 128 * 2;       // dS, 128 queries x 128 keys, MN-major, 128B swizzle
  static constexpr bool DS_IN_DO = TILE == DS_BYTES;   // D = 128: dS of a step over its dO stage
  static constexpr int OFF_DS = 6 * TILE;              // otherwise a tile of its own
  // dQ staging: one box of 32 rows x 32 FP32 (4 KB) per warp of the dQ warpgroup.
  static constexpr int OFF_STAGE = OFF_DS + (DS_IN_DO ? 0 : DS_BYTES);
  static constexpr int STAGE_BYTES = 4 * 32 * 128;
  static constexpr int OFF_LSE = OFF_STAGE + STAGE_BYTES;  // two stages of 128 floats
  static constexpr int OFF_NSD = OFF_LSE + 2 * 512;        // two stages of 128 floats
  static constexpr int SMEM_BYTES = OFF_NSD + 2 * 512 + 1024;
  static constexpr uint32_t SBO = 8 * SW_BYTES;
  static constexpr uint32_t TM_DK = 0, TM_DV = 128, TM_S = 256, TM_DP = 384, TMEM_COLS = 512;
  static constexpr int THREADS = 512;
  static constexpr int PRODUCER_WARP = 12, MMA_WARP = 13;
  // Register split: 512 threads launch with 128 registers each; the dQ
  // warpgroup (which holds a whole dQ row) grows to 168 and the TMA / MMA
  // warpgroup shrinks to 88.  128 + 128 + 168 + 88 = 4 * 128.
  static constexpr int LAUNCH_REGS = 128, DQ_REGS = 168, CTRL_REGS = 88;
  static_assert(2 * LAUNCH_REGS + DQ_REGS + CTRL_REGS == 4 * LAUNCH_REGS, "register split must add up");
  // Shared-memory offset of the dS tile of a step whose stages are `slot`.
  static constexpr int ds_offset(int slot) { return DS_IN_DO ? OFF_DO + slot * TILE : OFF_DS; }
  // Tensor-memory column of the packed P^T / dS^T of query columns
  // [16 kk, 16 kk + 16): half c = kk / 4 lives at 64 c.
  static constexpr uint32_t packed_col(int kk) { return (uint32_t)((kk >> 2) * 64 + (kk & 3) * 8); }
};

struct BwdBarriers {
  uint64_t kv_full;
  uint64_t q_full[2], q_empty[2];
  uint64_t do_full[2], do_empty[2];  // do_empty: the stage's dO and dS are read (after dQ_i)
  uint64_t dv_done;                  // dV_i is done (dO_i read by the tensor core for the last time)
  uint64_t s_full, dp_full;          // S^T / dP^T of the step are in tensor memory
  uint64_t p_ready, ds_ready;        // P^T / dS^T (and dS in shared memory) written (256 arrivals)
  uint64_t p_read;                   // P^T read back by the dS phase (256 arrivals)
  uint64_t dq_full;                  // dQ_i in tensor memory (the step's dK and dQ products are done)
  uint64_t dq_empty;                 // dQ_i read out (128 arrivals)
  uint64_t kv_done;                  // last dK / dV product done
  uint64_t fin;                      // every MMA the CTA issued has completed
  uint32_t tmem_base;
};

// Steps of a CTA: query heads h0 .. h0 + group - 1, each over query blocks
// qb_lo .. qb_lo + n_qb - 1.
struct BwdUnit {
  int b, hk, h0, kb0;            // batch, kv head, first query head, first key
  int qb_lo, n_qb, steps;
  __device__ __forceinline__ int head(int i) const { return h0 + i / n_qb; }
  __device__ __forceinline__ int q0(int i) const { return (qb_lo + i % n_qb) * 128; }
};

__device__ __forceinline__ void tma_tile(void* dst, const CUtensorMap* map, uint64_t* bar, int d0, int row, int head,
                                         int batch, bool swapped) {
  if (swapped)
    tma_load_4d(dst, map, bar, d0, head, row, batch);
  else
    tma_load_4d(dst, map, bar, d0, row, head, batch);
}

template <int D>
__device__ __forceinline__ void bwd_producer(const CUtensorMap* tmQ, const CUtensorMap* tmK, const CUtensorMap* tmV,
                                             const CUtensorMap* tmDO, BwdBarriers& sb, uint8_t* smem,
                                             const BwdUnit u, const BwdParams& p, int& q_issued, int& do_issued) {
  using C = BwdCfg<D>;
  const bool swq = p.hn_swapped & 1, swk = p.hn_swapped & 2, swv = p.hn_swapped & 4, swd = p.hn_swapped & 8;
  mbar_arrive_expect_tx(&sb.kv_full, 2 * C::TILE);
#pragma unroll
  for (int c = 0; c < C::NCHUNK; ++c) {
    tma_tile(smem + C::OFF_K + c * 128 * C::SW_BYTES, tmK, &sb.kv_full, c * C::SW_ELEMS, u.kb0, u.hk, u.b, swk);
    tma_tile(smem + C::OFF_V + c * 128 * C::SW_BYTES, tmV, &sb.kv_full, c * C::SW_ELEMS, u.kb0, u.hk, u.b, swv);
  }
  for (int i = 0; i < u.steps; ++i) {
    const int h = u.head(i), q0 = u.q0(i), slot = i & 1;
    const int64_t vec_row = ((int64_t)u.b * p.Hq + h) * p.Nq_pad + q0;
    if (i >= 2 && !mbar_wait(&sb.q_empty[slot], ((i >> 1) - 1) & 1, p.status)) return;
    mbar_arrive_expect_tx(&sb.q_full[slot], C::TILE + 512);
#pragma unroll
    for (int c = 0; c < C::NCHUNK; ++c)
      tma_tile(smem + C::OFF_Q + slot * C::TILE + c * 128 * C::SW_BYTES, tmQ, &sb.q_full[slot], c * C::SW_ELEMS, q0,
               h, u.b, swq);
    bulk_load(smem + C::OFF_LSE + slot * 512, p.nlse2 + vec_row, 512, &sb.q_full[slot]);
    q_issued = i + 1;
    if (i >= 2 && !mbar_wait(&sb.do_empty[slot], ((i >> 1) - 1) & 1, p.status)) return;
    mbar_arrive_expect_tx(&sb.do_full[slot], C::TILE + 512);
#pragma unroll
    for (int c = 0; c < C::NCHUNK; ++c)
      tma_tile(smem + C::OFF_DO + slot * C::TILE + c * 128 * C::SW_BYTES, tmDO, &sb.do_full[slot], c * C::SW_ELEMS,
               q0, h, u.b, swd);
    bulk_load(smem + C::OFF_NSD + slot * 512, p.nsd + vec_row, 512, &sb.do_full[slot]);
    do_issued = i + 1;
  }
}

// Waits (bounded) until the key/value tiles and the last load issued into each
// Q and dO stage have landed, so that no copy writes shared memory after the
// CTA exits (immediate after a normal run, whose consumers saw these phases).
template <int D>
__device__ __forceinline__ void bwd_producer_settle(BwdBarriers& sb, int q_issued, int do_issued) {
  mbar_wait(&sb.kv_full, 0, nullptr);
  for (int t = q_issued > 2 ? q_issued - 2 : 0; t < q_issued; ++t) mbar_wait(&sb.q_full[t & 1], (t >> 1) & 1, nullptr);
  for (int t = do_issued > 2 ? do_issued - 2 : 0; t < do_issued; ++t)
    mbar_wait(&sb.do_full[t & 1], (t >> 1) & 1, nullptr);
}

template <int D>
__device__ __forceinline__ void bwd_mma(BwdBarriers& sb, uint8_t* smem, uint32_t tmem, const BwdUnit u,
                                        uint32_t ab, int* status) {
  using C = BwdCfg<D>;
  const uint32_t id_s = instr_desc_f16(128, 128, ab, false, false);  // S^T, dP^T
  const uint32_t id_kv = instr_desc_f16(128, D, ab, false, true);    // dV, dK: A in tensor memory, B MN-major
  const uint32_t id_q = instr_desc_f16(128, D, ab, true, true);      // dQ: A = dS MN-major, B = K MN-major
  // K-major views (S^T, dP^T) and MN-major views (dV, dK, dQ) of the tiles.
  const uint64_t k_kmaj = smem_desc(smem_u32(smem + C::OFF_K), 16, C::SBO, C::SWIZZLE);
  const uint64_t v_kmaj = smem_desc(smem_u32(smem + C::OFF_V), 16, C::SBO, C::SWIZZLE);
  const uint64_t q_kmaj = smem_desc(smem_u32(smem + C::OFF_Q), 16, C::SBO, C::SWIZZLE);
  const uint64_t do_kmaj = smem_desc(smem_u32(smem + C::OFF_DO), 16, C::SBO, C::SWIZZLE);
  const uint64_t k_mn = smem_desc(smem_u32(smem + C::OFF_K), 128 * C::SW_BYTES, C::SBO, C::SWIZZLE);
  const uint64_t q_mn = smem_desc(smem_u32(smem + C::OFF_Q), 128 * C::SW_BYTES, C::SBO, C::SWIZZLE);
  const uint64_t do_mn = smem_desc(smem_u32(smem + C::OFF_DO), 128 * C::SW_BYTES, C::SBO, C::SWIZZLE);
  const uint64_t ds_mn0 = smem_desc(smem_u32(smem + C::ds_offset(0)), 128 * 128, 1024, kSw128);
  const uint64_t ds_mn1 = smem_desc(smem_u32(smem + C::ds_offset(1)), 128 * 128, 1024, kSw128);
  const uint64_t slot_step = (uint64_t)(C::TILE >> 4);
  const uint32_t tDK = tmem + C::TM_DK, tDV = tmem + C::TM_DV, tS = tmem + C::TM_S, tDP = tmem + C::TM_DP;

  // S^T of step i into its region (K-major Q of the step's stage).
  auto issue_s = [&](int i) -> bool {
    const int slot = i & 1;
    if (!mbar_wait(&sb.q_full[slot], (i >> 1) & 1, status)) return false;
    tc_fence_after();
    const uint64_t q_k = q_kmaj + slot * slot_step;
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      const uint64_t off =
          (uint64_t)(((kk / C::KSTEPS_PER_CHUNK) * 128 * C::SW_BYTES + (kk % C::KSTEPS_PER_CHUNK) * 32) >> 4);
      mma_ss(tS, k_kmaj + off, q_k + off, id_s, kk > 0 ? 1u : 0u);
    }
    mma_commit(&sb.s_full);
    return true;
  };
  if (!mbar_wait(&sb.kv_full, 0, status)) return;
  if (!issue_s(0)) return;
  for (int i = 0; i < u.steps; ++i) {
    const int slot = i & 1;
    const uint64_t q_m = q_mn + slot * slot_step;
    const uint64_t do_k = do_kmaj + slot * slot_step, do_m = do_mn + slot * slot_step;
    const uint64_t ds_mn = slot ? ds_mn1 : ds_mn0;
    // dP^T overwrites dQ_(i-1) (same region): it waits for the read-out.
    if (!mbar_wait(&sb.do_full[slot], (i >> 1) & 1, status)) return;
    if (i > 0 && !mbar_wait(&sb.dq_empty, (i - 1) & 1, status)) return;
    tc_fence_after();
    // dP^T = V dO^T.
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      const uint64_t off =
          (uint64_t)(((kk / C::KSTEPS_PER_CHUNK) * 128 * C::SW_BYTES + (kk % C::KSTEPS_PER_CHUNK) * 32) >> 4);
      mma_ss(tDP, v_kmaj + off, do_k + off, id_s, kk > 0 ? 1u : 0u);
    }
    mma_commit(&sb.dp_full);
    // dV += P^T dO over the step's 128 queries, 16 at a time.
    if (!mbar_wait(&sb.p_ready, i & 1, status)) return;
    tc_fence_after();
#pragma unroll
    for (int kk = 0; kk < 8; ++kk)
      mma_ts(tDV, tS + C::packed_col(kk), do_m + (uint64_t)((kk * 16 * C::SW_BYTES) >> 4), id_kv,
             (i > 0 || kk > 0) ? 1u : 0u);
    mma_commit(&sb.dv_done);
    // The next step's S^T over P^T_i, once dV_i (issued above) and the dS
    // phase have read it.
    if (i + 1 < u.steps) {
      if (!mbar_wait(&sb.p_read, i & 1, status)) return;
      if (!issue_s(i + 1)) return;
    }
    // dK += dS^T Q, then dQ_i = dS K over dS^T (read by the dK product just issued).
    if (!mbar_wait(&sb.ds_ready, i & 1, status)) return;
    tc_fence_after();
#pragma unroll
    for (int kk = 0; kk < 8; ++kk)
      mma_ts(tDK, tDP + C::packed_col(kk), q_m + (uint64_t)((kk * 16 * C::SW_BYTES) >> 4), id_kv,
             (i > 0 || kk > 0) ? 1u : 0u);
#pragma unroll
    for (int kk = 0; kk < 8; ++kk)
      mma_ss(tDP, ds_mn + (uint64_t)((kk * 16 * 128) >> 4), k_mn + (uint64_t)((kk * 16 * C::SW_BYTES) >> 4), id_q,
             kk > 0 ? 1u : 0u);
    mma_commit(&sb.dq_full);
    mma_commit(&sb.q_empty[slot]);
    mma_commit(&sb.do_empty[slot]);
  }
  mma_commit(&sb.kv_done);
  // Drain the arrivals no other role consumes.
  for (int i = u.steps > 2 ? u.steps - 2 : 0; i < u.steps; ++i)
    if (!mbar_wait(&sb.q_empty[i & 1], (i >> 1) & 1, status) || !mbar_wait(&sb.do_empty[i & 1], (i >> 1) & 1, status))
      return;
}

__device__ __forceinline__ bool bwd_warp_wait(uint64_t* bar, uint32_t parity, int* status) {
  // Fast path: every lane probes once, and a phase that has already
  // completed (the common case) costs one probe and a vote.  Otherwise lane 0
  // waits (bounded) and hands the outcome to the warp.
  if (__all_sync(0xffffffffu, mbar_try_wait(bar, parity))) return true;
  bool ok = true;
  if ((threadIdx.x & 31) == 0) ok = mbar_wait(bar, parity, status);
  return __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
}

template <bool BF16>
__device__ __forceinline__ uint32_t bwd_pack(float lo, float hi) {
  return BF16 ? pack_bf16x2(lo, hi) : pack_f16x2(lo, hi);
}
// The two 16-bit values of a packed word as floats (low half first).
template <bool BF16>
__device__ __forceinline__ void bwd_unpack(uint32_t w, float& lo, float& hi) {
  if (BF16) {
    lo = __uint_as_float(w << 16);
    hi = __uint_as_float(w & 0xffff0000u);
  } else {
    const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w));
    lo = f.x;
    hi = f.y;
  }
}

// Warpgroups 0 and 1: thread t owns key kb0 + t; warpgroup `half` the query
// columns [64 half, 64 half + 64) of every step.
template <int D, bool BF16>
__device__ __forceinline__ void bwd_compute(BwdBarriers& sb, uint8_t* smem, uint32_t tmem, const BwdUnit u,
                                            const BwdParams& p, int half) {
  using C = BwdCfg<D>;
  constexpr uint32_t FULL = 0xffffffffu;
  const int t = threadIdx.x & 127;
  const uint32_t lane_off = (uint32_t)(((threadIdx.x >> 5) & 3) * 32) << 16;
  const uint32_t tS = tmem + C::TM_S + lane_off + 64 * half, tDP = tmem + C::TM_DP + lane_off + 64 * half;
  const int key = u.kb0 + t;
  // Query rows that may read this key: c - win_left <= key <= c + win_right
  // with c = q + Nk - Nq, i.e. q in [key - delta - win_right, key - delta + win_left].
  const int64_t delta = (int64_t)p.Nk - p.Nq;
  int64_t qlo = (int64_t)key - delta - p.win_right, qhi = (int64_t)key - delta + p.win_left;
  if (qhi > p.Nq - 1) qhi = p.Nq - 1;
  if (qlo < 0) qlo = 0;
  if (key >= p.Nk) qhi = -1;  // padding key: no query reads it
  const float c2 = p.scale_log2, scale = p.scale;
  int* status = p.status;

  for (int i = 0; i < u.steps; ++i) {
    const int q0 = u.q0(i) + 64 * half, slot = i & 1;
    const int64_t lo_rel = qlo - q0, hi_rel = qhi - q0;
    const int lim_lo = lo_rel < -1 ? -1 : (int)lo_rel, lim_hi = hi_rel > 64 ? 64 : (int)hi_rel;
    const bool warp_masked = __any_sync(FULL, lim_lo > 0 || lim_hi < 63);
    const float2* nlse = reinterpret_cast<const float2*>(smem + C::OFF_LSE + slot * 512) + 32 * half;
    const float2* nsd = reinterpret_cast<const float2*>(smem + C::OFF_NSD + slot * 512) + 32 * half;
    // ---- P^T = exp2(c2 * s - lse2), 32 columns at a time, packed over the
    // first of this half's S^T columns.
    if (!bwd_warp_wait(&sb.s_full, i & 1, status)) return;
    tc_fence_after();
#pragma unroll
    for (int ch = 0; ch < 2; ++ch) {
      uint32_t sr[32];
      tmem_ld_x32(tS + 32 * ch, sr);
      tmem_ld_wait32(sr);
      uint32_t pk[16];
#pragma unroll
      for (int j = 0; j < 32; j += 2) {
        const int c = 32 * ch + j;
        const float2 nl = nlse[c / 2];
        float p0, p1;
        fma2(p0, p1, __uint_as_float(sr[j]), __uint_as_float(sr[j + 1]), c2, c2, nl.x, nl.y);
        p0 = ex2_approx(p0);
        p1 = ex2_approx(p1);
        if (warp_masked) {
          p0 = (c < lim_lo || c > lim_hi) ? 0.f : p0;
          p1 = (c + 1 < lim_lo || c + 1 > lim_hi) ? 0.f : p1;
        }
        pk[j / 2] = bwd_pack<BF16>(p0, p1);
      }
      tmem_st_x16(tS + 16 * ch, pk);
    }
    tmem_st_wait();
    tc_fence_before();
    mbar_arrive(&sb.p_ready);

    // ---- dS^T = P (scale * dP - scale * D), over this half's dP^T columns
    // and, as dS, into shared memory: row t = key t, 16-byte unit u of
    // queries 8u .. 8u + 7 of the half at unit u ^ (t mod 8) (128B swizzle).
    if (!bwd_warp_wait(&sb.dp_full, i & 1, status)) return;
    tc_fence_after();
    uint8_t* ds_row = smem + C::ds_offset(slot) + half * (128 * 128) + t * 128;
    // P^T of both chunks, read first so that the next S^T may overwrite it.
    uint32_t pk[32], dr[32];
    tmem_ld_x32(tS, pk);
    tmem_ld_x32(tDP, dr);
    tmem_ld_wait32(pk);
    fence_regs32(dr);
    tc_fence_before();
    mbar_arrive(&sb.p_read);
#pragma unroll
    for (int ch = 0; ch < 2; ++ch) {
      if (ch == 1) {
        tmem_ld_x32(tDP + 32, dr);
        tmem_ld_wait32(dr);
      }
      uint32_t ds[16];
#pragma unroll
      for (int j = 0; j < 32; j += 2) {
        const float2 nd = nsd[(32 * ch + j) / 2];
        float p0, p1, g0, g1;
        bwd_unpack<BF16>(pk[16 * ch + j / 2], p0, p1);
        fma2(g0, g1, __uint_as_float(dr[j]), __uint_as_float(dr[j + 1]), scale, scale, nd.x, nd.y);
        fma2(g0, g1, p0, p1, g0, g1, 0.f, 0.f);
        ds[j / 2] = bwd_pack<BF16>(g0, g1);
      }
      tmem_st_x16(tDP + 16 * ch, ds);
      if (ch == 0) {
        // The dS tile's shared memory is free once dV_i has read dO_i (dS
        // over dO) or dQ_{i-1} has read dS (a tile of its own).
        if (!bwd_warp_wait(&sb.dv_done, i & 1, status)) return;
        if (!C::DS_IN_DO && i > 0 && !bwd_warp_wait(&sb.dq_full, (i - 1) & 1, status)) return;
      }
#pragma unroll
      for (int un = 0; un < 4; ++un) {
        const int unit = 4 * ch + un;
        *reinterpret_cast<uint4*>(ds_row + ((unit ^ (t & 7)) << 4)) =
            make_uint4(ds[4 * un], ds[4 * un + 1], ds[4 * un + 2], ds[4 * un + 3]);
      }
    }
    fence_proxy_async_smem();
    tmem_st_wait();
    tc_fence_before();
    mbar_arrive(&sb.ds_ready);
  }

  // ---- Epilogue: dK (warpgroup 0) or dV (warpgroup 1) rows of this CTA's
  // keys, in the input type.
  const bool valid = key < p.Nk;
  uint8_t* row = half == 0 ? reinterpret_cast<uint8_t*>(p.dk) +
                                 2 * ((int64_t)u.b * p.dk_sb + (int64_t)u.hk * p.dk_sh + (int64_t)key * p.dk_sn)
                           : reinterpret_cast<uint8_t*>(p.dv) +
                                 2 * ((int64_t)u.b * p.dv_sb + (int64_t)u.hk * p.dv_sh + (int64_t)key * p.dv_sn);
  if (u.steps == 0) {  // no query reads these keys
    if (valid) {
#pragma unroll
      for (int c = 0; c < D; c += 8) *reinterpret_cast<uint4*>(row + 2 * c) = make_uint4(0u, 0u, 0u, 0u);
    }
    return;
  }
  if (!bwd_warp_wait(&sb.kv_done, 0, status)) return;
  tc_fence_after();
  const uint32_t tsrc = tmem + (half == 0 ? C::TM_DK : C::TM_DV) + lane_off;
#pragma unroll
  for (int c = 0; c < D; c += 32) {
    uint32_t r[32];
    tmem_ld_x32(tsrc + c, r);
    tmem_ld_wait32(r);
    uint32_t w[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) w[j] = bwd_pack<BF16>(__uint_as_float(r[2 * j]), __uint_as_float(r[2 * j + 1]));
    if (valid) {
      uint4* dst = reinterpret_cast<uint4*>(row + 2 * c);
      dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
      dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
      dst[2] = make_uint4(w[8], w[9], w[10], w[11]);
      dst[3] = make_uint4(w[12], w[13], w[14], w[15]);
    }
  }
}

// Warpgroup 2: thread t owns query row q0 + t of each step's dQ contribution.
// The row is read from tensor memory (which frees it for the next step).
// Each warp then stages its 32 rows, 32 columns at a time, in a swizzled box
// of its own, which its lane 0 adds to the FP32 dQ buffer with a TMA reduce
// (rows past Nq fall outside the map and are dropped) after the warp's
// previous box has left shared memory.  The four warps keep four reduces in
// flight; one 128-row box handed between the warps on mbarriers kept one, and
// the reduces' latency then set the step time.
template <int D>
__device__ __forceinline__ void bwd_dq(BwdBarriers& sb, uint8_t* smem, uint32_t tmem, const BwdUnit u,
                                       const BwdParams& p, const CUtensorMap* tmDQ) {
  using C = BwdCfg<D>;
  const int lane = threadIdx.x & 31, wq = (threadIdx.x >> 5) & 3;
  const uint32_t tDQ = tmem + C::TM_DP + ((uint32_t)(wq * 32) << 16);  // dQ_i lies over dP^T
  uint8_t* box_base = smem + C::OFF_STAGE + wq * 4096;
  uint8_t* stage_row = box_base + lane * 128;
  for (int i = 0; i < u.steps; ++i) {
    if (!bwd_warp_wait(&sb.dq_full, i & 1, p.status)) break;
    tc_fence_after();
    uint32_t r[D];
#pragma unroll
    for (int c = 0; c < D; c += 32) tmem_ld_x32(tDQ + c, r + c);
    tmem_ld_wait32(r);
#pragma unroll
    for (int c = 32; c < D; c += 32) fence_regs32(r + c);
    tc_fence_before();
    mbar_arrive(&sb.dq_empty);
    const int h = u.head(i), q0 = u.q0(i);
#pragma unroll
    for (int c = 0; c < D; c += 32) {
      if (lane == 0) bulk_wait_read_all();  // the warp's previous box has left shared memory
      __syncwarp();
#pragma unroll
      for (int un = 0; un < 8; ++un)
        *reinterpret_cast<uint4*>(stage_row + ((un ^ (lane & 7)) << 4)) =
            make_uint4(r[c + 4 * un], r[c + 4 * un + 1], r[c + 4 * un + 2], r[c + 4 * un + 3]);
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        tma_reduce_add_3d(tmDQ, box_base, c, q0 + 32 * wq, u.b * p.Hq + h);
        bulk_commit_group();
      }
    }
  }
  if (lane == 0) bulk_wait_all();
}

// Logical grid: x = key block, y = key/value head, z = batch (bwd_cta_coords).
template <int D, bool BF16>
__global__ void __launch_bounds__(512, 1)
    attn_bwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDO,
                    const __grid_constant__ CUtensorMap tmDQ, const BwdParams p) {
  using C = BwdCfg<D>;
  __shared__ BwdBarriers sb;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

  BwdUnit u;
  const int3 cta = bwd_cta_coords(p);
  u.kb0 = cta.x * C::BN;
  u.hk = cta.y;
  u.b = cta.z;
  u.h0 = u.hk * p.group;
  {
    // Query rows that can read one of the keys kb0 .. kb0 + 127 (clipped to Nk).
    const int64_t delta = (int64_t)p.Nk - p.Nq;
    const int64_t klast = min(u.kb0 + C::BN - 1, p.Nk - 1);  // >= kb0: the grid covers Nk
    int64_t qlo = (int64_t)u.kb0 - delta - p.win_right, qhi = klast - delta + p.win_left;
    if (qlo < 0) qlo = 0;
    if (qhi > p.Nq - 1) qhi = p.Nq - 1;
    u.qb_lo = (int)(qlo / C::BM);
    u.n_qb = qhi >= qlo ? (int)(qhi / C::BM) - u.qb_lo + 1 : 0;
    u.steps = u.n_qb * p.group;
  }
  const int warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) {
    mbar_init(&sb.kv_full, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&sb.q_full[s], 1);
      mbar_init(&sb.q_empty[s], 1);
      mbar_init(&sb.do_full[s], 1);
      mbar_init(&sb.do_empty[s], 1);
    }
    mbar_init(&sb.dv_done, 1);
    mbar_init(&sb.s_full, 1);
    mbar_init(&sb.dp_full, 1);
    mbar_init(&sb.p_ready, 256);
    mbar_init(&sb.ds_ready, 256);
    mbar_init(&sb.p_read, 256);
    mbar_init(&sb.dq_full, 1);
    mbar_init(&sb.dq_empty, 128);
    mbar_init(&sb.kv_done, 1);
    mbar_init(&sb.fin, 1);
    fence_mbar_init();
  }
  if (warp == C::PRODUCER_WARP && (threadIdx.x & 31) == 0) {
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
    tma_prefetch_desc(&tmDO);
    tma_prefetch_desc(&tmDQ);
  }
  if (warp == C::MMA_WARP) {
    tmem_alloc(&sb.tmem_base, C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sb.tmem_base;

  if (warp < 8) {
    bwd_compute<D, BF16>(sb, smem, tmem, u, p, warp >> 2);
  } else if (warp < 12) {
    regs_grow<C::DQ_REGS>();
    bwd_dq<D>(sb, smem, tmem, u, p, &tmDQ);
  } else {
    regs_shrink<C::CTRL_REGS>();
    if (u.steps > 0) {
      const bool lane0 = (threadIdx.x & 31) == 0;
      if (warp == C::PRODUCER_WARP) {
        if (lane0) {
          int q_issued = 0, do_issued = 0;
          bwd_producer<D>(&tmQ, &tmK, &tmV, &tmDO, sb, smem, u, p, q_issued, do_issued);
          bwd_producer_settle<D>(sb, q_issued, do_issued);
        }
        __syncwarp();
      } else if (warp == C::MMA_WARP) {
        if (lane0) {
          bwd_mma<D>(sb, smem, tmem, u, BF16 ? 1u : 0u, p.status);
          // Every MMA issued has completed before tensor memory is released
          // (immediate after a normal run; bounded after a wait ran out).
          mma_commit(&sb.fin);
          mbar_wait(&sb.fin, 0, nullptr);
        }
        __syncwarp();
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == C::MMA_WARP) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

}  // namespace etattn

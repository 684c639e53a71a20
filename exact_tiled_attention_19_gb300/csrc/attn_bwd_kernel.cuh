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
// atomics (a later launch converts it to the input type).
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
// Roles (384 threads):
//   warps 0-3   thread t owns key row t: P^T from S^T, dS^T from dP^T (into
//               tensor memory and, transposed, into shared memory for dQ);
//               the dK / dV epilogue.
//   warps 4-7   thread t owns query row t of dQ_i: reads it from tensor memory
//               and adds it to the FP32 dQ buffer.
//   warp 8      TMA: K and V once; per step Q (two stages) with its lse and
//               dO (one stage) with its D (two stages).
//   warp 9      tensor-memory allocation and MMA issue (one thread).
//
// Tensor memory (512 columns): dK [0, D), dV [128, 128 + D), S^T / P^T / dQ
// [256, 384), dP^T / dS^T [384, 512).
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
  float* dq_acc;                 // FP32 [B, Hq, Nq, D], zeroed before the launch
  const float* lse2;             // [B * Hq][Nq_pad]: lse * log2(e); +inf where a row reads no key
  const float* dvec;             // [B * Hq][Nq_pad]: D = <dO, O>; 0 on padding rows
  int Nq, Nk, Nq_pad;            // Nq_pad: Nq rounded up to 128
  int Hq, group;
  int win_left, win_right;       // as in the forward pass (causal: win_right = 0)
  float scale, scale_log2;
  int* status;
  int hn_swapped;                // bit 0/1/2/3: the q/k/v/dO tensor map orders (d, head, token, batch)
};

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
  static constexpr int OFF_DO = 4 * TILE;              // one stage
  static constexpr int OFF_DS = 5 * TILE;              // dS, 128 queries x 128 keys, MN-major, 128B swizzle
  static constexpr int DS_BYTES = 128 * 128 * 2;
  static constexpr int OFF_LSE = OFF_DS + DS_BYTES;    // two stages of 128 floats
  // D of a step is read until the dS of the step is written, after the dO
  // stage has been released: two stages, by step parity.
  static constexpr int OFF_DVEC = OFF_LSE + 2 * 512;
  static constexpr int SMEM_BYTES = OFF_DVEC + 2 * 512 + 1024;
  static constexpr uint32_t SBO = 8 * SW_BYTES;
  static constexpr uint32_t TM_DK = 0, TM_DV = 128, TM_S = 256, TM_DP = 384, TMEM_COLS = 512;
  static constexpr int THREADS = 384;
  static constexpr int PRODUCER_WARP = 8, MMA_WARP = 9;
};

struct BwdBarriers {
  uint64_t kv_full;
  uint64_t q_full[2], q_empty[2];
  uint64_t do_full, do_empty;
  uint64_t s_full, dp_full;      // S^T / dP^T of the step are in tensor memory
  uint64_t p_ready, ds_ready;    // P^T / dS^T (and dS in shared memory) written (128 arrivals)
  uint64_t dq_full;              // dQ_i in tensor memory (the step's dK and dQ products are done)
  uint64_t dq_empty;             // dQ_i read out (128 arrivals)
  uint64_t kv_done;              // last dK / dV product done
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
                                             const BwdUnit u, const BwdParams& p) {
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
    bulk_load(smem + C::OFF_LSE + slot * 512, p.lse2 + vec_row, 512, &sb.q_full[slot]);
    if (i >= 1 && !mbar_wait(&sb.do_empty, (i - 1) & 1, p.status)) return;
    mbar_arrive_expect_tx(&sb.do_full, C::TILE + 512);
#pragma unroll
    for (int c = 0; c < C::NCHUNK; ++c)
      tma_tile(smem + C::OFF_DO + c * 128 * C::SW_BYTES, tmDO, &sb.do_full, c * C::SW_ELEMS, q0, h, u.b, swd);
    bulk_load(smem + C::OFF_DVEC + slot * 512, p.dvec + vec_row, 512, &sb.do_full);
  }
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
  const uint64_t ds_mn = smem_desc(smem_u32(smem + C::OFF_DS), 128 * 128, 1024, kSw128);
  const uint64_t slot_step = (uint64_t)(C::TILE >> 4);
  const uint32_t tDK = tmem + C::TM_DK, tDV = tmem + C::TM_DV, tS = tmem + C::TM_S, tDP = tmem + C::TM_DP;

  if (!mbar_wait(&sb.kv_full, 0, status)) return;
  for (int i = 0; i < u.steps; ++i) {
    const int slot = i & 1;
    const uint64_t q_k = q_kmaj + slot * slot_step, q_m = q_mn + slot * slot_step;
    if (!mbar_wait(&sb.q_full[slot], (i >> 1) & 1, status)) return;
    if (i > 0 && !mbar_wait(&sb.dq_empty, (i - 1) & 1, status)) return;
    tc_fence_after();
    // S^T = K Q^T over d in 16-element steps.
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      const uint64_t off = (uint64_t)(((kk / C::KSTEPS_PER_CHUNK) * 128 * C::SW_BYTES + (kk % C::KSTEPS_PER_CHUNK) * 32) >> 4);
      mma_ss(tS, k_kmaj + off, q_k + off, id_s, kk > 0 ? 1u : 0u);
    }
    mma_commit(&sb.s_full);
    if (!mbar_wait(&sb.do_full, i & 1, status)) return;
    tc_fence_after();
    // dP^T = V dO^T.
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      const uint64_t off = (uint64_t)(((kk / C::KSTEPS_PER_CHUNK) * 128 * C::SW_BYTES + (kk % C::KSTEPS_PER_CHUNK) * 32) >> 4);
      mma_ss(tDP, v_kmaj + off, do_kmaj + off, id_s, kk > 0 ? 1u : 0u);
    }
    mma_commit(&sb.dp_full);
    // dV += P^T dO over the step's 128 queries, 16 at a time (8 packed columns).
    if (!mbar_wait(&sb.p_ready, i & 1, status)) return;
    tc_fence_after();
#pragma unroll
    for (int kk = 0; kk < 8; ++kk)
      mma_ts(tDV, tS + kk * 8, do_mn + (uint64_t)((kk * 16 * C::SW_BYTES) >> 4), id_kv, (i > 0 || kk > 0) ? 1u : 0u);
    mma_commit(&sb.do_empty);
    // dK += dS^T Q, then dQ_i = dS K (over the 128 keys) into the S^T columns.
    if (!mbar_wait(&sb.ds_ready, i & 1, status)) return;
    tc_fence_after();
#pragma unroll
    for (int kk = 0; kk < 8; ++kk)
      mma_ts(tDK, tDP + kk * 8, q_m + (uint64_t)((kk * 16 * C::SW_BYTES) >> 4), id_kv, (i > 0 || kk > 0) ? 1u : 0u);
#pragma unroll
    for (int kk = 0; kk < 8; ++kk)
      mma_ss(tS, ds_mn + (uint64_t)((kk * 16 * 128) >> 4), k_mn + (uint64_t)((kk * 16 * C::SW_BYTES) >> 4), id_q,
             kk > 0 ? 1u : 0u);
    mma_commit(&sb.dq_full);
    mma_commit(&sb.q_empty[slot]);
  }
  mma_commit(&sb.kv_done);
  // Drain the arrivals no other role consumes.
  for (int i = u.steps > 2 ? u.steps - 2 : 0; i < u.steps; ++i)
    if (!mbar_wait(&sb.q_empty[i & 1], (i >> 1) & 1, status)) return;
  if (u.steps > 0 && !mbar_wait(&sb.do_empty, (u.steps - 1) & 1, status)) return;
}

__device__ __forceinline__ bool bwd_warp_wait(uint64_t* bar, uint32_t parity, int* status) {
  bool ok = true;
  if ((threadIdx.x & 31) == 0) ok = mbar_wait(bar, parity, status);
  return __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
}

template <bool BF16>
__device__ __forceinline__ uint32_t bwd_pack(float lo, float hi) {
  return BF16 ? pack_bf16x2(lo, hi) : pack_f16x2(lo, hi);
}
template <bool BF16>
__device__ __forceinline__ float bwd_lo(uint32_t w) {
  return BF16 ? __uint_as_float(w << 16) : __half2float(__ushort_as_half((unsigned short)(w & 0xffffu)));
}
template <bool BF16>
__device__ __forceinline__ float bwd_hi(uint32_t w) {
  return BF16 ? __uint_as_float(w & 0xffff0000u) : __half2float(__ushort_as_half((unsigned short)(w >> 16)));
}

// Warps 0-3: thread t owns key kb0 + t.
template <int D, bool BF16>
__device__ __forceinline__ void bwd_compute(BwdBarriers& sb, uint8_t* smem, uint32_t tmem, const BwdUnit u,
                                            const BwdParams& p) {
  using C = BwdCfg<D>;
  constexpr uint32_t FULL = 0xffffffffu;
  const int t = threadIdx.x & 127;
  const uint32_t lane_off = (uint32_t)((threadIdx.x >> 5) * 32) << 16;
  const uint32_t tS = tmem + C::TM_S + lane_off, tDP = tmem + C::TM_DP + lane_off;
  const int key = u.kb0 + t;
  // Query rows that may read this key: c - win_left <= key <= c + win_right
  // with c = q + Nk - Nq, i.e. q in [key - delta - win_right, key - delta + win_left].
  const int64_t delta = (int64_t)p.Nk - p.Nq;
  int64_t qlo = (int64_t)key - delta - p.win_right, qhi = (int64_t)key - delta + p.win_left;
  if (qhi > p.Nq - 1) qhi = p.Nq - 1;
  if (qlo < 0) qlo = 0;
  if (key >= p.Nk) qhi = -1;  // padding key: no query reads it
  const float c2 = p.scale_log2;
  const float* lse_s = reinterpret_cast<const float*>(smem + C::OFF_LSE);
  const float* dvec_s = reinterpret_cast<const float*>(smem + C::OFF_DVEC);
  uint8_t* ds_row = smem + C::OFF_DS + t * 128;
  int* status = p.status;

  for (int i = 0; i < u.steps; ++i) {
    const int q0 = u.q0(i), slot = i & 1;
    const int64_t lo_rel = qlo - q0, hi_rel = qhi - q0;
    const int lim_lo = lo_rel < -1 ? -1 : (int)lo_rel, lim_hi = hi_rel > 128 ? 128 : (int)hi_rel;
    const bool warp_masked = __any_sync(FULL, lim_lo > 0 || lim_hi < 127);
    const float* lse = lse_s + slot * 128;
    const float* dvec = dvec_s + slot * 128;
    // ---- P^T = exp2(c2 * s - lse2): two 64-column halves, written over S^T.
    if (!bwd_warp_wait(&sb.s_full, i & 1, status)) return;
    tc_fence_after();
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      uint32_t sr[64];
      tmem_ld_x32(tS + half * 64, sr);
      tmem_ld_x32(tS + half * 64 + 32, sr + 32);
      tmem_ld_wait32(sr);
      fence_regs32(sr + 32);
      uint32_t pk[32];
#pragma unroll
      for (int j = 0; j < 64; j += 2) {
        const int c = half * 64 + j;
        float p0 = ex2_approx(fmaf(__uint_as_float(sr[j]), c2, -lse[c]));
        float p1 = ex2_approx(fmaf(__uint_as_float(sr[j + 1]), c2, -lse[c + 1]));
        if (warp_masked) {
          p0 = (c < lim_lo || c > lim_hi) ? 0.f : p0;
          p1 = (c + 1 < lim_lo || c + 1 > lim_hi) ? 0.f : p1;
        }
        pk[j / 2] = bwd_pack<BF16>(p0, p1);
      }
      tmem_st_x32(tS + half * 32, pk);
    }
    tmem_st_wait();
    tc_fence_before();
    mbar_arrive(&sb.p_ready);

    // ---- dS^T = scale * P (dP - D), over dP^T in tensor memory and, as dS,
    // into shared memory (row t = key t; 16-byte unit u of queries 8u..8u+7
    // of each 64-query half at unit u ^ (t mod 8): the 128-byte swizzle).
    if (!bwd_warp_wait(&sb.dp_full, i & 1, status)) return;
    if (i > 0 && !bwd_warp_wait(&sb.dq_full, (i - 1) & 1, status)) return;  // dQ_{i-1} has read dS
    tc_fence_after();
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      uint32_t dr[64], pk[32];
      tmem_ld_x32(tDP + half * 64, dr);
      tmem_ld_x32(tDP + half * 64 + 32, dr + 32);
      tmem_ld_x32(tS + half * 32, pk);
      tmem_ld_wait32(dr);
      fence_regs32(dr + 32);
      fence_regs32(pk);
      uint32_t ds[32];
#pragma unroll
      for (int j = 0; j < 64; j += 2) {
        const int c = half * 64 + j;
        const float d0 = bwd_lo<BF16>(pk[j / 2]) * (__uint_as_float(dr[j]) - dvec[c]) * p.scale;
        const float d1 = bwd_hi<BF16>(pk[j / 2]) * (__uint_as_float(dr[j + 1]) - dvec[c + 1]) * p.scale;
        ds[j / 2] = bwd_pack<BF16>(d0, d1);
      }
      tmem_st_x32(tDP + half * 32, ds);
      uint8_t* chunk = ds_row + half * (128 * 128);
#pragma unroll
      for (int un = 0; un < 8; ++un)
        *reinterpret_cast<uint4*>(chunk + ((un ^ (t & 7)) << 4)) =
            make_uint4(ds[4 * un], ds[4 * un + 1], ds[4 * un + 2], ds[4 * un + 3]);
    }
    fence_proxy_async_smem();
    tmem_st_wait();
    tc_fence_before();
    mbar_arrive(&sb.ds_ready);
  }

  // ---- Epilogue: dK and dV rows of this CTA's keys, in the input type.
  const bool valid = key < p.Nk;
  uint8_t* dk_row = reinterpret_cast<uint8_t*>(p.dk) +
                    2 * ((int64_t)u.b * p.dk_sb + (int64_t)u.hk * p.dk_sh + (int64_t)key * p.dk_sn);
  uint8_t* dv_row = reinterpret_cast<uint8_t*>(p.dv) +
                    2 * ((int64_t)u.b * p.dv_sb + (int64_t)u.hk * p.dv_sh + (int64_t)key * p.dv_sn);
  if (u.steps == 0) {  // no query reads these keys
    if (valid) {
#pragma unroll
      for (int c = 0; c < D; c += 8) {
        *reinterpret_cast<uint4*>(dk_row + 2 * c) = make_uint4(0u, 0u, 0u, 0u);
        *reinterpret_cast<uint4*>(dv_row + 2 * c) = make_uint4(0u, 0u, 0u, 0u);
      }
    }
    return;
  }
  if (!bwd_warp_wait(&sb.kv_done, 0, status)) return;
  tc_fence_after();
#pragma unroll
  for (int which = 0; which < 2; ++which) {
    const uint32_t tsrc = tmem + (which ? C::TM_DV : C::TM_DK) + lane_off;
    uint8_t* row = which ? dv_row : dk_row;
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
}

// Warps 4-7: thread t owns query row q0 + t of each step's dQ contribution.
template <int D>
__device__ __forceinline__ void bwd_dq(BwdBarriers& sb, uint32_t tmem, const BwdUnit u, const BwdParams& p) {
  using C = BwdCfg<D>;
  const int t = threadIdx.x & 127;
  const uint32_t tS = tmem + C::TM_S + ((uint32_t)(((threadIdx.x >> 5) & 3) * 32) << 16);
  for (int i = 0; i < u.steps; ++i) {
    if (!bwd_warp_wait(&sb.dq_full, i & 1, p.status)) return;
    tc_fence_after();
    uint32_t r[D];
#pragma unroll
    for (int c = 0; c < D; c += 32) tmem_ld_x32(tS + c, r + c);
    tmem_ld_wait32(r);
#pragma unroll
    for (int c = 32; c < D; c += 32) fence_regs32(r + c);
    tc_fence_before();
    mbar_arrive(&sb.dq_empty);
    const int q = u.q0(i) + t;
    if (q < p.Nq) {
      float4* dst = reinterpret_cast<float4*>(p.dq_acc + (((int64_t)u.b * p.Hq + u.head(i)) * p.Nq + q) * D);
#pragma unroll
      for (int c = 0; c < D / 4; ++c)
        atomicAdd(dst + c, make_float4(__uint_as_float(r[4 * c]), __uint_as_float(r[4 * c + 1]),
                                       __uint_as_float(r[4 * c + 2]), __uint_as_float(r[4 * c + 3])));
    }
  }
}

// Grid: x = key block, y = key/value head, z = batch.
template <int D, bool BF16>
__global__ void __launch_bounds__(384, 1)
    attn_bwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDO,
                    const BwdParams p) {
  using C = BwdCfg<D>;
  __shared__ BwdBarriers sb;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

  BwdUnit u;
  u.kb0 = blockIdx.x * C::BN;
  u.hk = blockIdx.y;
  u.b = blockIdx.z;
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
    }
    mbar_init(&sb.do_full, 1);
    mbar_init(&sb.do_empty, 1);
    mbar_init(&sb.s_full, 1);
    mbar_init(&sb.dp_full, 1);
    mbar_init(&sb.p_ready, 128);
    mbar_init(&sb.ds_ready, 128);
    mbar_init(&sb.dq_full, 1);
    mbar_init(&sb.dq_empty, 128);
    mbar_init(&sb.kv_done, 1);
    fence_mbar_init();
  }
  if (warp == C::PRODUCER_WARP && (threadIdx.x & 31) == 0) {
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
    tma_prefetch_desc(&tmDO);
  }
  if (warp == C::MMA_WARP) {
    tmem_alloc(&sb.tmem_base, C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sb.tmem_base;

  if (warp < 4) {
    bwd_compute<D, BF16>(sb, smem, tmem, u, p);
  } else if (warp < 8) {
    bwd_dq<D>(sb, tmem, u, p);
  } else if (u.steps > 0) {
    const bool lane0 = (threadIdx.x & 31) == 0;
    if (warp == C::PRODUCER_WARP) {
      if (lane0) bwd_producer<D>(&tmQ, &tmK, &tmV, &tmDO, sb, smem, u, p);
      __syncwarp();
    } else if (warp == C::MMA_WARP) {
      if (lane0) bwd_mma<D>(sb, smem, tmem, u, BF16 ? 1u : 0u, p.status);
      __syncwarp();
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

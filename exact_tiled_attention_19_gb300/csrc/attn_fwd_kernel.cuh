// Exact streaming attention forward for sm_103a: TMA-staged Q/K/V tiles,
// tcgen05 MMAs accumulating in tensor memory, warp-specialised roles, and two
// 128-row query sub-tiles per CTA that take turns on the tensor core.
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
// A CTA owns 256 query rows as two sub-tiles (rows [0,128) and [128,256) of
// the block).  Both read the same K/V tiles from shared memory.
//
// Roles (384 threads = 3 warpgroups):
//   warpgroup 0 (warps 0-3)  softmax + correction + epilogue of sub-tile 0:
//                            thread t owns row t (tensor-memory lane t).
//   warpgroup 1 (warps 4-7)  the same for sub-tile 1.
//   warp 8                   TMA producer: Q0, Q1 once, then K_j into a
//                            three-stage ring and V_j into a two-stage ring.
//   warp 9                   tensor-memory allocator and MMA issuer.
//   warps 10-11              no work (they complete warpgroup 2).
//
// Tensor memory (512 columns x 128 lanes, FP32 cells):
//   S_s  = columns [128 s, 128 s + 128)         score tile of sub-tile s
//   P_s  = columns [128 s, 128 s + 64)          P overwrites its own S (two 16-bit values per cell)
//   O_s  = columns [256 + 128 s, 256 + 128 s + D)
//
// MMA issue order per key tile j >= 1:
//   PV_0(j-1), S_0(j), PV_1(j-1), S_1(j)
// so the softmax of one sub-tile overlaps two MMA groups of the other, and a
// commit on S_s(j) also covers PV_s(j-1) (a commit tracks every earlier
// tcgen05 operation of the issuing thread): when the softmax of sub-tile s
// sees S_s(j), O_s is up to date and may be rescaled.  S_s(j+1) overwrites
// P_s(j) only after PV_s(j), which was issued before it by the same thread.
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

template <int D, int NSUB_>
struct TileCfg {
  static constexpr int NSUB = NSUB_;                   // 128-row query sub-tiles per CTA (1 or 2)
  static constexpr int BM = 128;                       // query rows per sub-tile
  static constexpr int BLOCK_M = NSUB * BM;            // query rows per CTA
  static constexpr int BN = 128;                       // keys per tile
  static constexpr int SW_ELEMS = D >= 64 ? 64 : 32;   // elements per swizzled smem row
  static constexpr int SW_BYTES = SW_ELEMS * 2;        // 128 B (D >= 64) or 64 B (D = 32)
  static constexpr uint32_t SWIZZLE = D >= 64 ? kSw128 : kSw64;
  static constexpr int NCHUNK = D / SW_ELEMS;          // TMA boxes per tile along d
  static constexpr int KSTEPS_PER_CHUNK = SW_ELEMS / 16;
  static constexpr int Q_BYTES = BM * D * 2;           // one sub-tile
  static constexpr int KV_BYTES = BN * D * 2;
  static constexpr int K_STAGES = 3;
  static constexpr int V_STAGES = 2;
  static constexpr int OFF_Q = 0;                      // Q_0 (then Q_1)
  static constexpr int OFF_K = NSUB * Q_BYTES;
  static constexpr int OFF_V = OFF_K + K_STAGES * KV_BYTES;
  static constexpr int SMEM_BYTES = OFF_V + V_STAGES * KV_BYTES + 1024;  // + alignment slack
  static constexpr uint32_t SBO = 8 * SW_BYTES;        // stride between 8-row swizzle atoms
  static constexpr uint32_t TM_S = 0, TM_O = NSUB * 128;  // + 128 per sub-tile
  static constexpr uint32_t TMEM_COLS = NSUB * 256;
  // Warps: 4 softmax warps per sub-tile, then the TMA warp and the MMA warp,
  // padded to whole warpgroups.
  static constexpr int PRODUCER_WARP = 4 * NSUB, MMA_WARP = 4 * NSUB + 1;
  static constexpr int THREADS = NSUB == 2 ? 384 : 256;
  // Register split: 384 threads launch with LAUNCH_REGS each; warpgroup 2
  // (TMA + MMA) shrinks to CTRL_REGS so that the two softmax warpgroups can
  // grow to SOFTMAX_REGS.  128*CTRL_REGS + 256*SOFTMAX_REGS == 384*LAUNCH_REGS.
  static constexpr int LAUNCH_REGS = 168;
  static constexpr int CTRL_REGS = 88;
  static constexpr int SOFTMAX_REGS = 208;
  static_assert(NSUB == 1 || 128 * CTRL_REGS + 256 * SOFTMAX_REGS <= THREADS * LAUNCH_REGS,
                "register split over budget");
};

__device__ __forceinline__ void fence_regs32(uint32_t* r) {
  asm volatile("" : ETATTN_RW8(r, 0), ETATTN_RW8(r, 8), ETATTN_RW8(r, 16), ETATTN_RW8(r, 24));
}

struct SmemBarriers {
  uint64_t q_full;
  uint64_t k_full[3], k_empty[3];
  uint64_t v_full[2], v_empty[2];
  uint64_t s_full[2];            // per sub-tile: S_s(j) is in tensor memory (and PV_s(j-1) is done)
  uint64_t p_full[2];            // per sub-tile: P_s(j) written and O_s corrected
  uint64_t o_done[2];            // per sub-tile: last PV_s has completed
  uint32_t tmem_base;
};

// Per-CTA work description shared by all roles.
struct Unit {
  int h, hk, b, bcoord;          // query head, kv head, batch/sequence index, batch coordinate of the maps
  int tok0;                      // first token of the sequence (packed batch), else 0
  int L;                         // sequence length
  int row0;                      // first query row (logical position) of sub-tile 0
  int n0, n1;                    // key tiles visited by sub-tile 0 / 1 (0 = sub-tile idle)
  __device__ __forceinline__ int n(int s) const { return s ? n1 : n0; }
  int n_max;
};

// ----------------------------------------------------------------- producer
// Runs on one thread.  (Waits are single-thread too: 32 lanes polling one
// mbarrier serialise on it and cost more than a tile's MMA issue slot.)
template <int D, int NSUB>
__device__ __forceinline__ void producer_role(const CUtensorMap* tmQ, const CUtensorMap* tmK,
                                              const CUtensorMap* tmV, SmemBarriers& sb, uint8_t* smem,
                                              const Unit u, int hn_swapped, int* status) {
  using C = TileCfg<D, NSUB>;
  const bool swq = hn_swapped & 1, swk = (hn_swapped >> 1) & 1, swv = (hn_swapped >> 2) & 1;
  {
    mbar_arrive_expect_tx(&sb.q_full, NSUB * C::Q_BYTES);
#pragma unroll
    for (int s = 0; s < NSUB; ++s)
#pragma unroll
      for (int c = 0; c < C::NCHUNK; ++c)
        tma_load_tile(smem + C::OFF_Q + s * C::Q_BYTES + c * C::BM * C::SW_BYTES, tmQ, &sb.q_full,
                      c * C::SW_ELEMS, u.tok0 + u.row0 + s * C::BM, u.h, u.bcoord, swq);
  }
  int ks = 0, kph = 0;  // K ring slot and its phase for tile j
  for (int j = 0; j < u.n_max; ++j) {
    // K_j goes to slot j % 3, whose previous tile j-3 must have been released.
    if (j >= C::K_STAGES && !mbar_wait(&sb.k_empty[ks], kph ^ 1, status)) return;
    {
      mbar_arrive_expect_tx(&sb.k_full[ks], C::KV_BYTES);
#pragma unroll
      for (int c = 0; c < C::NCHUNK; ++c)
        tma_load_tile(smem + C::OFF_K + ks * C::KV_BYTES + c * C::BN * C::SW_BYTES, tmK, &sb.k_full[ks],
                      c * C::SW_ELEMS, u.tok0 + j * C::BN, u.hk, u.bcoord, swk);
    }
    if (++ks == C::K_STAGES) {
      ks = 0;
      kph ^= 1;
    }
    const int vs = j & 1;
    if (j >= 2 && !mbar_wait(&sb.v_empty[vs], ((j - 2) >> 1) & 1, status)) return;
    {
      mbar_arrive_expect_tx(&sb.v_full[vs], C::KV_BYTES);
#pragma unroll
      for (int c = 0; c < C::NCHUNK; ++c)
        tma_load_tile(smem + C::OFF_V + vs * C::KV_BYTES + c * C::BN * C::SW_BYTES, tmV, &sb.v_full[vs],
                      c * C::SW_ELEMS, u.tok0 + j * C::BN, u.hk, u.bcoord, swv);
    }
  }
}

// ----------------------------------------------------------------- MMA issuer
// Descriptors are built once per CTA; every k-step then adds a compile-time
// offset (in 16-byte units) to the 64-bit descriptor.  The 14-bit address
// field cannot overflow: shared memory addresses stay below 2^18 bytes.
// Keeping the issuing thread's work per MMA to an add and the instruction
// itself is what lets the tensor core run at full rate (a descriptor rebuilt
// per MMA costs more cycles than a 128x128x16 MMA takes).
struct MmaDescs {
  uint64_t q0, q1;      // Q_s, K-major
  uint64_t k0, k1, k2;  // K slots, K-major
  uint64_t v0, v1;      // V slots, MN-major
};

// S_s = Q_s K^T: both K-major (d contiguous); a 16-element step moves 32 bytes
// inside a swizzled row, and a new d-chunk starts a new TMA box.
template <int D, int NSUB>
__device__ __forceinline__ void issue_s(const MmaDescs& md, uint32_t tmem, int s, int ks, uint32_t idesc) {
  using C = TileCfg<D, NSUB>;
  const uint64_t qd = s ? md.q1 : md.q0;
  const uint64_t kd = ks == 0 ? md.k0 : (ks == 1 ? md.k1 : md.k2);
  const uint32_t d_tmem = tmem + C::TM_S + s * 128;
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    const int c = kk / C::KSTEPS_PER_CHUNK, w = kk % C::KSTEPS_PER_CHUNK;
    const uint64_t qoff = (uint64_t)((c * C::BM * C::SW_BYTES + w * 32) >> 4);
    const uint64_t koff = (uint64_t)((c * C::BN * C::SW_BYTES + w * 32) >> 4);
    mma_ss(d_tmem, qd + qoff, kd + koff, idesc, kk > 0 ? 1u : 0u);
  }
}

// O_s (+)= P_s V: A = P_s from tensor memory (8 cells = 16 keys per step),
// B = V MN-major (d contiguous): 16 keys = 16 swizzled rows per step; LBO
// steps between d-chunks, SBO between 8-row groups.
template <int D, int NSUB>
__device__ __forceinline__ void issue_pv(const MmaDescs& md, uint32_t tmem, int s, int st, bool accumulate,
                                         uint32_t idesc) {
  using C = TileCfg<D, NSUB>;
  const uint64_t vd = st ? md.v1 : md.v0;
  const uint32_t p_base = tmem + C::TM_S + s * 128;
  const uint32_t d_tmem = tmem + C::TM_O + s * 128;
  const uint32_t acc0 = accumulate ? 1u : 0u;
#pragma unroll
  for (int kk = 0; kk < C::BN / 16; ++kk)
    mma_ts(d_tmem, p_base + kk * 8, vd + (uint64_t)((kk * 16 * C::SW_BYTES) >> 4), idesc, kk > 0 ? 1u : acc0);
}

// Runs on one thread: the tensor pipe queues only a couple of MMAs, so any
// cycle the issuing thread spends elsewhere between groups is idle tensor time.
template <int D, int NSUB>
__device__ __forceinline__ void mma_role(SmemBarriers& sb, uint8_t* smem, uint32_t tmem, const Unit u,
                                         uint32_t idesc_s, uint32_t idesc_pv, int* status) {
  using C = TileCfg<D, NSUB>;
  MmaDescs md;
  md.q0 = smem_desc(smem_u32(smem + C::OFF_Q), 16, C::SBO, C::SWIZZLE);
  md.q1 = md.q0 + (uint64_t)(C::Q_BYTES >> 4);
  md.k0 = smem_desc(smem_u32(smem + C::OFF_K), 16, C::SBO, C::SWIZZLE);
  md.k1 = md.k0 + (uint64_t)(C::KV_BYTES >> 4);
  md.k2 = md.k1 + (uint64_t)(C::KV_BYTES >> 4);
  md.v0 = smem_desc(smem_u32(smem + C::OFF_V), C::BN * C::SW_BYTES, C::SBO, C::SWIZZLE);
  md.v1 = md.v0 + (uint64_t)(C::KV_BYTES >> 4);
  if (!mbar_wait(&sb.q_full, 0, status)) return;

  int ks = 0, kph = 0;  // K ring slot / phase of the next key tile
  if (!mbar_wait(&sb.k_full[0], 0, status)) return;
  tc_fence_after();
#pragma unroll
  for (int sub = 0; sub < 2; ++sub) {
    if (u.n(sub) > 0) {
      issue_s<D, NSUB>(md, tmem, sub, 0, idesc_s);
      mma_commit(&sb.s_full[sub]);
    }
  }
  mma_commit(&sb.k_empty[0]);
  ks = 1;
  for (int j = 1; j <= u.n_max; ++j) {
    const int i = j - 1;  // key tile whose PV products are issued in this step
    const bool has_k = j < u.n_max;
    if (has_k && !mbar_wait(&sb.k_full[ks], kph, status)) return;
#pragma unroll
    for (int sub = 0; sub < 2; ++sub) {
      if (i < u.n(sub)) {  // PV_sub(i)
        if (!mbar_wait(&sb.v_full[i & 1], (i >> 1) & 1, status) || !mbar_wait(&sb.p_full[sub], i & 1, status)) return;
        tc_fence_after();
        issue_pv<D, NSUB>(md, tmem, sub, i & 1, i > 0, idesc_pv);
        if (i == u.n(sub) - 1) mma_commit(&sb.o_done[sub]);
      }
      if (sub == 1) mma_commit(&sb.v_empty[i & 1]);  // every PV product of tile i is issued
      if (j < u.n(sub)) {  // S_sub(j)
        issue_s<D, NSUB>(md, tmem, sub, ks, idesc_s);
        mma_commit(&sb.s_full[sub]);
      }
    }
    if (has_k) {
      mma_commit(&sb.k_empty[ks]);
      if (++ks == C::K_STAGES) {
        ks = 0;
        kph ^= 1;
      }
    }
  }
  // Drain: wait for the commit arrivals nobody else consumes (the last
  // tiles' ring releases and the final PV of each sub-tile) so that no
  // arrival can land in shared memory after the CTA exits.
  for (int t = u.n_max > C::K_STAGES ? u.n_max - C::K_STAGES : 0; t < u.n_max; ++t)
    if (!mbar_wait(&sb.k_empty[t % C::K_STAGES], (t / C::K_STAGES) & 1, status)) return;
  for (int t = u.n_max >= 2 ? u.n_max - 2 : 0; t < u.n_max; ++t)
    if (!mbar_wait(&sb.v_empty[t & 1], (t >> 1) & 1, status)) return;
#pragma unroll
  for (int sub = 0; sub < 2; ++sub)
    if (u.n(sub) > 0 && !mbar_wait(&sb.o_done[sub], 0, status)) return;
}

// ----------------------------------------------------------------- softmax / correction / epilogue
// Warp-wide wait: lane 0 polls the barrier and the outcome is broadcast, so
// one thread per warp (not 32) touches the barrier word.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, int* status) {
  bool ok = true;
  if ((threadIdx.x & 31) == 0) ok = mbar_wait(bar, parity, status);
  return __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
}

template <bool BF16>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  return BF16 ? pack_bf16x2(lo, hi) : pack_f16x2(lo, hi);
}

template <int D, int NSUB, bool BF16>
__device__ __forceinline__ void softmax_role(SmemBarriers& sb, uint32_t tmem, const FwdParams& p, const Unit u,
                                             int s) {
  using C = TileCfg<D, NSUB>;
  constexpr uint32_t FULL = 0xffffffffu;
  const int n = s ? u.n1 : u.n0;
  if (n == 0) return;
  const int t = threadIdx.x & 127;  // query row inside the sub-tile = tensor-memory lane
  const uint32_t lane_off = (uint32_t)(((threadIdx.x >> 5) & 3) * 32) << 16;
  const uint32_t tS = tmem + C::TM_S + s * 128 + lane_off;
  const uint32_t tO = tmem + C::TM_O + s * 128 + lane_off;
  const int row_pos = u.row0 + s * C::BM + t;  // logical position inside the sequence
  const float c2 = p.scale_log2;
  int* status = p.status;
  // Last eligible key position of this row: the diagonal under the causal
  // mask, and never past the end of the sequence.
  const int last_key = p.causal ? min(row_pos, u.L - 1) : u.L - 1;
  float m_run = -INFINITY;  // running maximum of the raw scores (scale > 0)
  float l_run = 0.f;        // sum of exp2(c2 * (s - m_run)) over the keys seen

  for (int j = 0; j < n; ++j) {
    if (!warp_wait(&sb.s_full[s], j & 1, status)) return;
    tc_fence_after();
    // Scores arrive in two halves: the maximum of the first half is taken
    // while the second half is still being read from tensor memory.
    uint32_t sr[C::BN];
    tmem_ld_x32(tS + 0, sr + 0);
    tmem_ld_x32(tS + 32, sr + 32);
    tmem_ld_wait32(sr);
    fence_regs32(sr + 32);
    tmem_ld_x32(tS + 64, sr + 64);
    tmem_ld_x32(tS + 96, sr + 96);

    float sv[C::BN];
    // Mask keys past the diagonal (causal) or past the sequence end.
    const int lim = last_key - j * C::BN;
    const bool masked = lim < C::BN - 1;
    // Only diagonal and tail tiles need masking; the test is warp-uniform so
    // that other tiles skip the per-element selects entirely.
    const bool warp_masked = __any_sync(FULL, masked);
#pragma unroll
    for (int i = 0; i < C::BN / 2; ++i) sv[i] = __uint_as_float(sr[i]);
    if (warp_masked) {
#pragma unroll
      for (int i = 0; i < C::BN / 2; ++i) sv[i] = i > lim ? -INFINITY : sv[i];
    }
    float mx0 = fmaxf(sv[0], sv[1]), mx1 = fmaxf(sv[2], sv[3]);
    float mx2 = fmaxf(sv[4], sv[5]), mx3 = fmaxf(sv[6], sv[7]);
#pragma unroll
    for (int i = 8; i < C::BN / 2; i += 8) {
      mx0 = max3(mx0, sv[i], sv[i + 1]);
      mx1 = max3(mx1, sv[i + 2], sv[i + 3]);
      mx2 = max3(mx2, sv[i + 4], sv[i + 5]);
      mx3 = max3(mx3, sv[i + 6], sv[i + 7]);
    }
    tmem_ld_wait32(sr + 64);
    fence_regs32(sr + 96);
#pragma unroll
    for (int i = C::BN / 2; i < C::BN; ++i) sv[i] = __uint_as_float(sr[i]);
    if (warp_masked) {
#pragma unroll
      for (int i = C::BN / 2; i < C::BN; ++i) sv[i] = i > lim ? -INFINITY : sv[i];
    }
#pragma unroll
    for (int i = C::BN / 2; i < C::BN; i += 8) {
      mx0 = max3(mx0, sv[i], sv[i + 1]);
      mx1 = max3(mx1, sv[i + 2], sv[i + 3]);
      mx2 = max3(mx2, sv[i + 4], sv[i + 5]);
      mx3 = max3(mx3, sv[i + 6], sv[i + 7]);
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
    // p = exp2(s * c2 - m * c2): the scaling runs two lanes per instruction,
    // the row sum in four independent pairs of accumulators.
    uint32_t pk[C::BN / 2];
    float ra0 = 0.f, ra1 = 0.f, rb0 = 0.f, rb1 = 0.f, rc0 = 0.f, rc1 = 0.f, rd0 = 0.f, rd1 = 0.f;
#pragma unroll
    for (int i = 0; i < C::BN / 2; i += 4) {
      float x[8];
#pragma unroll
      for (int k = 0; k < 4; ++k)
        fma2(x[2 * k], x[2 * k + 1], sv[2 * (i + k)], sv[2 * (i + k) + 1], c2, c2, neg_mc, neg_mc);
#pragma unroll
      for (int k = 0; k < 8; ++k) x[k] = ex2_approx(x[k]);
      add2(ra0, ra1, x[0], x[1]);
      add2(rb0, rb1, x[2], x[3]);
      add2(rc0, rc1, x[4], x[5]);
      add2(rd0, rd1, x[6], x[7]);
#pragma unroll
      for (int k = 0; k < 4; ++k) pk[i + k] = pack2<BF16>(x[2 * k], x[2 * k + 1]);
    }
    l_run = l_run * alpha + (((ra0 + rb0) + (rc0 + rd0)) + ((ra1 + rb1) + (rc1 + rd1)));

    // Correction: O_s *= alpha for rows whose maximum moved.  PV_s(j-1) has
    // completed: the commit that signalled S_s(j) covers it.
    if (j > 0 && __any_sync(FULL, rescale)) {
#pragma unroll
      for (int c = 0; c < D; c += 32) {
        uint32_t o[32];
        tmem_ld_x32(tO + c, o);
        tmem_ld_wait32(o);
#pragma unroll
        for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
        tmem_st_x32(tO + c, o);
      }
    }
    tmem_st_x32(tS, pk);  // P_s(j) over the first 64 cells of S_s(j)
    tmem_st_x32(tS + 32, pk + 32);
    tmem_st_wait();
    tc_fence_before();
    mbar_arrive(&sb.p_full[s]);
  }

  // Epilogue: O = O_acc / l in the input type, lse = scale * m + ln l.
  if (!warp_wait(&sb.o_done[s], 0, status)) return;
  tc_fence_after();
  const bool valid = row_pos < u.L;
  const float inv_l = 1.f / l_run;
  uint8_t* orow = reinterpret_cast<uint8_t*>(p.o) +
                  2 * ((int64_t)u.b * p.o_sb + (int64_t)u.h * p.o_sh + (int64_t)(u.tok0 + row_pos) * p.o_sn);
#pragma unroll
  for (int c = 0; c < D; c += 32) {
    uint32_t o[32];
    tmem_ld_x32(tO + c, o);
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
    p.lse[(int64_t)u.b * p.lse_sb + (int64_t)u.h * p.lse_sh + u.tok0 + row_pos] = m_run * p.scale + __logf(l_run);
}

// ----------------------------------------------------------------- kernel
// Grid: x = query block (NSUB * 128 rows) counted from the last one,
// y = query head, z = batch (or sequence).  CTAs are dispatched in that order,
// so the CTAs running at any time mostly belong to a few heads and share
// their K/V tiles in L2, and within a head the longest causal rows start
// first.  NSUB = 2 (two sub-tiles taking turns on the tensor core) is the
// throughput configuration; NSUB = 1 gives small problems twice as many CTAs.
template <int D, int NSUB, bool BF16>
__global__ void __launch_bounds__(TileCfg<D, NSUB>::THREADS, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const FwdParams p) {
  using C = TileCfg<D, NSUB>;
  __shared__ SmemBarriers sb;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

  Unit u;
  u.h = blockIdx.y;
  u.b = blockIdx.z;
  u.hk = u.h / p.group;
  u.L = p.N;
  u.tok0 = 0;
  u.bcoord = u.b;
  if (p.cu_seqlens != nullptr) {
    const int s0 = p.cu_seqlens[u.b], s1 = p.cu_seqlens[u.b + 1];
    if (s0 < 0 || s1 < s0 || s1 > p.total_tokens || s1 - s0 > p.max_seqlen) {
      if (threadIdx.x == 0) atomicCAS(p.status, 0, (int)kDevBadSeqlens);
      return;
    }
    u.L = s1 - s0;
    u.tok0 = s0;
    u.bcoord = 0;
  }
  const int block = (int)gridDim.x - 1 - (int)blockIdx.x;
  u.row0 = block * C::BLOCK_M;
  if (u.row0 >= u.L) return;  // uniform across the CTA
  const int n_all = (u.L + C::BN - 1) / C::BN;
  {
    const int first1 = u.row0 + C::BM;
    u.n0 = p.causal ? u.row0 / C::BN + 1 : n_all;  // row0 < L here
    u.n1 = (NSUB == 1 || first1 >= u.L) ? 0 : (p.causal ? first1 / C::BN + 1 : n_all);
  }
  u.n_max = max(u.n0, u.n1);
  const int warp = threadIdx.x >> 5;

  if (threadIdx.x == 0) {
    mbar_init(&sb.q_full, 1);
#pragma unroll
    for (int i = 0; i < C::K_STAGES; ++i) {
      mbar_init(&sb.k_full[i], 1);
      mbar_init(&sb.k_empty[i], 1);
    }
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sb.v_full[i], 1);
      mbar_init(&sb.v_empty[i], 1);
      mbar_init(&sb.s_full[i], 1);
      mbar_init(&sb.p_full[i], 128);
      mbar_init(&sb.o_done[i], 1);
    }
    fence_mbar_init();
  }
  if (warp == C::PRODUCER_WARP && (threadIdx.x & 31) == 0) {
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
  }
  if (warp == C::MMA_WARP) {
    tmem_alloc(&sb.tmem_base, C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sb.tmem_base;

  if (warp < 4 * NSUB) {
    if constexpr (NSUB == 2) regs_grow<C::SOFTMAX_REGS>();
    softmax_role<D, NSUB, BF16>(sb, tmem, p, u, warp >> 2);
  } else {
    if constexpr (NSUB == 2) regs_shrink<C::CTRL_REGS>();
    const bool lane0 = (threadIdx.x & 31) == 0;
    if (warp == C::PRODUCER_WARP) {
      if (lane0) producer_role<D, NSUB>(&tmQ, &tmK, &tmV, sb, smem, u, p.hn_swapped, p.status);
      __syncwarp();
    } else if (warp == C::MMA_WARP) {
      constexpr uint32_t ab = BF16 ? 1u : 0u;
      constexpr uint32_t idesc_s = instr_desc_f16(128, C::BN, ab, false, false);
      constexpr uint32_t idesc_pv = instr_desc_f16(128, D, ab, false, true);
      if (lane0) mma_role<D, NSUB>(sb, smem, tmem, u, idesc_s, idesc_pv, p.status);
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

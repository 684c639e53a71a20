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
// Query and key lengths may differ ("Attention algorithms and data
// movement", lesson 04): query row r of Lq sits at key position
// c = r + Lk - Lq (the last query aligns with the last key).  Row r may read
// keys lo <= j <= hi with hi = min(Lk - 1, c + win_right) and
// lo = max(0, c - win_left); causal attention is win_right = 0, a local
// window (same page, lesson 07) bounds win_left.  Each sub-tile streams only
// the key tiles some of its rows may read, and a row that may read none gets
// O = 0 and lse = -inf.
//
// Split-KV ("Intermediate and advanced extension", workshop row "Split
// softmax" and "Logic review before implementation"): with part_o set, the
// CTAs of one query block are spread over num_splits slices of the key tiles,
// and each writes its rows' partial state (O_s = acc_s / l_s in FP32 and
// lse_s = scale * m_s + ln l_s, or 0 and -inf for a slice with no eligible
// key) instead of O; a second launch on the same stream merges the slices.
//
// Grouped-query packing (general build): with qpack = P > 1, a 128-row
// sub-tile holds 128 / P query tokens of each of P query heads that share one
// key/value head ("Attention algorithms and data movement", lesson 05), so a
// few-query call (a decode step) streams each K/V tile once for the group and
// fills P times more of the tile.
//
// Key split (KS, for problems too small to fill the GPU): both sub-tiles
// hold the same 128 query rows and take alternate key tiles (even / odd), so
// the two softmax chains of a CTA take turns on the tensor core instead of
// running one after the other; at the end sub-tile 1 hands its (m, l) to
// sub-tile 0 through shared memory and its O through tensor memory, and
// sub-tile 0 merges the two states ("Attention algorithms and data
// movement", lesson 01: merging normalised partial states) and writes the
// rows.
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

// Key-window bound meaning "no bound": any offset >= the longest sequence
// acts the same, and c +/- kUnboundedWindow stays inside int32 for
// |c| < 2^30.
constexpr int kUnboundedWindow = (1 << 30) - 1;

struct FwdParams {
  void* o;
  float* lse;
  int64_t o_sb, o_sh, o_sn;      // element strides of o (batch/sequence, head, token); d-stride 1
  int64_t lse_sb, lse_sh;        // element strides of lse (batch, head); token stride 1
  const int* cu_seqlens_q;       // packed batch query offsets, or nullptr for the batched layout
  const int* cu_seqlens_k;       // packed batch key offsets (may equal cu_seqlens_q)
  int Nq, Nk;                    // batched: query / key tokens per sequence
  int total_q, total_k;          // packed batch: total query / key tokens
  int max_seqlen_q, max_seqlen_k;  // packed batch: bounds on every length
  int Hq, group;                 // query heads, Hq / Hkv
  int win_left, win_right;       // key j is eligible for a row at key position c iff
                                 // c - win_left <= j <= c + win_right (causal: win_right = 0)
  float* part_o;                 // split-KV partial outputs, or nullptr: FP32, D per row, row r of
                                 // slice s at (s * part_stride + r) * D, r the row's lse index
  float* part_lse;               // split-KV partial lse at s * part_stride + r
  int64_t part_stride;           // rows per slice (the size of lse)
  int num_splits, split_tiles;   // key-tile slices; key tiles per slice
  int qpack;                     // query heads per 128-row sub-tile (1, or a power of two dividing group)
  int num_global;                // global tokens (the global-token build), else 0
  int win_right_causal;          // 0 under the causal mask, else kUnboundedWindow: the bound a global
                                 // token's connections keep
  float scale;                   // logit scale
  float scale_log2;              // scale * log2(e)
  int* status;                   // device status word
  int hn_swapped;                // bit 0/1/2: the q/k/v tensor map orders (d, head, token, batch)
                                 // instead of (d, token, head, batch)
  int grid_x, grid_y, grid_z;    // the logical grid: x = query block (x key slices) counted from the last,
                                 // y = query head (pack), z = batch / sequence
  int sched_q, sched_rem;        // sched_q > 0: a 1-D launch of grid_x * grid_y * grid_z CTAs in grouped
                                 // longest-first order (cta_coords); the (y, z) pairs form groups of
                                 // sched_q + 1 pairs (the first sched_rem groups) and sched_q pairs.
                                 // sched_q = 0: the 3-D grid itself
  uint32_t div_m[4];             // exact reciprocals (DivMagic) of grid_x, sched_q + 1, sched_q, grid_y
  uint32_t div_k[4];
};

// Division of n < 2^31 by a divisor d >= 1 fixed at launch, as a multiply and
// a shift: with l = ceil(log2 d), k = 31 + l and m = ceil(2^k / d) (which fits
// in 32 bits), floor(n / d) = (n * m) >> k exactly.  Proof: n * m / 2^k =
// n / d + n * e / (d * 2^k) with e = m * d - 2^k in [0, d), and
// n * e < 2^31 * 2^l = 2^k, so the excess stays below 1 / d and cannot carry
// the quotient past the next integer.  The host computes (m, k).
__device__ __forceinline__ uint32_t div_magic(uint32_t n, uint32_t m, uint32_t k) {
  return (uint32_t)(((uint64_t)n * m) >> k);
}

// The logical (x, y, z) of this CTA.  The hardware starts CTAs in increasing
// linear index.  With sched_q > 0 the grid is launched 1-D and the (y, z)
// pairs (y fastest) are cut into contiguous groups of near-equal size; a
// group's CTAs come one after another, ordered by x (so the longest causal
// blocks of every pair of the group start first), then by pair.  The CTAs
// running at any time then read the K/V of one group of heads, which stays in
// L2, while the last CTAs to start are the shortest blocks of the last group
// instead of a whole head's longest block (the causal tail).  The map runs at
// every CTA's start, before any load is issued, so its divisions are
// multiply-shifts (div_magic) rather than the general integer division.
__device__ __forceinline__ int3 cta_coords(const FwdParams& p) {
  if (p.sched_q <= 0) return make_int3((int)blockIdx.x, (int)blockIdx.y, (int)blockIdx.z);
  const uint32_t lin = blockIdx.x, gx = (uint32_t)p.grid_x, gy = (uint32_t)p.grid_y;
  const uint32_t q = (uint32_t)p.sched_q, big = (uint32_t)p.sched_rem * (q + 1);  // pairs in the larger groups
  // Each pair contributes gx CTAs, so CTA lin lies in the group holding the
  // (lin / gx)-th pair.
  const uint32_t pi = div_magic(lin, p.div_m[0], p.div_k[0]);
  const bool large = pi < big;
  const uint32_t size = large ? q + 1 : q, dm = large ? p.div_m[1] : p.div_m[2], dk = large ? p.div_k[1] : p.div_k[2];
  const uint32_t first = large ? div_magic(pi, dm, dk) * size : big + div_magic(pi - big, dm, dk) * q;
  const uint32_t r = lin - first * gx;
  const uint32_t x = div_magic(r, dm, dk);
  const uint32_t pair = first + (r - x * size);
  const uint32_t z = div_magic(pair, p.div_m[3], p.div_k[3]);
  return make_int3((int)x, (int)(pair - z * gy), (int)z);
}

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
  // grow to SOFTMAX_REGS.  128*CTRL_REGS + 256*SOFTMAX_REGS <= 384*LAUNCH_REGS.
  static constexpr int LAUNCH_REGS = 168;
  static constexpr int CTRL_REGS = 88;
  static constexpr int SOFTMAX_REGS = 208;
  static_assert(NSUB == 1 || 128 * CTRL_REGS + 256 * SOFTMAX_REGS <= THREADS * LAUNCH_REGS,
                "register split over budget");
};

struct SmemBarriers {
  uint64_t q_full;
  uint64_t k_full[3], k_empty[3];
  uint64_t v_full[2], v_empty[2];
  uint64_t s_full[2];            // per sub-tile: S_s(j) is in tensor memory (and PV_s(j-1) is done)
  uint64_t p_full[2];            // per sub-tile: P_s(j) written and O_s corrected
  uint64_t p_half[2];            // per sub-tile: the first half of P_s(j) (keys 0-63) written, O_s corrected
  uint64_t o_done[2];            // per sub-tile: last PV_s has completed
  uint64_t merge_ready;          // key split: sub-tile 1's (m, l) and O are final (128 arrivals)
  uint64_t fin;                  // after a wait that ran out: every MMA issued so far has completed
  float merge_m[128], merge_l[128];  // key split: sub-tile 1's running max and sum per row
  uint32_t tmem_base;
  uint32_t split_mask;           // bit s: sub-tile s takes P as two 16-bit parts (split_mask())
};

// Per-CTA work description shared by all roles.  Key tiles are streamed in
// the order kt0, kt0 + 1, ..., kt0 + n_tot - 1; sub-tile s reads streamed
// tiles f_s .. f_s + n_s - 1 of them (the two ranges overlap or touch).
struct Unit {
  int h, hk, b, bcoord;          // (first) query head, kv head, batch/sequence index, batch coordinate of the maps
  int P, span;                   // query heads per sub-tile, query tokens per sub-tile (P * span = 128)
  int tok0q, tok0k;              // first query / key token of the sequence (packed batch), else 0
  int Lq, Lk;                    // query / key length of the sequence
  int delta;                     // Lk - Lq: query row r sits at key position r + delta
  int row0;                      // first query row (logical position) of sub-tile 0
  int kt0, n_tot;                // first key tile streamed, tiles streamed
  int f0, f1;                    // first streamed tile read by sub-tile 0 / 1
  int n0, n1;                    // tiles read by sub-tile 0 / 1 (0 = nothing to read)
  int split;                     // key-tile slice of a split-KV launch (else 0)
  int ng, wt0;                   // global-token build: streamed tiles of the global phase; key tile of
                                 // the first window-phase tile (streamed tile ng)
  int ga0, ga1;                  // global-token build: global-phase tiles read by sub-tile 0 / 1
  __device__ __forceinline__ int n(int s) const { return s ? n1 : n0; }
  __device__ __forceinline__ int ga(int s) const { return s ? ga1 : ga0; }
  __device__ __forceinline__ int f(int s) const { return s ? f1 : f0; }
  // Sub-tile s reads streamed tile j.
  __device__ __forceinline__ bool reads(int s, int j) const { return (unsigned)(j - f(s)) < (unsigned)n(s); }
};

// Keys [lo, hi] (none when lo > hi) the row at key position c reads.
// Without global tokens: its window.  With G global tokens ("Attention
// algorithms and data movement", lesson 07, global-token unions) a row reads
// the global keys and its window, both under the causal mask (limit h = c,
// or the last key), and a global row (c < G) reads every key up to h.  That
// is two disjoint key intervals, streamed as two phases: part 1, the global
// keys [0, min(G - 1, h)]; part 0, the rest: [G, h] for a global row and the
// window clipped below at G otherwise.  No key is counted in both.
__device__ __forceinline__ int2 row_key_range(int c, const Unit& u, const FwdParams& p, int part) {
  int lo = max(0, c - p.win_left), hi = min(u.Lk - 1, c + p.win_right);
  if (p.num_global > 0) {
    const int G = p.num_global, h = min(u.Lk - 1, c + p.win_right_causal);
    if (part == 1) {
      lo = 0;
      hi = min(G - 1, h);
    } else if (c < G) {
      lo = G;
      hi = h;
    } else {
      lo = max(lo, G);
    }
  }
  return make_int2(lo, hi);
}

// Key tiles [first, end) that some row of the query tokens [r0, r0 + span)
// (clipped to the sequence) may read; {0, 0} when none may read any key.
// A row's first key never decreases with its position; its last key does
// not either, except that a global row may end past the first non-global
// row's window: the first and last rows' ranges bound every row's.
__device__ __forceinline__ int2 sub_tile_key_tiles(int r0, int span, const Unit& u, const FwdParams& p, int bn,
                                                   int part = 0) {
  if (r0 >= u.Lq) return make_int2(0, 0);
  const int c_first = r0 + u.delta, c_last = min(r0 + span - 1, u.Lq - 1) + u.delta;
  const int2 a = row_key_range(c_first, u, p, part), b = row_key_range(c_last, u, p, part);
  const int lo = min(a.x, b.x), hi = max(a.y, b.y);
  if (hi < lo) return make_int2(0, 0);
  return make_int2(lo / bn, hi / bn + 1);
}

// Sub-tiles with a row that reads fewer than kFewKeys keys take P at about
// twice the input type's precision: P = P_hi + P_lo, both rounded to the input
// type (P_lo the rounding residual of P_hi), and O gains both products.  Such
// rows (the start of a causal sequence, a narrow window) hold few weights, so
// one 16-bit rounding of a large weight would move O by up to a relative half
// unit of the input type, on top of the output's own rounding; with many keys
// the roundings average out: at 128 keys and more, a CPU model of this
// kernel's arithmetic keeps every BF16 element of the batched, GQA and packed
// causal workloads within 0.0078 of the exact result, the output rounding
// itself.  Both ends of the sub-tile's valid rows bound the key counts in
// between (a row's first and last keys never decrease with its position,
// except for global rows, which read more keys).
constexpr int kFewKeys = 128;
__device__ __forceinline__ int few_keys(int r0, int span, const Unit& u, const FwdParams& p) {
  if (r0 >= u.Lq) return 0;
  int fewest = 1 << 30;
  for (int end = 0; end < 2; ++end) {
    const int c = (end ? min(r0 + span - 1, u.Lq - 1) : r0) + u.delta;
    const int2 a = row_key_range(c, u, p, 0);
    int cnt = max(0, a.y - a.x + 1);
    if (p.num_global > 0) {
      const int2 g = row_key_range(c, u, p, 1);
      cnt += max(0, g.y - g.x + 1);
    }
    fewest = min(fewest, cnt);
  }
  return fewest < kFewKeys ? 1 : 0;
}
// Bit s set: sub-tile s takes the split P (the key split's two sub-tiles
// hold the same rows).  One thread computes it at the CTA's set-up, after it
// has issued the first loads (ahead of them it delays every CTA's start), and
// the roles read it from shared memory.  A CTA with a split sub-tile runs the
// SPLIT instantiation of its softmax and MMA roles; every other CTA runs code
// without any trace of the second product.  The split code is only compiled
// into the kernel (template SPL) that the host launches when some row of the
// call may read fewer than kFewKeys keys, and only for BF16: FP16's 11-bit P
// keeps the error within the FP16 bound.
template <int NSUB, bool KS>
__device__ __forceinline__ uint32_t split_mask(const Unit& u, const FwdParams& p) {
  if (KS) return few_keys(u.row0, u.span, u, p) ? 3u : 0u;
  return (uint32_t)few_keys(u.row0, u.span, u, p) | (NSUB == 2 ? (uint32_t)few_keys(u.row0 + u.span, u.span, u, p) << 1 : 0u);
}

// ----------------------------------------------------------------- producer
// Runs on one thread.  (Waits are single-thread too: 32 lanes polling one
// mbarrier serialise on it and cost more than a tile's MMA issue slot.)
// Loads Q and key tiles j_from .. n_tot - 1 (with j_from = 0 the Q tiles
// too).  The first call, with j_to = 1, runs before the CTA's first barrier:
// the Q and first K / V tiles are then in flight while tensor memory is
// allocated; every later slot may still be in use and is waited for.
template <int D, int NSUB, bool KS, bool GLB>
__device__ __forceinline__ void producer_role(const CUtensorMap* tmQ, const CUtensorMap* tmK,
                                              const CUtensorMap* tmV, SmemBarriers& sb, uint8_t* smem,
                                              const Unit u, int hn_swapped, int* status, int j_from, int j_to,
                                              int& k_issued, int& v_issued) {
  using C = TileCfg<D, NSUB>;
  constexpr int NQ = KS ? 1 : NSUB;  // Q tiles: the key split's sub-tiles share their rows
  const bool swq = hn_swapped & 1, swk = (hn_swapped >> 1) & 1, swv = (hn_swapped >> 2) & 1;
  if (u.n_tot == 0) return;  // no row of this CTA reads a key
  if (j_from == 0) {
    mbar_arrive_expect_tx(&sb.q_full, NQ * C::Q_BYTES);
#pragma unroll
    for (int s = 0; s < NQ; ++s)
#pragma unroll
      for (int c = 0; c < C::NCHUNK; ++c)
        tma_load_tile(smem + C::OFF_Q + s * C::Q_BYTES + c * C::BM * C::SW_BYTES, tmQ, &sb.q_full,
                      c * C::SW_ELEMS, u.tok0q + u.row0 + s * u.span, u.h, u.bcoord, swq);
  }
  int ks = j_from % C::K_STAGES, kph = (j_from / C::K_STAGES) & 1;  // K ring slot and its phase for tile j
  for (int j = j_from; j < min(j_to, u.n_tot); ++j) {
    // Streamed tile j: key tile kt0 + j; in the global-token build the global
    // phase's key tiles 0 .. ng - 1, then the window phase's from wt0 on.
    const int key0 = u.tok0k + (GLB ? (j < u.ng ? j : u.wt0 + (j - u.ng)) : u.kt0 + j) * C::BN;
    // K_j goes to slot j % 3, whose previous tile j-3 must have been released.
    if (j >= C::K_STAGES && !mbar_wait(&sb.k_empty[ks], kph ^ 1, status)) return;
    {
      mbar_arrive_expect_tx(&sb.k_full[ks], C::KV_BYTES);
#pragma unroll
      for (int c = 0; c < C::NCHUNK; ++c)
        tma_load_tile(smem + C::OFF_K + ks * C::KV_BYTES + c * C::BN * C::SW_BYTES, tmK, &sb.k_full[ks],
                      c * C::SW_ELEMS, key0, u.hk, u.bcoord, swk);
      k_issued = j + 1;
    }
    if (++ks == C::K_STAGES) {
      ks = 0;
      kph ^= 1;
    }
    const int vs = j & 1;
    // V_j's slot held V_(j-2).  The key split releases it on its own barrier;
    // the other builds release it with step j - 1's commit on K_(j-1)'s slot.
    if constexpr (KS) {
      if (j >= 2 && !mbar_wait(&sb.v_empty[vs], ((j - 2) >> 1) & 1, status)) return;
    } else {
      if (j >= 2 && !mbar_wait(&sb.k_empty[(j - 1) % C::K_STAGES], ((j - 1) / C::K_STAGES) & 1, status)) return;
    }
    {
      mbar_arrive_expect_tx(&sb.v_full[vs], C::KV_BYTES);
#pragma unroll
      for (int c = 0; c < C::NCHUNK; ++c)
        tma_load_tile(smem + C::OFF_V + vs * C::KV_BYTES + c * C::BN * C::SW_BYTES, tmV, &sb.v_full[vs],
                      c * C::SW_ELEMS, key0, u.hk, u.bcoord, swv);
      v_issued = j + 1;
    }
  }
}

// Waits (bounded) until the last load issued into every ring slot has landed,
// so that no copy writes shared memory after the CTA exits.  After a normal
// run the consumers already saw these phases complete and every wait returns
// at once; after a wait ran out the loads still in flight are waited for.
template <int D, int NSUB>
__device__ __forceinline__ void producer_settle(SmemBarriers& sb, int k_issued, int v_issued) {
  using C = TileCfg<D, NSUB>;
  mbar_wait(&sb.q_full, 0, nullptr);
  for (int t = k_issued > C::K_STAGES ? k_issued - C::K_STAGES : 0; t < k_issued; ++t)
    mbar_wait(&sb.k_full[t % C::K_STAGES], (t / C::K_STAGES) & 1, nullptr);
  for (int t = v_issued > 2 ? v_issued - 2 : 0; t < v_issued; ++t) mbar_wait(&sb.v_full[t & 1], (t >> 1) & 1, nullptr);
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
// With split: then A = P_lo (columns [64, 128) of S_s) times the same V,
// accumulated onto O_s.  That second product is rare (only sub-tiles with
// few keys take it), so its loop is not unrolled: the issuing thread runs with
// few registers, and unrolled it would hold eight more addresses.
// H = 0 / 1 issues the steps of keys 0-63 / 64-127 only (released by p_half
// and p_full), H = 2 all of them.
template <int D, int NSUB, int H = 2>
__device__ __forceinline__ void issue_pv(const MmaDescs& md, uint32_t tmem, int s, int st, bool accumulate,
                                         uint32_t idesc, bool split) {
  using C = TileCfg<D, NSUB>;
  constexpr int K0 = H == 1 ? C::BN / 32 : 0, K1 = H == 0 ? C::BN / 32 : C::BN / 16;
  const uint64_t vd = st ? md.v1 : md.v0;
  const uint32_t p_base = tmem + C::TM_S + s * 128;
  const uint32_t d_tmem = tmem + C::TM_O + s * 128;
  const uint32_t acc0 = accumulate ? 1u : 0u;
#pragma unroll
  for (int kk = K0; kk < K1; ++kk)
    mma_ts(d_tmem, p_base + kk * 8, vd + (uint64_t)((kk * 16 * C::SW_BYTES) >> 4), idesc, kk > 0 ? 1u : acc0);
  if (split) {
#pragma unroll 1
    for (int kk = K0; kk < K1; ++kk)
      mma_ts(d_tmem, p_base + 64 + kk * 8, vd + (uint64_t)((kk * 16 * C::SW_BYTES) >> 4), idesc, 1u);
  }
}

// Runs on one thread: the tensor pipe queues only a couple of MMAs, so any
// cycle the issuing thread spends elsewhere between groups is idle tensor time.
// GEN = false is the square, window-free case, where both sub-tiles start at
// streamed tile 0 and the per-tile range tests fold away at compile time.
template <int D, int NSUB, bool GEN, bool KS, bool GLB, bool SPLIT>
__device__ __forceinline__ void mma_role(SmemBarriers& sb, uint8_t* smem, uint32_t tmem, const Unit u,
                                         uint32_t idesc_s, uint32_t idesc_pv, int* status) {
  using C = TileCfg<D, NSUB>;
  MmaDescs md;
  md.q0 = smem_desc(smem_u32(smem + C::OFF_Q), 16, C::SBO, C::SWIZZLE);
  md.q1 = KS ? md.q0 : md.q0 + (uint64_t)(C::Q_BYTES >> 4);
  md.k0 = smem_desc(smem_u32(smem + C::OFF_K), 16, C::SBO, C::SWIZZLE);
  md.k1 = md.k0 + (uint64_t)(C::KV_BYTES >> 4);
  md.k2 = md.k1 + (uint64_t)(C::KV_BYTES >> 4);
  md.v0 = smem_desc(smem_u32(smem + C::OFF_V), C::BN * C::SW_BYTES, C::SBO, C::SWIZZLE);
  md.v1 = md.v0 + (uint64_t)(C::KV_BYTES >> 4);
  // Sub-tile `sub` reads streamed tile j; its own count of that tile.
  // Key split: sub-tile s reads the streamed tiles j = s mod 2.
  // Global-token build: sub-tile s reads the global phase's streamed tiles
  // 0 .. ga(s) - 1 and then n(s) - ga(s) window-phase tiles from f(s) on.
  auto reads = [&](int sub, int j) {
    if constexpr (GLB)
      return j < u.ng ? j < u.ga(sub) : (unsigned)(j - u.f(sub)) < (unsigned)(u.n(sub) - u.ga(sub));
    else
      return KS ? ((j & 1) == sub && j < u.n_tot) : (GEN ? u.reads(sub, j) : j < u.n(sub));
  };
  auto own = [&](int sub, int j) {
    if constexpr (GLB)
      return j < u.ng ? j : u.ga(sub) + (j - u.f(sub));
    else
      return KS ? j >> 1 : (GEN ? j - u.f(sub) : j);
  };
  if (u.n_tot == 0) return;  // no row of this CTA reads a key
  const uint32_t split = SPLIT ? sb.split_mask : 0u;  // SPLIT = false: no second product anywhere
  if (!mbar_wait(&sb.q_full, 0, status)) return;

  if constexpr (KS) {
    // Key split: sub-tile s owns the streamed tiles t = 2 jl + s.  Step jl
    // issues PV_0(jl-1), S_0(jl), PV_1(jl-1), S_1(jl), so the two chains
    // take turns on the tensor core as the two sub-tiles of a regular CTA
    // do.  K tile t sits in ring slot t mod 3 (phase t / 3), V tile t in
    // slot t mod 2 (phase t / 2).
    for (int jl = 0; jl <= u.n0; ++jl) {
#pragma unroll
      for (int sub = 0; sub < 2; ++sub) {
        const int tp = 2 * (jl - 1) + sub;  // tile whose PV product is issued now
        if (jl > 0 && tp < u.n_tot) {
          if (!mbar_wait(&sb.v_full[tp & 1], (tp >> 1) & 1, status) ||
              !mbar_wait(&sb.p_full[sub], (jl - 1) & 1, status))
            return;
          tc_fence_after();
          issue_pv<D, NSUB>(md, tmem, sub, tp & 1, jl > 1, idesc_pv, (split >> sub) & 1u);
          if (jl - 1 == u.n(sub) - 1) mma_commit(&sb.o_done[sub]);
          mma_commit(&sb.v_empty[tp & 1]);
        }
        const int tn = 2 * jl + sub;  // tile whose S product is issued now
        if (tn < u.n_tot) {
          if (!mbar_wait(&sb.k_full[tn % C::K_STAGES], (tn / C::K_STAGES) & 1, status)) return;
          tc_fence_after();
          issue_s<D, NSUB>(md, tmem, sub, tn % C::K_STAGES, idesc_s);
          mma_commit(&sb.s_full[sub]);
          mma_commit(&sb.k_empty[tn % C::K_STAGES]);
        }
      }
    }
  } else {
  int ks = 0, kph = 0;  // K ring slot / phase of the next key tile
  if (!mbar_wait(&sb.k_full[0], 0, status)) return;
  tc_fence_after();
#pragma unroll
  for (int sub = 0; sub < 2; ++sub) {
    if (reads(sub, 0)) {
      issue_s<D, NSUB>(md, tmem, sub, 0, idesc_s);
      mma_commit(&sb.s_full[sub]);
    }
  }
  mma_commit(&sb.k_empty[0]);
  ks = 1;
  // Step j issues the PV products of streamed tile j - 1 and the S products
  // of tile j, interleaved by sub-tile.
  // The step's one release commit (on K_j's slot, after S_1(j)) also
  // covers the PV products of tile j - 1 issued before it, so it frees V_(j-1)'s
  // slot as well: the producer waits on it for V_(j+1) too.  Every wait and
  // commit costs this thread a couple of hundred cycles of tensor idle time,
  // so each step makes one release commit and waits for V only once.
  for (int j = 1; j <= u.n_tot; ++j) {
    const int i = j - 1;  // key tile whose PV products are issued in this step
    const bool has_k = j < u.n_tot;
    if (has_k && !mbar_wait(&sb.k_full[ks], kph, status)) return;
    bool v_ready = false;
#pragma unroll
    for (int sub = 0; sub < 2; ++sub) {
      if (reads(sub, i)) {  // PV_sub(i)
        const int li = own(sub, i);
        if (!v_ready && !mbar_wait(&sb.v_full[i & 1], (i >> 1) & 1, status)) return;
        v_ready = true;
        if (!mbar_wait(&sb.p_half[sub], li & 1, status)) return;
        tc_fence_after();
        issue_pv<D, NSUB, 0>(md, tmem, sub, i & 1, li > 0, idesc_pv, (split >> sub) & 1u);
        if (!mbar_wait(&sb.p_full[sub], li & 1, status)) return;
        tc_fence_after();
        issue_pv<D, NSUB, 1>(md, tmem, sub, i & 1, li > 0, idesc_pv, (split >> sub) & 1u);
        if (li == u.n(sub) - 1) mma_commit(&sb.o_done[sub]);
      }
      if (has_k && reads(sub, j)) {  // S_sub(j)
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
  }
  // Drain: wait for the commit arrivals nobody else consumes (the last
  // tiles' ring releases and the final PV of each sub-tile) so that no
  // arrival can land in shared memory after the CTA exits.
  for (int t = u.n_tot > C::K_STAGES ? u.n_tot - C::K_STAGES : 0; t < u.n_tot; ++t)
    if (!mbar_wait(&sb.k_empty[t % C::K_STAGES], (t / C::K_STAGES) & 1, status)) return;
  if constexpr (KS)
    for (int t = u.n_tot >= 2 ? u.n_tot - 2 : 0; t < u.n_tot; ++t)
      if (!mbar_wait(&sb.v_empty[t & 1], (t >> 1) & 1, status)) return;
#pragma unroll
  for (int sub = 0; sub < 2; ++sub)
    if (u.n(sub) > 0 && !mbar_wait(&sb.o_done[sub], 0, status)) return;
}

// ----------------------------------------------------------------- softmax / correction / epilogue
// Warp-wide wait: while the phase is still open, lane 0 alone polls the
// barrier and the outcome is broadcast, so one thread per warp (not 32)
// keeps touching the barrier word.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, int* status) {
  // Fast path: every lane probes once, and a phase that has already
  // completed (the common case) costs one probe and a vote.  Otherwise lane 0
  // waits (bounded) and hands the outcome to the warp.
  if (__all_sync(0xffffffffu, mbar_try_wait(bar, parity))) return true;
  bool ok = true;
  if ((threadIdx.x & 31) == 0) ok = mbar_wait(bar, parity, status);
  return __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
}

template <bool BF16>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  return BF16 ? pack_bf16x2(lo, hi) : pack_f16x2(lo, hi);
}
template <bool BF16>
__device__ __forceinline__ void unpack2(uint32_t w, float& lo, float& hi) {
  if constexpr (BF16)
    unpack_bf16x2(w, lo, hi);
  else
    unpack_f16x2(w, lo, hi);
}

// GEN = false is the square, window-free case: every row reads key 0 in the
// first tile, so no row meets a tile with m = -inf and no lower edge exists.
template <int D, int NSUB, bool BF16, bool GEN, bool KS, bool GLB, bool SPLIT>
__device__ __forceinline__ void softmax_role(SmemBarriers& sb, uint32_t tmem, const FwdParams& p, const Unit u,
                                             int s) {
  using C = TileCfg<D, NSUB>;
  constexpr uint32_t FULL = 0xffffffffu;
  const int n = u.n(s);
  const int t = threadIdx.x & 127;  // row inside the sub-tile = tensor-memory lane
  // Row t holds query head u.h + hl at token tl of the sub-tile.  A packed Q
  // box is laid out head-major ((d, token, head) maps) or token-major
  // ((d, head, token) maps).
  int hl = 0, tl = t;
  if (GEN && u.P > 1) {
    if (p.hn_swapped & 1) {
      hl = t & (u.P - 1);
      tl = t / u.P;
    } else {
      hl = t / u.span;
      tl = t & (u.span - 1);
    }
  }
  const int head = u.h + hl;
  const int row_pos = u.row0 + (KS ? 0 : s * u.span) + tl;  // logical position inside the query sequence
  const bool valid = row_pos < u.Lq;
  // Output row and lse addresses (formed where they are used, so that they
  // hold no registers across the tile loop).
  auto o_row = [&]() {
    return reinterpret_cast<uint8_t*>(p.o) +
           2 * ((int64_t)u.b * p.o_sb + (int64_t)head * p.o_sh + (int64_t)(u.tok0q + row_pos) * p.o_sn);
  };
  auto lse_index = [&]() { return (int64_t)u.b * p.lse_sb + (int64_t)head * p.lse_sh + u.tok0q + row_pos; };
  auto lse_at = [&]() { return p.lse + lse_index(); };
  // Split-KV partial row: FP32 O_s and lse_s of this CTA's key slice.
  auto part_index = [&]() { return (int64_t)u.split * p.part_stride + lse_index(); };
  auto part_row = [&]() { return p.part_o + part_index() * D; };
  const bool split_mode = GEN && p.part_o != nullptr;
  if (KS && s == 1 && n == 0) {  // key split, nothing for sub-tile 1: an empty state
    sb.merge_m[t] = -INFINITY;
    sb.merge_l[t] = 0.f;
    mbar_arrive(&sb.merge_ready);
    return;
  }
  if (n == 0) {  // no row of this sub-tile may read a key: O = 0, lse = -inf
    if (valid) {
      if (split_mode) {
        float* prow = part_row();
#pragma unroll
        for (int c = 0; c < D; c += 4) *reinterpret_cast<uint4*>(prow + c) = make_uint4(0u, 0u, 0u, 0u);
        p.part_lse[part_index()] = -INFINITY;
      } else {
        uint8_t* orow = o_row();
#pragma unroll
        for (int c = 0; c < D; c += 8) *reinterpret_cast<uint4*>(orow + c * 2) = make_uint4(0u, 0u, 0u, 0u);
        if (p.lse != nullptr) *lse_at() = -INFINITY;
      }
    }
    return;
  }
  // A warp none of whose rows exists (all past the query length: a ragged
  // last block) keeps the barrier protocol and nothing else.  It releases
  // each score tile without writing P (the PV product then fills only rows
  // that are never stored), hands sub-tile 0 an empty state under the key
  // split, and skips the epilogue.
  if (!__any_sync(FULL, valid)) {
    for (int j = 0; j < n; ++j) {
      if (!warp_wait(&sb.s_full[s], j & 1, p.status)) return;
      if constexpr (!KS) mbar_arrive(&sb.p_half[s]);
      mbar_arrive(&sb.p_full[s]);
    }
    if (KS && s == 1) {
      sb.merge_m[t] = -INFINITY;
      sb.merge_l[t] = 0.f;
      mbar_arrive(&sb.merge_ready);
    }
    return;
  }
  const uint32_t lane_off = (uint32_t)(((threadIdx.x >> 5) & 3) * 32) << 16;
  const uint32_t tS = tmem + C::TM_S + s * 128 + lane_off;
  const uint32_t tO = tmem + C::TM_O + s * 128 + lane_off;
  const float c2 = p.scale_log2;
  constexpr bool split_p = SPLIT;  // the MMA thread adds the second product
  int* status = p.status;
  // Keys this row may read, as offsets from the first key of the current
  // tile: lim_lo <= i <= lim_hi.  Both move down by one tile per step.
  const int c_row = row_pos + u.delta;
  const int kb0 = (u.kt0 + u.f(s)) * C::BN;
  int lim_hi, lim_lo;
  int win_hi = 0, win_lo = 0;  // global-token build: the window phase's limits, taken up at tile ga(s)
  if constexpr (GLB) {
    // The global phase reads key tiles 0 .. ga(s) - 1 (limits of part 1), the
    // window phase the tiles from wt0 + (f(s) - ng) on (limits of part 0).
    const int2 kg = row_key_range(c_row, u, p, 1), kw = row_key_range(c_row, u, p, 0);
    const int kbw = (u.wt0 + (u.f(s) - u.ng)) * C::BN;
    win_hi = kw.y - kbw;
    win_lo = kw.x - kbw;
    lim_hi = u.ga(s) > 0 ? kg.y : win_hi;
    lim_lo = u.ga(s) > 0 ? kg.x : win_lo;
  } else if constexpr (GEN) {
    const int2 kr = row_key_range(c_row, u, p, 0);
    lim_hi = kr.y - kb0;
    lim_lo = kr.x - kb0;
  } else {
    lim_hi = min(u.Lk - 1, c_row + p.win_right) - kb0;
    lim_lo = max(0, c_row - p.win_left) - kb0;
  }
  float m_run = -INFINITY;  // running maximum of the raw scores (scale > 0)
  bool window_first = true;  // global-token build: no window-phase key of this row seen yet
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
    // Mask keys past the diagonal (causal), the window or the sequence end.
    // Only tiles on those edges need masking; the tests are warp-uniform so
    // that other tiles skip the per-element selects entirely, and a lower
    // edge (a window's left end) exists only for windowed calls.
    const bool warp_masked = __any_sync(FULL, GEN ? (lim_hi < C::BN - 1 || lim_lo > 0) : lim_hi < C::BN - 1);
    const bool warp_lower = GEN && warp_masked && __any_sync(FULL, lim_lo > 0);
#pragma unroll
    for (int i = 0; i < C::BN / 2; ++i) sv[i] = __uint_as_float(sr[i]);
    if (warp_lower) {
#pragma unroll
      for (int i = 0; i < C::BN / 2; ++i) sv[i] = (i > lim_hi || i < lim_lo) ? -INFINITY : sv[i];
    } else if (warp_masked) {
#pragma unroll
      for (int i = 0; i < C::BN / 2; ++i) sv[i] = i > lim_hi ? -INFINITY : sv[i];
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
    if (warp_lower) {
#pragma unroll
      for (int i = C::BN / 2; i < C::BN; ++i) sv[i] = (i > lim_hi || i < lim_lo) ? -INFINITY : sv[i];
    } else if (warp_masked) {
#pragma unroll
      for (int i = C::BN / 2; i < C::BN; ++i) sv[i] = i > lim_hi ? -INFINITY : sv[i];
    }
    lim_hi -= (KS ? 2 : 1) * C::BN;  // the key split's sub-tiles take every other tile
    lim_lo -= (KS ? 2 : 1) * C::BN;
    if constexpr (GLB) {
      if (j + 1 == u.ga(s)) {  // the next tile opens the window phase
        lim_hi = win_hi;
        lim_lo = win_lo;
      }
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
    // than 8 in log2 units (always on the first tile, and always when the row
    // sees its first eligible key: -inf to finite compares as +inf > 8).
    bool rescale = (j == 0) || (m_new - m_run) * c2 > 8.f;
    // Global-token build: the global phase sets the reference maximum from the
    // global keys alone, so the row's first window-phase tile that holds one
    // of its keys takes up any larger maximum exactly; otherwise a small
    // window's dominant key would enter P as a rounded value above 1 instead
    // of exactly 1, and O would lose about a 16-bit rounding of its largest
    // term.
    if constexpr (GLB) {
      if (j >= u.ga(s) && m_tile != -INFINITY) {
        rescale = rescale || (window_first && m_new > m_run);
        window_first = false;
      }
    }
    float alpha = 1.f;
    if (rescale) {
      alpha = (j == 0) ? 0.f : ex2_approx((m_run - m_new) * c2);
      m_run = m_new;
    }
    // A row that has not met an eligible key yet keeps m = -inf; its masked
    // scores must still give p = exp2(-inf) = 0, not exp2(-inf + inf).
    const float neg_mc = (GEN && m_run == -INFINITY) ? 0.f : -m_run * c2;
    // Correction: O_s *= alpha for rows whose maximum moved.  PV_s(j-1) has
    // completed: the commit that signalled S_s(j) covers it.  It comes before
    // any part of P_s(j) is released, since the PV products add onto O_s.
    // (Sixteen columns at a time: the scores are still held in registers.)
    if (j > 0 && __any_sync(FULL, rescale)) {
#pragma unroll 1
      for (int c = 0; c < D; c += 16) {
        uint32_t o[16];
        tmem_ld_x16(tO + c, o);
        tmem_ld_wait16(o);
#pragma unroll
        for (int i = 0; i < 16; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
        tmem_st_x16(tO + c, o);
      }
    }
    // p = exp2(s * c2 - m * c2): the scaling runs two lanes per instruction,
    // the row sum in four independent pairs of accumulators.  P_s(j) goes
    // over the first 64 cells of S_s(j) in two halves: keys 0-63 are stored as
    // soon as they are ready and released on p_half, so that the first half of
    // the PV product runs on the tensor core while keys 64-127 are computed
    // (the release waits two more steps of the loop, hiding the stores).
    // With split_p, P = P_hi + P_lo: the residual P - P_hi, rounded, goes to
    // columns [64, 128) (whose scores are in registers already), four columns
    // at a time, so that no array of it is held.
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
      if constexpr (split_p) {
        uint32_t r[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          float h0, h1, d0, d1;
          unpack2<BF16>(pk[i + k], h0, h1);
          fma2(d0, d1, h0, h1, -1.f, -1.f, x[2 * k], x[2 * k + 1]);
          r[k] = pack2<BF16>(d0, d1);
        }
        tmem_st_x4(tS + 64 + i, r[0], r[1], r[2], r[3]);
      }
      if (i == 28) tmem_st_x32(tS, pk);  // keys 0-63
      if constexpr (!KS) {
        if (i == 36) {
          tmem_st_wait();
          tc_fence_before();
          mbar_arrive(&sb.p_half[s]);
        }
      }
    }
    l_run = l_run * alpha + (((ra0 + rb0) + (rc0 + rd0)) + ((ra1 + rb1) + (rc1 + rd1)));
    tmem_st_x32(tS + 32, pk + 32);  // keys 64-127
    tmem_st_wait();
    tc_fence_before();
    mbar_arrive(&sb.p_full[s]);
  }

  // Epilogue: O = O_acc / l in the input type, lse = scale * m + ln l.  A
  // row that met no eligible key has l = 0 and O_acc = 0 (every p was 0):
  // it gets O = 0 and lse = -inf.
  if (!warp_wait(&sb.o_done[s], 0, status)) return;
  tc_fence_after();
  if (KS && s == 1) {  // hand the state to sub-tile 0
    sb.merge_m[t] = m_run;
    sb.merge_l[t] = l_run;
    tc_fence_before();
    mbar_arrive(&sb.merge_ready);
    return;
  }
  // Key split: merge sub-tile 1's state into this one, rescaling both to the
  // larger reference maximum; O_1 is read from sub-tile 1's columns.
  float w0 = 1.f, w1 = 0.f;
  if (KS) {
    if (!warp_wait(&sb.merge_ready, 0, status)) return;
    tc_fence_after();
    const float m1 = sb.merge_m[t], l1 = sb.merge_l[t];
    if (l1 > 0.f) {
      const float mm = fmaxf(m_run, m1);
      w0 = l_run > 0.f ? ex2_approx((m_run - mm) * c2) : 0.f;
      w1 = ex2_approx((m1 - mm) * c2);
      l_run = l_run * w0 + l1 * w1;
      m_run = mm;
    }
  }
  const bool nonempty = l_run > 0.f;
  const float inv_l = nonempty ? 1.f / l_run : 0.f;
  if (split_mode) {
    float* prow = part_row();
#pragma unroll
    for (int c = 0; c < D; c += 32) {
      uint32_t o[32];
      tmem_ld_x32(tO + c, o);
      tmem_ld_wait32(o);
      if (valid) {
        uint4* dst = reinterpret_cast<uint4*>(prow + c);
#pragma unroll
        for (int i = 0; i < 8; ++i)
          dst[i] = make_uint4(__float_as_uint(__uint_as_float(o[4 * i]) * inv_l),
                              __float_as_uint(__uint_as_float(o[4 * i + 1]) * inv_l),
                              __float_as_uint(__uint_as_float(o[4 * i + 2]) * inv_l),
                              __float_as_uint(__uint_as_float(o[4 * i + 3]) * inv_l));
      }
    }
    if (valid)
      p.part_lse[part_index()] = nonempty ? m_run * p.scale + __logf(l_run) : -INFINITY;
    return;
  }
  uint8_t* orow = o_row();
  const float s0 = w0 * inv_l, s1 = w1 * inv_l;
#pragma unroll
  for (int c = 0; c < D; c += 32) {
    uint32_t o[32];
    tmem_ld_x32(tO + c, o);
    tmem_ld_wait32(o);
    if (KS && u.n1 > 0) {  // + w1 * O_1 (sub-tile 1's accumulator, same lanes; CTA-uniform branch)
      uint32_t o1[32];
      tmem_ld_x32(tO + 128 + c, o1);
      tmem_ld_wait32(o1);
#pragma unroll
      for (int i = 0; i < 32; ++i)
        o[i] = __float_as_uint(fmaf(__uint_as_float(o1[i]), s1, __uint_as_float(o[i]) * s0));
    } else if (KS) {
#pragma unroll
      for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * s0);
    }
    const float sc = KS ? 1.f : inv_l;
    uint32_t w[16];
#pragma unroll
    for (int i = 0; i < 16; ++i)
      w[i] = pack2<BF16>(__uint_as_float(o[2 * i]) * sc, __uint_as_float(o[2 * i + 1]) * sc);
    if (valid) {
      uint4* dst = reinterpret_cast<uint4*>(orow + c * 2);
      dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
      dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
      dst[2] = make_uint4(w[8], w[9], w[10], w[11]);
      dst[3] = make_uint4(w[12], w[13], w[14], w[15]);
    }
  }
  if (valid && p.lse != nullptr) *lse_at() = nonempty ? m_run * p.scale + __logf(l_run) : -INFINITY;
}

// ----------------------------------------------------------------- kernel
// Logical grid: x = query block (NSUB * 128 rows) counted from the last one,
// y = query head, z = batch (or sequence), dispatched in the grouped
// longest-first order of cta_coords: the CTAs running at any time belong to
// one group of heads and share its K/V tiles in L2, and within the group the
// longest causal rows start first.  NSUB = 2 (two sub-tiles taking turns on the tensor core) is the
// throughput configuration; NSUB = 1 gives small problems twice as many CTAs.
// GEN = true handles unequal lengths and windows; the square, window-free
// case compiles without their per-tile tests (they cost about 3% there).
template <int D, int NSUB, bool BF16, bool GEN, bool KS, bool GLB, bool SPL>
__global__ void __launch_bounds__(TileCfg<D, NSUB>::THREADS, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const FwdParams p) {
  using C = TileCfg<D, NSUB>;
  __shared__ SmemBarriers sb;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

  // The next launch on the stream may be scheduled now.  Barrier set-up and
  // the tensor-memory allocation touch no global memory and run before this
  // grid waits for the previous one (whose outputs may be its inputs, or
  // whose inputs its outputs); everything after the wait may read and write.
  pdl_launch_dependents();
  const int warp = threadIdx.x >> 5;
  const bool producer = warp == C::PRODUCER_WARP && (threadIdx.x & 31) == 0;
  if (producer) {
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
      mbar_init(&sb.p_half[i], 128);
      mbar_init(&sb.o_done[i], 1);
    }
    mbar_init(&sb.merge_ready, 128);
    mbar_init(&sb.fin, 1);
    fence_mbar_init();
    fence_proxy_async_smem();  // the initialised barriers, as the TMA (async proxy) will see them
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
  }
  if (warp == C::MMA_WARP) {
    tmem_alloc(&sb.tmem_base, C::TMEM_COLS);
    tmem_relinquish();
  }
  pdl_wait();

  // The CTA's work; `active` is uniform across the CTA.
  bool active = true;
  const int3 cta = cta_coords(p);
  Unit u;
  u.P = GEN ? p.qpack : 1;
  u.span = C::BM / u.P;
  u.h = cta.y * u.P;
  u.b = cta.z;
  u.hk = u.h / p.group;
  u.Lq = p.Nq;
  u.Lk = p.Nk;
  u.tok0q = u.tok0k = 0;
  u.bcoord = u.b;
  if (p.cu_seqlens_q != nullptr) {
    const int q0 = p.cu_seqlens_q[u.b], q1 = p.cu_seqlens_q[u.b + 1];
    const int k0 = p.cu_seqlens_k[u.b], k1 = p.cu_seqlens_k[u.b + 1];
    if (q0 < 0 || q1 < q0 || q1 > p.total_q || q1 - q0 > p.max_seqlen_q || k0 < 0 || k1 < k0 ||
        k1 > p.total_k || k1 - k0 > p.max_seqlen_k) {
      if (threadIdx.x == 0) atomicCAS(p.status, 0, (int)kDevBadSeqlens);
      active = false;
    }
    u.Lq = q1 - q0;
    u.Lk = k1 - k0;
    u.tok0q = q0;
    u.tok0k = k0;
    u.bcoord = 0;
  }
  // x counts query blocks from the last one; in a split-KV launch the slices
  // of one block are adjacent.
  int block = p.grid_x - 1 - cta.x;
  u.split = 0;
  if (GEN && p.part_o != nullptr) {
    u.split = cta.x % p.num_splits;
    block = p.grid_x / p.num_splits - 1 - cta.x / p.num_splits;
  }
  u.row0 = block * (KS ? 1 : NSUB) * u.span;
  if (u.row0 >= u.Lq) active = false;
  u.delta = u.Lk - u.Lq;
  u.kt0 = u.n_tot = u.f0 = u.f1 = u.n0 = u.n1 = 0;
  u.ng = u.wt0 = u.ga0 = u.ga1 = 0;
  if (!active) {
  } else if (GLB) {
    // Global tokens: each sub-tile streams the global keys' tiles (part 1,
    // from key tile 0), then the tiles of the rest of its rows' keys (part 0).
    // The CTA streams the longest global phase, then the union of the
    // window phases; a tile holding both key G - 1 and later keys is read in
    // both phases, masked to disjoint keys.
    const int2 g0 = sub_tile_key_tiles(u.row0, u.span, u, p, C::BN, 1);
    const int2 g1 = NSUB == 2 ? sub_tile_key_tiles(u.row0 + u.span, u.span, u, p, C::BN, 1) : make_int2(0, 0);
    const int2 w0 = sub_tile_key_tiles(u.row0, u.span, u, p, C::BN, 0);
    const int2 w1 = NSUB == 2 ? sub_tile_key_tiles(u.row0 + u.span, u.span, u, p, C::BN, 0) : make_int2(0, 0);
    u.ga0 = g0.y;  // part 1 starts at key tile 0 (or is empty: {0, 0})
    u.ga1 = g1.y;
    u.ng = max(u.ga0, u.ga1);
    const bool a0 = w0.y > w0.x, a1 = w1.y > w1.x;
    u.wt0 = a0 ? (a1 ? min(w0.x, w1.x) : w0.x) : (a1 ? w1.x : 0);
    u.n_tot = u.ng + ((a0 || a1) ? max(a0 ? w0.y : 0, a1 ? w1.y : 0) - u.wt0 : 0);
    u.f0 = a0 ? u.ng + w0.x - u.wt0 : u.ng;
    u.n0 = u.ga0 + (a0 ? w0.y - w0.x : 0);
    u.f1 = a1 ? u.ng + w1.x - u.wt0 : u.ng;
    u.n1 = u.ga1 + (a1 ? w1.y - w1.x : 0);
  } else if (KS) {  // one row block; sub-tile s takes the streamed tiles j = s mod 2
    const int2 r = sub_tile_key_tiles(u.row0, u.span, u, p, C::BN);
    u.kt0 = r.x;
    u.n_tot = r.y > r.x ? r.y - r.x : 0;
    u.f0 = 0;
    u.f1 = 1;
    u.n0 = (u.n_tot + 1) / 2;
    u.n1 = u.n_tot / 2;
  } else {
    int2 r0 = sub_tile_key_tiles(u.row0, u.span, u, p, C::BN);
    int2 r1 = NSUB == 2 ? sub_tile_key_tiles(u.row0 + u.span, u.span, u, p, C::BN) : make_int2(0, 0);
    if (GEN && p.part_o != nullptr && p.num_global == 0) {  // keep this slice's key tiles
      const int lo = u.split * p.split_tiles, hi = lo + p.split_tiles;
      r0 = make_int2(max(r0.x, lo), min(r0.y, hi));
      r1 = make_int2(max(r1.x, lo), min(r1.y, hi));
    }
    const bool a0 = r0.y > r0.x, a1 = r1.y > r1.x;
    u.kt0 = a0 ? (a1 ? min(r0.x, r1.x) : r0.x) : (a1 ? r1.x : 0);
    u.n_tot = (a0 || a1) ? max(a0 ? r0.y : 0, a1 ? r1.y : 0) - u.kt0 : 0;
    u.f0 = a0 ? r0.x - u.kt0 : 0;
    u.n0 = a0 ? r0.y - r0.x : 0;
    u.f1 = a1 ? r1.x - u.kt0 : 0;
    u.n1 = a1 ? r1.y - r1.x : 0;
  }
  // Q and the first key tile go out before the CTA's barrier: their slots
  // are free and only this thread has touched the barriers yet.
  int k_issued = 0, v_issued = 0;  // key / value tiles the producer has issued
  if (producer && active)
    producer_role<D, NSUB, KS, GLB>(&tmQ, &tmK, &tmV, sb, smem, u, p.hn_swapped, p.status, 0, 1, k_issued, v_issued);
  if (SPL && producer) sb.split_mask = active ? split_mask<NSUB, KS>(u, p) : 0u;
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sb.tmem_base;

  if (!active) {
  } else if (warp < 4 * NSUB) {
    if constexpr (NSUB == 2) regs_grow<C::SOFTMAX_REGS>();
    if (SPL && ((sb.split_mask >> (warp >> 2)) & 1u))
      softmax_role<D, NSUB, BF16, GEN, KS, GLB, SPL>(sb, tmem, p, u, warp >> 2);
    else
      softmax_role<D, NSUB, BF16, GEN, KS, GLB, false>(sb, tmem, p, u, warp >> 2);
  } else {
    if constexpr (NSUB == 2) regs_shrink<C::CTRL_REGS>();
    const bool lane0 = (threadIdx.x & 31) == 0;
    if (warp == C::PRODUCER_WARP) {
      if (lane0) {
        producer_role<D, NSUB, KS, GLB>(&tmQ, &tmK, &tmV, sb, smem, u, p.hn_swapped, p.status, 1, 1 << 30, k_issued,
                                   v_issued);
        if (u.n_tot > 0) producer_settle<D, NSUB>(sb, k_issued, v_issued);
      }
      __syncwarp();
    } else if (warp == C::MMA_WARP) {
      constexpr uint32_t ab = BF16 ? 1u : 0u;
      constexpr uint32_t idesc_s = instr_desc_f16(128, C::BN, ab, false, false);
      constexpr uint32_t idesc_pv = instr_desc_f16(128, D, ab, false, true);
      if (lane0) {
        if (SPL && sb.split_mask != 0u)
          mma_role<D, NSUB, GEN, KS, GLB, SPL>(sb, smem, tmem, u, idesc_s, idesc_pv, p.status);
        else
          mma_role<D, NSUB, GEN, KS, GLB, false>(sb, smem, tmem, u, idesc_s, idesc_pv, p.status);
        // Every MMA this thread issued has completed before tensor memory is
        // released (immediate after a normal run; bounded after a wait ran out).
        mma_commit(&sb.fin);
        mbar_wait(&sb.fin, 0, nullptr);
      }
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

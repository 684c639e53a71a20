/*
 * etattn.h: C ABI of the exact streaming self-attention forward pass for
 * NVIDIA GB300 (sm_103a).
 *
 * Operation ("Intermediate and advanced extension", workshop table row
 * "Streaming attention" and "Logic review before implementation"):
 *
 *   O_i   = sum_{j in E(i)} exp(s_ij - M_i) v_j / sum_{j in E(i)} exp(s_ij - M_i)
 *   lse_i = M_i + ln sum_{j in E(i)} exp(s_ij - M_i)        (natural log, FP32)
 *   s_ij  = scale * <q_i, k_j>,   M_i = max_{j in E(i)} s_ij
 *
 * computed tile by tile with a running maximum and a rescaled exponential sum,
 * rescaling both the numerator accumulator and the denominator whenever the
 * maximum grows, without ever materialising the score matrix.  E(i) is every
 * key, or under the causal mask the keys j <= i (the diagonal is included, so
 * no causal row of a square problem is empty).  Grouped-query attention
 * ("Attention algorithms and data movement", lesson 05): query head h reads
 * key/value head h / (Hq / Hkv).  Packed variable-length batches (same page,
 * lesson 04): positions are logical positions inside each sequence and no key
 * is eligible across sequences.
 *
 * The *_ex entry points add unequal query and key lengths (same page, lesson
 * 04) and local windows (same page, lesson 07).  Query row i of Lq sits at
 * key position c_i = i + Lk - Lq, so that the last query row aligns with the
 * last key (a decode step or a chunk of new tokens over a longer cache).  Key
 * j is eligible for row i iff
 *     j <= c_i                        (causal)
 *     c_i - window_left <= j          (window_left  >= 0; negative = no bound)
 *     j <= c_i + window_right         (window_right >= 0; negative = no bound)
 * A row with no eligible key (Lk = 0, or Lq > Lk under the causal mask, or a
 * window past the keys) gets O_i = 0 and lse_i = -inf.  The *_global entry
 * points add global tokens (same page, lesson 07): with G of them, key j is
 * also eligible when j < G, and every key when c_i < G, both still under the
 * causal mask but not the window.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - q, k, v, o are DEVICE pointers to FP16 or BF16 data (all four the same
 *    type, chosen by `dtype`); lse is a DEVICE pointer to FP32 or NULL (then
 *    no logsumexp is written).  Strides are in ELEMENTS, not bytes.
 *  - The caller owns every buffer.  Inputs are only read; o and lse are only
 *    written (o and lse must not overlap q, k, v or each other).  The library
 *    allocates no device memory per call.
 *  - Calls are asynchronous on `stream` (a cudaStream_t; NULL = the legacy
 *    default stream) and never synchronise the host.
 *  - Every argument is validated before anything is launched; a non-zero
 *    return value is an ETATTN_ERR_* code and nothing was launched.  No C++
 *    exception crosses this boundary.
 *  - Supported: head dim D in {32, 64, 128}; the d-stride of every tensor is
 *    1; all other strides and every base pointer are 16-byte aligned (TMA
 *    rule); scale is finite and > 0.
 *  - Empty work (B, Hq or N equal to 0; or no query tokens) is a successful
 *    no-op.
 *  - Limits: every length <= 2^30 tokens; B, Hq and num_seqs <= 65535.
 */
#ifndef ETATTN_H
#define ETATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Element types of q, k, v, o. */
enum etattn_dtype { ETATTN_F16 = 0, ETATTN_BF16 = 1 };

/* Status codes. */
enum etattn_status {
  ETATTN_OK = 0,
  ETATTN_ERR_NULL_PTR = 1,     /* a required pointer is NULL */
  ETATTN_ERR_BAD_DTYPE = 2,    /* dtype is not ETATTN_F16 / ETATTN_BF16 */
  ETATTN_ERR_BAD_SHAPE = 3,    /* negative size, D not in {32,64,128}, or a size beyond the limits */
  ETATTN_ERR_BAD_HEADS = 4,    /* Hkv <= 0 or Hq not a multiple of Hkv */
  ETATTN_ERR_BAD_STRIDE = 5,   /* d-stride != 1, negative stride, or a stride not a multiple of 16 bytes */
  ETATTN_ERR_BAD_ALIGN = 6,    /* a base pointer is not 16-byte aligned */
  ETATTN_ERR_ALIAS = 7,        /* o or lse overlaps an input, or o overlaps lse */
  ETATTN_ERR_BAD_SCALE = 8,    /* scale is not finite or not > 0 */
  ETATTN_ERR_BAD_SEQLENS = 9,  /* cu_seqlens not non-decreasing from 0 to total_tokens, or a length > max_seqlen */
  ETATTN_ERR_LAUNCH = 10,      /* a CUDA runtime call failed (the CUDA error is in etattn_last_cuda_error) */
  ETATTN_ERR_DEVICE = 11,      /* the device reported a failure (see etattn_read_device_status) */
  ETATTN_ERR_NO_DEVICE = 12,   /* no sm_103 device is current */
};

/*
 * attn_fwd: batched multi-head (optionally grouped-query) self-attention.
 *
 *   q  : logical [B, Hq,  N, D], element (b,h,n,d) at q[b*sq[0] + h*sq[1] + n*sq[2] + d*sq[3]]
 *   k,v: logical [B, Hkv, N, D], strides sk / sv likewise
 *   o  : logical [B, Hq,  N, D], strides so likewise
 *   lse: [B, Hq, N] contiguous FP32 (or NULL)
 *   strides: 16 int64 values, sq[4], sk[4], sv[4], so[4], each (b, h, n, d).
 *            [B,H,N,D]-contiguous and [B,N,H,D]-contiguous storage are both
 *            expressible; the d-stride must be 1.
 *   causal : 0 = every key eligible; 1 = keys j <= i (diagonal included)
 *   scale  : logit scale (commonly 1/sqrt(D))
 */
int attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv, int N,
             int D, int dtype, const int64_t* strides, int causal, float scale, void* stream);

/*
 * attn_fwd_varlen: packed variable-length batch of num_seqs sequences.
 *
 *   q  : logical [T, Hq,  D], element (t,h,d) at q[t*sq[0] + h*sq[1] + d*sq[2]]
 *   k,v: logical [T, Hkv, D]
 *   o  : logical [T, Hq,  D]
 *   lse: [Hq, T] contiguous FP32 (or NULL)
 *   strides: 12 int64 values, sq[3], sk[3], sv[3], so[3], each (t, h, d).
 *   cu_seqlens: DEVICE int32 [num_seqs + 1]; sequence s owns tokens
 *            cu_seqlens[s] .. cu_seqlens[s+1]-1 and its logical positions
 *            are 0 .. L_s-1.  It must be non-decreasing from 0 to T with
 *            every L_s <= max_seqlen.
 *   cu_seqlens_host: optional HOST mirror of cu_seqlens (may be NULL).  When
 *            given it is validated before launch (ETATTN_ERR_BAD_SEQLENS);
 *            otherwise the kernel checks each sequence it reads and, on a bad
 *            entry, skips that sequence and records ETATTN_ERR_BAD_SEQLENS in
 *            the device status word (see etattn_read_device_status).
 */
int attn_fwd_varlen(const void* q, const void* k, const void* v, void* o, float* lse, const int32_t* cu_seqlens,
                    const int32_t* cu_seqlens_host, int num_seqs, int max_seqlen, int total_tokens, int Hq,
                    int Hkv, int D, int dtype, const int64_t* strides, int causal, float scale, void* stream);

/*
 * attn_fwd_ex: attn_fwd with Nq query and Nk key tokens per sequence and an
 * optional local window (eligibility rule at the top of this file).
 *
 *   q, o: logical [B, Hq, Nq, D];  k, v: logical [B, Hkv, Nk, D];
 *   lse : [B, Hq, Nq] contiguous FP32 (or NULL);  strides as for attn_fwd.
 *   window_left, window_right: key offsets before / after the row's key
 *           position; a negative value is no bound.  With causal = 1 the
 *           right bound is the diagonal whatever window_right says.
 * Nq = 0 (or B or Hq = 0) is a no-op.  Nk = 0 is valid: every row is empty
 * and k, v may be NULL.  attn_fwd(..., N, ...) equals
 * attn_fwd_ex(..., Nq = N, Nk = N, ..., window_left = -1, window_right = -1, ...).
 */
int attn_fwd_ex(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv, int Nq,
                int Nk, int D, int dtype, const int64_t* strides, int causal, int window_left, int window_right,
                float scale, void* stream);

/*
 * attn_fwd_splitkv: attn_fwd_ex with the keys cut into num_splits slices that
 * run as separate CTAs, for few query rows over many keys (a decode step).
 * "Intermediate and advanced extension", workshop row "Split softmax" and
 * "Logic review before implementation": a first launch writes every row's
 * partial state per slice (O_s = acc_s / l_s and lse_s = scale*m_s + ln l_s,
 * FP32), a second launch on the same stream merges the slices (rescaling the
 * partial sums to the common maximum) and normalises; no cross-block wait.
 * The result is the same operation as attn_fwd_ex up to rounding order.
 *
 *   q, k, v, o, lse, strides, causal, windows, scale: as for attn_fwd_ex.
 *   num_splits: 1 .. 1024 key slices of ceil(ceil(Nk/128) / num_splits)
 *           128-key tiles each (attn_fwd_splitkv_plan suggests one).  With
 *           num_splits = 1 (or Nk = 0) the call is attn_fwd_ex and the
 *           workspace is not used (it may be NULL).
 *   workspace: caller-owned DEVICE scratch, 256-byte aligned, of at least
 *           attn_fwd_splitkv_workspace_size(B, Hq, Nq, D, num_splits)
 *           bytes, private to this call until the merge launch completes on
 *           `stream` (two calls in flight must not share one).  It may hold
 *           anything on entry: every slice writes every row before the merge
 *           reads it.  It must not overlap q, k, v, o or lse
 *           (ETATTN_ERR_ALIAS); too small or num_splits out of range is
 *           ETATTN_ERR_BAD_SHAPE; misaligned is ETATTN_ERR_BAD_ALIGN.
 */
int attn_fwd_splitkv(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv,
                     int Nq, int Nk, int D, int dtype, const int64_t* strides, int causal, int window_left,
                     int window_right, float scale, int num_splits, void* workspace, size_t workspace_bytes,
                     void* stream);

/* Bytes of workspace attn_fwd_splitkv needs (0 when num_splits <= 1, or for
 * invalid sizes): num_splits * B*Hq*Nq * (4*D + 4) plus alignment padding. */
size_t attn_fwd_splitkv_workspace_size(int B, int Hq, int Nq, int D, int num_splits);

/*
 * attn_fwd_global: attn_fwd_ex plus num_global global tokens
 * ("Attention algorithms and data movement", lesson 07, global-token
 * unions).  The first num_global key positions are global: every row may
 * also read the global keys j < num_global, and a global row (key position
 * c < num_global) may read every key; both still obey the causal mask and
 * ignore the window.  Row i's eligible keys are the union of its window and
 * those connections, each key counted once.  One launch streams, for every
 * query tile, the global keys' tiles and then the rest of its rows' keys.
 *
 *   q, k, v, o, lse, strides, causal, windows, scale: as for attn_fwd_ex.
 *   num_global: >= 0.  With 0, or when the window already holds every key
 *           the causal mask allows (no left bound, and causal or no right
 *           bound), the call is attn_fwd_ex.
 * Returns the codes of attn_fwd_ex; num_global < 0 is ETATTN_ERR_BAD_SHAPE.
 */
int attn_fwd_global(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv,
                    int Nq, int Nk, int D, int dtype, const int64_t* strides, int causal, int window_left,
                    int window_right, int num_global, float scale, void* stream);

/*
 * attn_fwd_varlen_splitkv: attn_fwd_varlen_ex with the keys of every
 * sequence cut into num_splits slices (as attn_fwd_splitkv does for the
 * batched layout), for packed batches of few query rows over long keys.
 * Slice s of a sequence holds its key tiles s*m .. s*m + m - 1 with
 * m = ceil(ceil(max_seqlen_k / 128) / num_splits).
 *
 *   arguments as for attn_fwd_varlen_ex, plus num_splits, workspace and
 *   workspace_bytes as for attn_fwd_splitkv; the workspace holds
 *   attn_fwd_varlen_splitkv_workspace_size(total_q, Hq, D, num_splits) bytes
 *   (one partial row per slice, query head and query token).
 */
int attn_fwd_varlen_splitkv(const void* q, const void* k, const void* v, void* o, float* lse,
                            const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k, const int32_t* cu_seqlens_q_host,
                            const int32_t* cu_seqlens_k_host, int num_seqs, int max_seqlen_q, int max_seqlen_k,
                            int total_q, int total_k, int Hq, int Hkv, int D, int dtype, const int64_t* strides,
                            int causal, int window_left, int window_right, float scale, int num_splits,
                            void* workspace, size_t workspace_bytes, void* stream);

/* Bytes of workspace attn_fwd_varlen_splitkv needs (0 when num_splits <= 1 or
 * for invalid sizes): num_splits * total_q*Hq * (4*D + 4) plus padding. */
size_t attn_fwd_varlen_splitkv_workspace_size(int total_q, int Hq, int D, int num_splits);

/* A split count for attn_fwd_varlen_splitkv: attn_fwd_splitkv_plan for a
 * batch of num_seqs sequences of max_seqlen_q queries over max_seqlen_k keys
 * (the launch's grid covers every sequence at the longest lengths).  Same
 * return codes as attn_fwd_splitkv_plan. */
int attn_fwd_varlen_splitkv_plan(int num_seqs, int Hq, int Hkv, int max_seqlen_q, int max_seqlen_k,
                                 int* num_splits);

/*
 * attn_fwd_varlen_global: attn_fwd_varlen_ex plus num_global global tokens
 * per sequence (the first num_global positions of each sequence), with the
 * rule of attn_fwd_global; with num_global = 0, or a window that already
 * holds every key the causal mask allows, the call is attn_fwd_varlen_ex.
 */
int attn_fwd_varlen_global(const void* q, const void* k, const void* v, void* o, float* lse,
                           const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k, const int32_t* cu_seqlens_q_host,
                           const int32_t* cu_seqlens_k_host, int num_seqs, int max_seqlen_q, int max_seqlen_k,
                           int total_q, int total_k, int Hq, int Hkv, int D, int dtype, const int64_t* strides,
                           int causal, int window_left, int window_right, int num_global, float scale, void* stream);

/* A split count for attn_fwd_splitkv on the current device: enough CTAs for
 * about four per SM when the query tiles alone do not fill the GPU, each
 * slice at least four key tiles; 1 when splitting would not help.  (Fewer
 * than 128 query tokens of a grouped-query problem share a 128-row tile
 * among up to Hq/Hkv query heads, so Hkv enters the count.)  Returns
 * ETATTN_OK, ETATTN_ERR_NULL_PTR, ETATTN_ERR_BAD_SHAPE, ETATTN_ERR_BAD_HEADS
 * or ETATTN_ERR_NO_DEVICE. */
int attn_fwd_splitkv_plan(int B, int Hq, int Hkv, int Nq, int Nk, int* num_splits);

/*
 * attn_fwd_splitkv_noalloc: attn_fwd_splitkv without a workspace argument,
 * for callers that cannot allocate device memory at call time (a runtime
 * whose device memory all belongs to its own pool with no allocation hook for
 * this call, or a plugin handed only the step's tensors).  The pages have no
 * counterpart of this entry point.
 *
 * The partial states go to one scratch buffer of 16 MiB that the library
 * owns for each device (a statically sized device array; no allocation at any
 * call).  A problem whose attn_fwd_splitkv_workspace_size(B, Hq, Nq, D,
 * num_splits) exceeds 16 MiB is refused with ETATTN_ERR_BAD_SHAPE before any
 * device work; num_splits = 1 (or Nk = 0) needs no scratch.  Nothing in the
 * scratch has to start at zero.  Because the buffer is shared, two calls on
 * one device must not overlap in time: calls on one stream are ordered, but
 * calls on different streams, or from different host threads, without an
 * ordering between them race on the scratch and may return wrong results.
 * The first call on each device looks up the buffer's address (a CUDA
 * runtime query) and sets kernel attributes; make that first call before any
 * stream capture begins.  Other arguments, results and errors are those of
 * attn_fwd_splitkv.
 */
int attn_fwd_splitkv_noalloc(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq,
                             int Hkv, int Nq, int Nk, int D, int dtype, const int64_t* strides, int causal,
                             int window_left, int window_right, float scale, int num_splits, void* stream);

/*
 * attn_bwd: gradients of the attention of attn_fwd_ex ("Attention algorithms
 * and data movement", lesson 03: recompute the probabilities and
 * differentiate the normalised row from the saved normalisation state).
 * Given the forward's inputs, its output O, its logsumexp and the upstream
 * gradient dO, it writes
 *     dQ = scale * dS K,   dK = scale * dS^T Q,   dV = P^T dO,
 * with P_ij = exp(scale*<q_i,k_j> - lse_i) on eligible pairs (0 elsewhere),
 * dS = P * (dO V^T - D) and D_i = <dO_i, O_i>.  Under grouped-query attention
 * dK and dV of a key/value head sum over the query heads that read it.
 *
 *   q, o, dout, dq: logical [B, Hq, Nq, D];  k, v, dk, dv: [B, Hkv, Nk, D]
 *   lse : [B, Hq, Nq] contiguous FP32, as attn_fwd / attn_fwd_ex wrote it
 *         (natural log of the scaled logits; -inf on rows that read no key)
 *   strides: 32 int64 values, (b, h, n, d) for q, k, v, o, dout, dq, dk, dv
 *         in that order; d-strides 1, the others as for attn_fwd.
 *   causal, window_left, window_right, scale: as for the forward call.
 *   workspace: caller-owned DEVICE scratch, 256-byte aligned, at least
 *         attn_bwd_workspace_size(B, Hq, Nq, D) bytes (FP32 dQ plus two FP32
 *         values per query row), private to the call until its last launch
 *         has run on `stream`; its contents on entry do not matter.
 * Inputs (q, k, v, o, lse, dout) are only read.  dq, dk, dv must not overlap
 * an input, the workspace or each other (ETATTN_ERR_ALIAS).  Nq = 0 gives dk =
 * dv = 0 (q, o, lse, dout, dq may be NULL); Nk = 0 gives dq = 0 (k, v, dk, dv
 * may be NULL).  The call enqueues three kernels (row statistics, the
 * gradients, dQ conversion) and returns; errors as for attn_fwd.
 */
int attn_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dout, void* dq,
             void* dk, void* dv, int B, int Hq, int Hkv, int Nq, int Nk, int D, int dtype, const int64_t* strides,
             int causal, int window_left, int window_right, float scale, void* workspace, size_t workspace_bytes,
             void* stream);

/* Workspace bytes attn_bwd needs (0 for empty or invalid sizes). */
size_t attn_bwd_workspace_size(int B, int Hq, int Nq, int D);

/*
 * attn_fwd_varlen_ex: attn_fwd_varlen with separate packed query and key
 * offsets and an optional local window.
 *
 *   q, o: logical [total_q, Hq, D];  k, v: logical [total_k, Hkv, D];
 *   lse : [Hq, total_q] contiguous FP32 (or NULL);  strides as for
 *         attn_fwd_varlen (12 values, (t, h, d) for q, k, v, o).
 *   cu_seqlens_q / cu_seqlens_k: DEVICE int32 [num_seqs + 1]; sequence s
 *         owns query tokens cu_seqlens_q[s] .. cu_seqlens_q[s+1]-1 and key
 *         tokens cu_seqlens_k[s] .. cu_seqlens_k[s+1]-1 (both required; they
 *         may be the same array).  Each must rise from 0 to its total with
 *         every length <= max_seqlen_q / max_seqlen_k.
 *   cu_seqlens_q_host / cu_seqlens_k_host: optional HOST mirrors, each
 *         validated before launch when given (ETATTN_ERR_BAD_SEQLENS);
 *         otherwise the kernel checks each sequence as attn_fwd_varlen does.
 * A sequence with no keys gives O = 0 and lse = -inf on its rows; with
 * total_k = 0, k and v may be NULL.
 */
int attn_fwd_varlen_ex(const void* q, const void* k, const void* v, void* o, float* lse,
                       const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k, const int32_t* cu_seqlens_q_host,
                       const int32_t* cu_seqlens_k_host, int num_seqs, int max_seqlen_q, int max_seqlen_k,
                       int total_q, int total_k, int Hq, int Hkv, int D, int dtype, const int64_t* strides, int causal,
                       int window_left, int window_right, float scale, void* stream);

/*
 * attn_fwd_host: attn_fwd for callers whose q, k, v live in HOST memory and
 * who want O (and lse) back in host memory, all in one call.
 *
 *   *_host: HOST buffers, contiguous [B,H,N,D] (q, o: H = Hq; k, v: H = Hkv)
 *           and lse_host [B,Hq,N] FP32 (or NULL).  Pinned (page-locked)
 *           memory lets the copies run asynchronously; pageable memory works
 *           but the copies then block the calling thread.
 *   *_dev : caller-owned DEVICE buffers of the same sizes and layouts; the
 *           inputs are staged there and the outputs computed there.  lse_dev
 *           must be NULL exactly when lse_host is NULL.
 * The call cuts the problem into up to 8 chunks (runs of whole batches; with
 * B = 1, runs of KV heads with their query heads) and pipelines them: chunk
 * c + 1's inputs are copied to the device while chunk c's kernel runs, and
 * chunk c's outputs are copied back meanwhile.  The kernels run on `stream`;
 * the copies run on two copy streams of the library's own (one per device,
 * created on first use and kept), which first wait for the work already on
 * `stream`, and `stream` waits for the last copy before anything enqueued
 * after the call.  So, seen from `stream`, the call is ordered like one
 * operation: synchronise `stream` before reading o_host / lse_host, and do
 * not change q_host / k_host / v_host before then.  It returns once all of
 * it is enqueued.  Arguments are validated (as for attn_fwd, on the device
 * buffers) before anything is enqueued.  Each chunk computes its rows as
 * the whole call would.  Nothing is allocated on the device.
 */
int attn_fwd_host(const void* q_host, const void* k_host, const void* v_host, void* o_host, float* lse_host,
                  void* q_dev, void* k_dev, void* v_dev, void* o_dev, float* lse_dev, int B, int Hq, int Hkv, int N,
                  int D, int dtype, int causal, float scale, void* stream);

/*
 * attn_fwd_varlen_host: attn_fwd_varlen with host buffers, as attn_fwd_host.
 *   q/k/v/o host and device buffers: contiguous [T,H,D]; lse [Hq,T] FP32 or NULL.
 *   cu_seqlens_host (required) is validated on the host and copied to the
 *   caller-owned device buffer cu_seqlens_dev (int32 [num_seqs+1]).
 * The chunks are the runs of whole sequences that attn_fwd_varlen_host_plan
 * returns for max_chunks = 8 (about equal token counts): a chunk's tokens are
 * contiguous rows of q/k/v/o and one column band of lse.  The run with the
 * fewest tokens is processed first and, of the others, the one whose lengths
 * have the smallest sum of squares last; the rest in order.
 */
int attn_fwd_varlen_host(const void* q_host, const void* k_host, const void* v_host, void* o_host, float* lse_host,
                         const int32_t* cu_seqlens_host, void* q_dev, void* k_dev, void* v_dev, void* o_dev,
                         float* lse_dev, int32_t* cu_seqlens_dev, int num_seqs, int max_seqlen, int total_tokens,
                         int Hq, int Hkv, int D, int dtype, int causal, float scale, void* stream);

/*
 * attn_fwd_varlen_host_plan: the chunks attn_fwd_varlen_host pipelines.
 * Host-only (no device call).  Cuts the num_seqs sequences of the HOST
 * offsets cu_seqlens_host[0..num_seqs] into k <= min(max_chunks, 8, num_seqs)
 * runs of consecutive sequences of about equal token counts: a run ends after
 * the first sequence whose cumulative token count reaches the next multiple
 * of total / k_max (the last run takes the rest).  seq_bounds (caller-owned,
 * int32 [k + 1], so 9 entries suffice) receives 0 = b_0 < b_1 < ... < b_k =
 * num_seqs; run c holds sequences b_c .. b_(c+1) - 1.  Returns k (0 when
 * num_seqs == 0), or a negative status: -ETATTN_ERR_NULL_PTR,
 * -ETATTN_ERR_BAD_SHAPE (num_seqs < 0 or max_chunks < 1),
 * -ETATTN_ERR_BAD_SEQLENS (offsets that decrease).
 */
int attn_fwd_varlen_host_plan(const int32_t* cu_seqlens_host, int num_seqs, int max_chunks, int32_t* seq_bounds);

/* Human-readable name of a status code (static storage, never NULL). */
const char* etattn_status_string(int code);

/* The cudaError_t value of the last ETATTN_ERR_LAUNCH on this thread (0 if none). */
int etattn_last_cuda_error(void);

/*
 * Read the device status word of the current device that kernels set on a
 * failure they detect themselves (a bounded wait that ran out, or a bad
 * cu_seqlens entry).  Synchronises `stream`.  *out receives ETATTN_OK or the
 * ETATTN_ERR_* code; when clear != 0 the word is reset to 0 afterwards.
 * Returns ETATTN_OK or ETATTN_ERR_LAUNCH.
 */
int etattn_read_device_status(int* out, int clear, void* stream);

/*
 * Self-test of the kernels' failure detection ("Intermediate and advanced
 * extension", "Logic review before implementation": ordered launches, no
 * spin barrier that could wait forever).  Every wait of the attention
 * kernels' pipelines is bounded; this call checks that path on the device
 * without disturbing a real launch.  It enqueues on `stream` one tiny kernel
 * in which one thread waits, through the same bounded mbarrier wait as the
 * pipelines but with a limit of limit_us microseconds, on a barrier that
 * nothing arrives at.  The wait runs out and records a timeout in the device
 * status word, so a following etattn_read_device_status reports
 * ETATTN_ERR_DEVICE (and clears it when asked).  The kernel holds no tensor
 * memory and starts no copy or MMA.  limit_us must lie in [1, 1000000].
 * Returns ETATTN_OK, ETATTN_ERR_BAD_SHAPE (limit out of range),
 * ETATTN_ERR_NO_DEVICE or ETATTN_ERR_LAUNCH.
 */
int etattn_selftest_wait_timeout(int limit_us, void* stream);

/* Library version as MAJOR*10000 + MINOR*100 + PATCH. */
int etattn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* ETATTN_H */

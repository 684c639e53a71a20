// Host side of the C ABI declared in etattn.h: argument validation (all of it
// before any CUDA call), TMA tensor-map encoding and kernel launch.
//
// The validation contract follows "Intermediate and advanced extension",
// "Code review and execution gates": shapes, layouts, dtypes, index spans and
// launch knobs are checked before a kernel is invoked, inputs are read-only
// and outputs are separate allocations.
#include <algorithm>
#include <atomic>
#include <climits>
#include <cmath>
#include <cstdint>
#include <mutex>
#include <vector>

#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include "attn_bwd_kernel.cuh"
#include "attn_fwd_kernel.cuh"
#include "etattn.h"
#include "launchers.h"

namespace etattn {

// Device status word shared by every launch on a device (0 = ok).
__device__ int g_status_word;

// Split-KV scratch of attn_fwd_splitkv_noalloc: a fixed, module-owned buffer
// for callers that cannot hand over device memory (see that entry point).
// Its size bounds the problems it accepts.  Nothing in it has to start at
// zero: every key slice writes every row's partial state before the merge
// launch reads it.
constexpr size_t kNoAllocScratchBytes = size_t(16) << 20;
static __device__ __align__(256) unsigned char g_splitkv_scratch[kNoAllocScratchBytes];

// Self-test of the bounded waits: one thread waits, with the given limit, on
// an mbarrier that nothing arrives at, through the same mbar_wait every
// pipeline role uses.  The wait runs out and records kDevWaitTimeout in the
// status word.  The kernel holds no tensor memory and starts no copy or MMA,
// so its early return leaves nothing in flight.
__global__ void wait_selftest_kernel(unsigned long long limit_ns, int* status) {
  __shared__ uint64_t bar;
  if (threadIdx.x != 0) return;
  mbar_init(&bar, 1);
  fence_mbar_init();
  (void)mbar_wait(&bar, 0, status, limit_ns);
}

namespace {

constexpr int kMaxTokens = 1 << 30;      // token coordinates stay well inside int32
constexpr int kMaxGridYZ = 65535;         // heads and batch/sequences map to grid y and z
thread_local int t_last_cuda_error = 0;

int fail_cuda(cudaError_t e) {
  t_last_cuda_error = (int)e;
  return ETATTN_ERR_LAUNCH;
}

// ---------------------------------------------------------------- validation helpers
struct View {         // a strided tensor of rank <= 4, sizes and strides in elements
  const void* ptr;
  int rank;
  int64_t size[4];
  int64_t stride[4];
};

// Byte span [lo, hi) touched by a view (hi == lo when it is empty).
void span_of(const View& v, size_t esz, uintptr_t* lo, uintptr_t* hi) {
  *lo = reinterpret_cast<uintptr_t>(v.ptr);
  uint64_t last = 0;
  for (int i = 0; i < v.rank; ++i) {
    if (v.size[i] == 0) {
      *hi = *lo;
      return;
    }
    last += (uint64_t)(v.size[i] - 1) * (uint64_t)v.stride[i];
  }
  *hi = *lo + (last + 1) * esz;
}

bool overlaps(const View& a, size_t ea, const View& b, size_t eb) {
  uintptr_t alo, ahi, blo, bhi;
  span_of(a, ea, &alo, &ahi);
  span_of(b, eb, &blo, &bhi);
  if (alo == ahi || blo == bhi) return false;
  return alo < bhi && blo < ahi;
}

// d-stride 1; every other stride of an extent > 1 positive and a multiple of
// 16 bytes.  A view with an extent of 0 addresses nothing and passes.
bool strides_ok(const View& v, size_t esz) {
  for (int i = 0; i < v.rank; ++i)
    if (v.size[i] == 0) return true;
  if (v.stride[v.rank - 1] != 1) return false;
  for (int i = 0; i < v.rank - 1; ++i) {
    if (v.size[i] <= 1) continue;
    if (v.stride[i] <= 0) return false;
    if (((uint64_t)v.stride[i] * esz) % 16 != 0) return false;
    if ((uint64_t)v.stride[i] * esz >= (1ull << 40)) return false;
  }
  return true;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// ---------------------------------------------------------------- device / driver plumbing
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  return g_encode;
}

struct DeviceInfo {
  std::atomic<int> state{0};  // 0 unknown, 1 ok, 2 unsupported
  int* status_word = nullptr;
  int num_sms = 0;
};
DeviceInfo g_devices[64];
std::mutex g_device_mu;

// Current device, checked to be sm_103, with its status-word address.
int current_device(int* dev_out, int** status_out, int* num_sms_out = nullptr) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || dev < 0 || dev >= 64) {
    cudaGetLastError();
    return ETATTN_ERR_NO_DEVICE;
  }
  DeviceInfo& d = g_devices[dev];
  if (d.state.load(std::memory_order_acquire) == 0) {
    std::lock_guard<std::mutex> lk(g_device_mu);
    if (d.state.load() == 0) {
      int major = 0, minor = 0;
      if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
          cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) {
        cudaGetLastError();
        return ETATTN_ERR_NO_DEVICE;
      }
      if (major != 10 || minor != 3) {
        d.state.store(2);
      } else {
        if (cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
          cudaGetLastError();
          return ETATTN_ERR_NO_DEVICE;
        }
        void* sym = nullptr;
        cudaError_t se = cudaGetSymbolAddress(&sym, g_status_word);
        if (se != cudaSuccess) return fail_cuda(se);
        d.status_word = static_cast<int*>(sym);
        d.state.store(1, std::memory_order_release);
      }
    }
  }
  if (d.state.load() != 1) return ETATTN_ERR_NO_DEVICE;
  *dev_out = dev;
  *status_out = d.status_word;
  if (num_sms_out) *num_sms_out = d.num_sms;
  return ETATTN_OK;
}

// 4-D tensor map over (d, token, head, batch) with a box of one 128-row tile
// of SW elements along d: 128 tokens of one head, or with box_heads = P > 1,
// 128 / P tokens of P heads.  If the token stride exceeds the head stride
// the two middle axes are exchanged so that strides grow outward; *swapped
// says so.
int encode_map(CUtensorMap* map, int dtype, const void* ptr, int D, int64_t n_tokens, int64_t n_heads,
               int64_t n_batch, int64_t s_tok, int64_t s_head, int64_t s_batch, bool* swapped, int box_heads = 1) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
  if (!enc) return fail_cuda(cudaErrorNotSupported);
  const uint64_t esz = 2;
  const int sw_elems = D >= 64 ? 64 : 32;
  // Strides of extent-1 axes are never used; give them a harmless value.
  uint64_t reach = 16;
  if (n_tokens > 1) reach = std::max<uint64_t>(reach, (uint64_t)s_tok * esz * (uint64_t)n_tokens);
  if (n_heads > 1) reach = std::max<uint64_t>(reach, (uint64_t)s_head * esz * (uint64_t)n_heads);
  if (n_batch > 1) reach = std::max<uint64_t>(reach, (uint64_t)s_batch * esz * (uint64_t)n_batch);
  reach = (reach + 15) & ~uint64_t(15);
  const uint64_t bt = n_tokens > 1 ? (uint64_t)s_tok * esz : reach;
  const uint64_t bh = n_heads > 1 ? (uint64_t)s_head * esz : reach;
  const uint64_t bb = n_batch > 1 ? (uint64_t)s_batch * esz : reach;
  const bool sw = n_tokens > 1 && n_heads > 1 && bt > bh;
  cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)(sw ? n_heads : n_tokens), (cuuint64_t)(sw ? n_tokens : n_heads),
                        (cuuint64_t)n_batch};
  cuuint64_t strides[3] = {sw ? bh : bt, sw ? bt : bh, bb};
  const cuuint32_t box_tok = 128u / (cuuint32_t)box_heads, box_head = (cuuint32_t)box_heads;
  cuuint32_t box[4] = {(cuuint32_t)sw_elems, sw ? box_head : box_tok, sw ? box_tok : box_head, 1u};
  cuuint32_t estride[4] = {1, 1, 1, 1};
  CUresult r = enc(map, dtype == ETATTN_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 4,
                   const_cast<void*>(ptr), dims, strides, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   D >= 64 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail_cuda(cudaErrorInvalidValue);
  *swapped = sw;
  return ETATTN_OK;
}

// (m, k) with floor(n / d) = (n * m) >> k for every n < 2^31 (the kernel's
// div_magic): l = ceil(log2 d), k = 31 + l, m = ceil(2^k / d) < 2^32.
void div_magic_of(uint32_t d, uint32_t* m, uint32_t* k) {
  uint32_t l = 0;
  while ((1ull << l) < d) ++l;
  *k = 31 + l;
  *m = (uint32_t)(((1ull << *k) + d - 1) / d);
}

// Keys read by the query row at key position c of a sequence with Lk keys
// (the kernel's row_key_range, both parts): the window [c - wl, c + wr]
// clipped to the keys; with G global tokens also the global keys [0, G) and,
// for a global row (c < G), every key up to its causal limit (c + wrc).
int64_t keys_of_row(int64_t c, int64_t Lk, int64_t wl, int64_t wr, int64_t wrc, int64_t G) {
  const int64_t lo = std::max<int64_t>(0, c - wl), hi = std::min<int64_t>(Lk - 1, c + wr);
  if (G <= 0) return std::max<int64_t>(0, hi - lo + 1);
  const int64_t h = std::min<int64_t>(Lk - 1, c + wrc);
  const int64_t glob = std::max<int64_t>(0, std::min<int64_t>(G - 1, h) + 1);
  const int64_t rest = c < G ? std::max<int64_t>(0, h - G + 1) : std::max<int64_t>(0, hi - std::max(lo, G) + 1);
  return glob + rest;
}

// Whether some query row of a sequence (Lq queries over Lk keys, bottom-right
// aligned: row r at key position r + Lk - Lq) reads at least one and fewer
// than kFewKeys keys, so that the kernel's split-P path may run.  The count is
// piecewise linear in r, its pieces meeting where one clip of row_key_range
// starts or stops binding; the smallest non-zero count is at the end of a
// piece, so the first and last rows and the rows next to every breakpoint
// decide it.
bool has_few_key_rows(int64_t Lq, int64_t Lk, int64_t wl, int64_t wr, int64_t wrc, int64_t G) {
  if (Lq <= 0 || Lk <= 0) return false;
  const int64_t delta = Lk - Lq;
  const int64_t cs[] = {0, wl, Lk - 1 - wr, Lk - 1 + wl, -wr, G - 1, G, G + wl, Lk - 1 - wrc, Lk - 1, G - wr};
  std::vector<int64_t> rows = {0, Lq - 1};
  for (int64_t c : cs)
    for (int64_t d = -1; d <= 1; ++d) rows.push_back(c + d - delta);
  for (int64_t r : rows) {
    if (r < 0 || r >= Lq) continue;
    const int64_t n = keys_of_row(r + delta, Lk, wl, wr, wrc, G);
    if (n > 0 && n < kFewKeys) return true;
  }
  return false;
}

// Launch over `tokens` query rows per (head, batch/sequence).  Two 128-row
// sub-tiles per CTA keep the tensor core busier, but halve the CTA count; a
// problem that would not fill the GPU with two-sub-tile CTAs runs one
// sub-tile per CTA instead.  `general` selects the kernel built for unequal
// query/key lengths and windows; square window-free calls take the other.
//
// In a split-KV launch (p.part_o set) every query block gets p.num_splits
// CTAs, one per key slice.
//
// With grouped-query packing (p.qpack = P > 1) `tokens` counts rows (query
// tokens x P) and gy head packs; such launches use one sub-tile per CTA.
//
// A problem whose 128-row blocks fill at most half the SMs and whose rows
// read more than one key tile (`key_tiles`, the most any row block streams)
// runs the key-split build instead: one row block per CTA, its two
// sub-tiles taking alternate key tiles.
cudaError_t launch(int D, int dtype, const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                   const FwdParams& p, int64_t tokens, unsigned gy, unsigned gz, int num_sms, bool general,
                   bool few_keys, cudaStream_t s, int64_t key_tiles = 0, int ks_force = -1) {
  const bool bf = dtype == ETATTN_BF16;
  const int64_t splits = p.part_o != nullptr ? p.num_splits : 1;
  const int64_t blocks1 = (tokens + 127) / 128, blocks2 = (tokens + 255) / 256;
  // The key split halves every CTA's key range and doubles the CTAs: for
  // problems that would not fill half the SMs, and for general (unequal-
  // length) problems of at least 16 key tiles whose equal CTAs would leave the
  // last wave partly empty: c CTAs take ceil(c / SMs) waves of one length, 2c
  // key-split CTAs ceil(2c / SMs) waves of half of it (taken when that is at
  // least 5 % shorter).  ks_force >= 0: a chunk of a larger call takes the
  // whole call's choice (the split changes the order of the sum over key
  // tiles).
  const int64_t ctas2 = blocks2 * (int64_t)gy * gz, ctas1 = blocks1 * (int64_t)gy * gz;
  const bool ks_waves = general && key_tiles >= 16 && ctas2 > num_sms &&
                        ((ctas1 + num_sms - 1) / num_sms) * 100 < ((ctas2 + num_sms - 1) / num_sms) * 2 * 95;
  const bool ksplit = splits == 1 && p.qpack == 1 && p.num_global == 0 && key_tiles >= 2 &&
                      (ks_force >= 0 ? ks_force == 1 : (2 * ctas1 <= num_sms || ks_waves));
  // Up to 128 query rows fill one sub-tile: a second one would only idle.
  const int nsub = (p.qpack > 1 || tokens <= 128 || blocks2 * (int64_t)gy * gz * splits < num_sms) ? 1 : 2;
  const int64_t gx = (ksplit || nsub == 1 ? blocks1 : blocks2) * splits;
  if (gx > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  FwdParams pp = p;
  pp.grid_x = (int)gx;
  pp.grid_y = (int)gy;
  pp.grid_z = (int)gz;
  // Grouped longest-first dispatch (the kernel's cta_coords): groups of G
  // (head, batch) pairs, G the smallest power of two whose CTAs fill the SMs
  // once, so that the last group alone still spreads its shortest blocks over
  // the GPU.  A grid too large for one dimension keeps the plain 3-D order.
  // A grid that fits in one wave starts all at once: it keeps the 3-D order.
  dim3 g((unsigned)gx, gy, gz);
  pp.sched_q = pp.sched_rem = 0;
  const int64_t pairs = (int64_t)gy * gz;
  if (gx * pairs > num_sms && gx * pairs <= 0x7fffffffLL) {
    int64_t G = 1;
    while (G * gx < num_sms && G < pairs) G *= 2;
    const int64_t groups = (pairs + G - 1) / G;  // near-equal groups: pairs / groups, the first pairs % groups one more
    pp.sched_q = (int)(pairs / groups);
    pp.sched_rem = (int)(pairs % groups);
    const uint32_t divisors[4] = {(uint32_t)gx, (uint32_t)pp.sched_q + 1, (uint32_t)pp.sched_q, gy};
    for (int i = 0; i < 4; ++i) div_magic_of(divisors[i], &pp.div_m[i], &pp.div_k[i]);
    g = dim3((unsigned)(gx * pairs), 1, 1);
  }
  switch (D) {
    case 32:
      return bf ? launch_fwd_d32_1(q, k, v, pp, g, nsub, general, ksplit, few_keys, s)
                : launch_fwd_d32_0(q, k, v, pp, g, nsub, general, ksplit, few_keys, s);
    case 64:
      return bf ? launch_fwd_d64_1(q, k, v, pp, g, nsub, general, ksplit, few_keys, s)
                : launch_fwd_d64_0(q, k, v, pp, g, nsub, general, ksplit, few_keys, s);
    default:
      return bf ? launch_fwd_d128_1(q, k, v, pp, g, nsub, general, ksplit, few_keys, s)
                : launch_fwd_d128_0(q, k, v, pp, g, nsub, general, ksplit, few_keys, s);
  }
}

bool head_dim_ok(int D) { return D == 32 || D == 64 || D == 128; }

// 3-D FP32 map over the backward's dQ buffer [rows_bh = B * Hq][Nq][D] for
// TMA reduce-adds of (32 columns x 32 rows) boxes, 128-byte swizzled; rows
// past Nq of a (batch, head) fall outside the map.
int encode_dq_map(CUtensorMap* map, float* dq_acc, int D, int64_t Nq, int64_t rows_bh) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
  if (!enc) return fail_cuda(cudaErrorNotSupported);
  cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)Nq, (cuuint64_t)rows_bh};
  cuuint64_t strides[2] = {(cuuint64_t)D * 4, (cuuint64_t)Nq * D * 4};
  cuuint32_t box[3] = {32u, 32u, 1u};
  cuuint32_t estride[3] = {1, 1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, dq_acc, dims, strides, box, estride,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail_cuda(cudaErrorInvalidValue);
  return ETATTN_OK;
}

constexpr int kMaxSplits = 1024;

// Query heads packed into one 128-row tile: the largest power of two that
// divides the group size, when the general build runs fewer than 128 query
// tokens per sequence (so that a tile would otherwise stay mostly empty).
int qpack_of(bool general, int group, int64_t q_tokens) {
  if (!general || group <= 1 || q_tokens >= 128) return 1;
  int P = 1;
  while (P < 128 && group % (2 * P) == 0) P *= 2;
  return P;
}
constexpr size_t kWorkspaceAlign = 256;

// Split-KV workspace: FP32 partial O (num_splits x rows x D), then, at a
// 256-byte boundary, FP32 partial lse (num_splits x rows).  0 if it would
// not fit in size_t.
size_t splitkv_lse_offset(int64_t rows, int D, int num_splits) {
  const double bytes = (double)num_splits * (double)rows * D * 4.0;
  if (bytes > 1e18) return 0;
  return ((size_t)num_splits * (size_t)rows * (size_t)D * 4 + kWorkspaceAlign - 1) / kWorkspaceAlign *
         kWorkspaceAlign;
}
size_t splitkv_bytes(int64_t rows, int D, int num_splits) {
  if (num_splits <= 1 || rows <= 0) return 0;
  const size_t off = splitkv_lse_offset(rows, D, num_splits);
  if (off == 0) return 0;
  return off + (size_t)num_splits * (size_t)rows * 4;
}

// Key slices for a split-KV call on a GPU of num_sms SMs, given the CTAs of
// one slice (units).  Each slice keeps at least four 128-key tiles.  The
// count minimises a simple time model: the waves of CTAs (one CTA per SM at
// a time) times the tiles of one CTA plus a fixed cost of about two tiles
// (Q load, tensor-memory setup, partial-state write), so that the last wave
// is not left mostly idle.  1 when the query tiles alone fill the GPU.
int plan_splits(int64_t units, int64_t key_tiles, int num_sms) {
  if (units <= 0 || key_tiles < 8 || units >= 2 * (int64_t)num_sms) return 1;
  auto cost = [&](int64_t s, int64_t per) { return ((units * s + num_sms - 1) / num_sms) * (per + 2); };
  int best = 1;
  int64_t best_cost = cost(1, key_tiles);
  const int64_t s_max = std::min<int64_t>(key_tiles / 4, kMaxSplits);
  for (int64_t s = 2; s <= s_max; ++s) {
    const int64_t per = (key_tiles + s - 1) / s;
    if ((key_tiles + per - 1) / per != s) continue;  // the same slices as a smaller count
    const int64_t c = cost(s, per);
    if (c < best_cost) {
      best = (int)s;
      best_cost = c;
    }
  }
  return best;
}

// Split-KV arguments of fwd_impl.
struct SplitArgs {
  int num_splits;
  void* workspace;
  size_t workspace_bytes;
};

// Address of g_splitkv_scratch on the current device, looked up once per
// device (the first call on a device makes this runtime query).
std::atomic<void*> g_scratch_addr[64];
std::mutex g_scratch_mu;

int noalloc_scratch(void** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || dev < 0 || dev >= 64) {
    cudaGetLastError();
    return ETATTN_ERR_NO_DEVICE;
  }
  void* addr = g_scratch_addr[dev].load(std::memory_order_acquire);
  if (addr == nullptr) {
    std::lock_guard<std::mutex> lk(g_scratch_mu);
    addr = g_scratch_addr[dev].load();
    if (addr == nullptr) {
      e = cudaGetSymbolAddress(&addr, g_splitkv_scratch);
      if (e != cudaSuccess || addr == nullptr) return fail_cuda(e != cudaSuccess ? e : cudaErrorInvalidSymbol);
      g_scratch_addr[dev].store(addr, std::memory_order_release);
    }
  }
  *out = addr;
  return ETATTN_OK;
}

}  // namespace
}  // namespace etattn

using namespace etattn;

namespace {

// Effective key-window offsets: negative or huge means no bound; causal
// attention caps the right offset at 0 (the diagonal).
int window_left_of(int wl) { return (wl < 0 || wl > kUnboundedWindow) ? kUnboundedWindow : wl; }
int window_right_of(int wr, int causal) {
  if (causal) return 0;
  return (wr < 0 || wr > kUnboundedWindow) ? kUnboundedWindow : wr;
}

// Validates every argument; launches only when do_launch is set.
int fwd_impl(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv, int Nq,
             int Nk, int D, int dtype, const int64_t* strides, int causal, int window_left, int window_right,
             float scale, void* stream, bool do_launch, const SplitArgs* split = nullptr, int num_global = 0,
             int ks_force = -1) {
  if (dtype != ETATTN_F16 && dtype != ETATTN_BF16) return ETATTN_ERR_BAD_DTYPE;
  if (B < 0 || Hq < 0 || Nq < 0 || Nk < 0 || !head_dim_ok(D)) return ETATTN_ERR_BAD_SHAPE;
  if (Nq > kMaxTokens || Nk > kMaxTokens || B > kMaxGridYZ || Hq > kMaxGridYZ) return ETATTN_ERR_BAD_SHAPE;
  if (Hkv <= 0 || Hq % Hkv != 0) return ETATTN_ERR_BAD_HEADS;
  if (!std::isfinite(scale) || !(scale > 0.f)) return ETATTN_ERR_BAD_SCALE;
  if (strides == nullptr) return ETATTN_ERR_NULL_PTR;
  if (num_global < 0 || (num_global > 0 && split != nullptr)) return ETATTN_ERR_BAD_SHAPE;
  if (B == 0 || Hq == 0 || Nq == 0) return ETATTN_OK;  // empty output: nothing to do
  const bool has_keys = Nk > 0;
  if (!q || !o || (has_keys && (!k || !v))) return ETATTN_ERR_NULL_PTR;

  const View vq{q, 4, {B, Hq, Nq, D}, {strides[0], strides[1], strides[2], strides[3]}};
  const View vk{k, 4, {B, Hkv, Nk, D}, {strides[4], strides[5], strides[6], strides[7]}};
  const View vv{v, 4, {B, Hkv, Nk, D}, {strides[8], strides[9], strides[10], strides[11]}};
  const View vo{o, 4, {B, Hq, Nq, D}, {strides[12], strides[13], strides[14], strides[15]}};
  const View vl{lse, 3, {B, Hq, Nq, 0}, {(int64_t)Hq * Nq, Nq, 1, 0}};
  for (const View* t : {&vq, &vk, &vv, &vo})
    if (!strides_ok(*t, 2)) return ETATTN_ERR_BAD_STRIDE;
  for (const void* ptr : {q, (const void*)o})
    if (!aligned16(ptr)) return ETATTN_ERR_BAD_ALIGN;
  if (has_keys && (!aligned16(k) || !aligned16(v))) return ETATTN_ERR_BAD_ALIGN;
  if (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)) return ETATTN_ERR_BAD_ALIGN;
  for (const View* t : {&vq, &vk, &vv})
    if (overlaps(vo, 2, *t, 2) || (lse && overlaps(vl, 4, *t, 2))) return ETATTN_ERR_ALIAS;
  if (lse && overlaps(vl, 4, vo, 2)) return ETATTN_ERR_ALIAS;
  // Split-KV: slices of the keys, merged by a second launch through the
  // caller's workspace (unused with one slice or no keys).
  const int64_t rows = (int64_t)B * Hq * Nq;
  const bool splitting = split != nullptr && split->num_splits > 1 && has_keys;
  if (split != nullptr && (split->num_splits < 1 || split->num_splits > kMaxSplits)) return ETATTN_ERR_BAD_SHAPE;
  if (splitting) {
    const size_t need = splitkv_bytes(rows, D, split->num_splits);
    if (need == 0) return ETATTN_ERR_BAD_SHAPE;
    if (split->workspace == nullptr) return ETATTN_ERR_NULL_PTR;
    if (reinterpret_cast<uintptr_t>(split->workspace) % kWorkspaceAlign) return ETATTN_ERR_BAD_ALIGN;
    if (split->workspace_bytes < need) return ETATTN_ERR_BAD_SHAPE;
    const View vw{split->workspace, 1, {(int64_t)need, 0, 0, 0}, {1, 0, 0, 0}};
    for (const View* t : {&vq, &vk, &vv, &vo})
      if (overlaps(vw, 1, *t, 2)) return ETATTN_ERR_ALIAS;
    if (lse && overlaps(vw, 1, vl, 4)) return ETATTN_ERR_ALIAS;
  }
  if (!do_launch) return ETATTN_OK;

  int dev = 0;
  int* status = nullptr;
  int num_sms = 0;
  if (int rc = current_device(&dev, &status, &num_sms)) return rc;

  // Equal lengths and no left bound: every row reads key 0, so the square
  // kernel applies whatever the right bound.  A split-KV slice can hold no
  // key of a row: the general build guards that.
  const bool general = Nq != Nk || window_left_of(window_left) != kUnboundedWindow || splitting || num_global > 0;
  const int qpack = qpack_of(general, Hq / Hkv, Nq);

  CUtensorMap mq, mk, mv;
  bool swq = false, swk = false, swv = false;
  if (int rc = encode_map(&mq, dtype, q, D, Nq, Hq, B, strides[2], strides[1], strides[0], &swq, qpack)) return rc;
  if (has_keys) {
    if (int rc = encode_map(&mk, dtype, k, D, Nk, Hkv, B, strides[6], strides[5], strides[4], &swk)) return rc;
    if (int rc = encode_map(&mv, dtype, v, D, Nk, Hkv, B, strides[10], strides[9], strides[8], &swv)) return rc;
  } else {
    // No keys: every row is empty and the kernel loads no K/V tile; the
    // query map stands in for the unused key and value maps.
    mk = mq;
    mv = mq;
    swk = swv = swq;
  }

  FwdParams p{};
  p.o = o;
  p.lse = lse;
  p.o_sb = strides[12];
  p.o_sh = strides[13];
  p.o_sn = strides[14];
  p.lse_sb = (int64_t)Hq * Nq;
  p.lse_sh = Nq;
  p.cu_seqlens_q = p.cu_seqlens_k = nullptr;
  p.Nq = Nq;
  p.Nk = Nk;
  p.total_q = Nq;
  p.total_k = Nk;
  p.max_seqlen_q = Nq;
  p.max_seqlen_k = Nk;
  p.Hq = Hq;
  p.group = Hq / Hkv;
  p.win_left = window_left_of(window_left);
  p.win_right = window_right_of(window_right, causal);
  p.scale = scale;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.status = status;
  p.hn_swapped = (swq ? 1 : 0) | (swk ? 2 : 0) | (swv ? 4 : 0);
  p.qpack = qpack;
  // Global tokens: the global-token build streams each sub-tile's global keys,
  // then the rest of its rows' keys (the kernel's per-row key ranges).
  p.num_global = has_keys ? std::min(num_global, kMaxTokens) : 0;
  p.win_right_causal = causal ? 0 : kUnboundedWindow;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (splitting) {
    const int key_tiles = (Nk + 127) / 128;
    uint8_t* ws = static_cast<uint8_t*>(split->workspace);
    p.part_o = reinterpret_cast<float*>(ws);
    p.part_lse = reinterpret_cast<float*>(ws + splitkv_lse_offset(rows, D, split->num_splits));
    p.part_stride = rows;
    p.num_splits = split->num_splits;
    p.split_tiles = (key_tiles + split->num_splits - 1) / split->num_splits;
  }
  const bool few = dtype == ETATTN_BF16 && has_few_key_rows(Nq, Nk, p.win_left, p.win_right, p.win_right_causal,
                                                            p.num_global);
  cudaError_t e = launch(D, dtype, mq, mk, mv, p, (int64_t)Nq * qpack, (unsigned)(Hq / qpack), (unsigned)B, num_sms,
                         general, few, st, (Nk + 127) / 128, ks_force);
  if (e != cudaSuccess) return fail_cuda(e);
  if (splitting) {
    CombineParams c{};
    c.part_o = p.part_o;
    c.part_lse = p.part_lse;
    c.rows = rows;
    c.num_splits = p.num_splits;
    c.o = o;
    c.lse = lse;
    c.o_sb = strides[12];
    c.o_sh = strides[13];
    c.o_sn = strides[14];
    c.Hq = Hq;
    c.Nq = Nq;
    c.packed = 0;
    c.total = 0;
    e = launch_combine(D, dtype == ETATTN_BF16, c, st);
    if (e != cudaSuccess) return fail_cuda(e);
  }
  return ETATTN_OK;
}

// Backward workspace: FP32 dQ [B, Hq, Nq, D], then at 256-byte boundaries the
// per-row -lse * log2(e) and -scale * <dO, O>, each [B * Hq][Nq_pad].
struct BwdLayout {
  size_t dq_off, lse2_off, dvec_off, total;
};
BwdLayout bwd_layout(int64_t B, int64_t Hq, int64_t Nq, int D) {
  auto up = [](size_t x) { return (x + kWorkspaceAlign - 1) / kWorkspaceAlign * kWorkspaceAlign; };
  const int64_t nq_pad = (Nq + 127) / 128 * 128;
  BwdLayout L{};
  L.dq_off = 0;
  L.lse2_off = up((size_t)(B * Hq * Nq) * D * 4);
  L.dvec_off = L.lse2_off + up((size_t)(B * Hq * nq_pad) * 4);
  L.total = L.dvec_off + up((size_t)(B * Hq * nq_pad) * 4);
  return L;
}

// Backward pass: validation, then three launches on `stream` (row
// statistics, the backward kernel, dQ conversion).
int bwd_impl(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dout, void* dq,
             void* dk, void* dv, int B, int Hq, int Hkv, int Nq, int Nk, int D, int dtype, const int64_t* strides,
             int causal, int window_left, int window_right, float scale, void* workspace, size_t workspace_bytes,
             void* stream) {
  if (dtype != ETATTN_F16 && dtype != ETATTN_BF16) return ETATTN_ERR_BAD_DTYPE;
  if (B < 0 || Hq < 0 || Nq < 0 || Nk < 0 || !head_dim_ok(D)) return ETATTN_ERR_BAD_SHAPE;
  if (Nq > kMaxTokens || Nk > kMaxTokens || B > kMaxGridYZ || Hq > kMaxGridYZ) return ETATTN_ERR_BAD_SHAPE;
  if (Hkv <= 0 || Hq % Hkv != 0) return ETATTN_ERR_BAD_HEADS;
  if (!std::isfinite(scale) || !(scale > 0.f)) return ETATTN_ERR_BAD_SCALE;
  if (strides == nullptr) return ETATTN_ERR_NULL_PTR;
  if (B == 0 || Hq == 0 || (Nq == 0 && Nk == 0)) return ETATTN_OK;
  const bool has_q = Nq > 0, has_k = Nk > 0;
  if (has_q && (!q || !o || !lse || !dout || !dq)) return ETATTN_ERR_NULL_PTR;
  if (has_k && (!k || !v || !dk || !dv)) return ETATTN_ERR_NULL_PTR;
  const int64_t* st = strides;
  auto view = [&](const void* ptr, int idx, int H, int N) {
    return View{ptr, 4, {B, H, N, D}, {st[4 * idx], st[4 * idx + 1], st[4 * idx + 2], st[4 * idx + 3]}};
  };
  const View vq = view(q, 0, Hq, Nq), vk = view(k, 1, Hkv, Nk), vv = view(v, 2, Hkv, Nk), vo = view(o, 3, Hq, Nq);
  const View vdo = view(dout, 4, Hq, Nq), vdq = view(dq, 5, Hq, Nq), vdk = view(dk, 6, Hkv, Nk),
             vdv = view(dv, 7, Hkv, Nk);
  const View vl{lse, 3, {B, Hq, Nq, 0}, {(int64_t)Hq * Nq, Nq, 1, 0}};
  for (const View* t : {&vq, &vk, &vv, &vo, &vdo, &vdq, &vdk, &vdv})
    if (!strides_ok(*t, 2)) return ETATTN_ERR_BAD_STRIDE;
  if (has_q)
    for (const void* ptr : {q, o, dout, (const void*)dq})
      if (!aligned16(ptr)) return ETATTN_ERR_BAD_ALIGN;
  if (has_k)
    for (const void* ptr : {k, v, (const void*)dk, (const void*)dv})
      if (!aligned16(ptr)) return ETATTN_ERR_BAD_ALIGN;
  if (has_q && (reinterpret_cast<uintptr_t>(lse) & 3u)) return ETATTN_ERR_BAD_ALIGN;
  // Outputs overlap no input and no other output.
  const BwdLayout L = bwd_layout(B, Hq, Nq, D);
  const View vw{workspace, 1, {(int64_t)L.total, 0, 0, 0}, {1, 0, 0, 0}};
  for (const View* out : {&vdq, &vdk, &vdv}) {
    for (const View* in : {&vq, &vk, &vv, &vo, &vdo})
      if (overlaps(*out, 2, *in, 2)) return ETATTN_ERR_ALIAS;
    if (has_q && overlaps(*out, 2, vl, 4)) return ETATTN_ERR_ALIAS;
  }
  if (overlaps(vdq, 2, vdk, 2) || overlaps(vdq, 2, vdv, 2) || overlaps(vdk, 2, vdv, 2)) return ETATTN_ERR_ALIAS;
  // Workspace: FP32 dQ and row statistics, private to the call.
  if (has_q) {
    if (workspace == nullptr) return ETATTN_ERR_NULL_PTR;
    if (reinterpret_cast<uintptr_t>(workspace) % kWorkspaceAlign) return ETATTN_ERR_BAD_ALIGN;
    if (workspace_bytes < L.total) return ETATTN_ERR_BAD_SHAPE;
    for (const View* t : {&vq, &vk, &vv, &vo, &vdo, &vdq, &vdk, &vdv})
      if (overlaps(vw, 1, *t, 2)) return ETATTN_ERR_ALIAS;
    if (overlaps(vw, 1, vl, 4)) return ETATTN_ERR_ALIAS;
  }

  int dev = 0;
  int* status = nullptr;
  int num_sms = 0;
  if (int rc = current_device(&dev, &status, &num_sms)) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const bool bf = dtype == ETATTN_BF16;
  const int nq_pad = (Nq + 127) / 128 * 128;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  float* dq_acc = has_q ? reinterpret_cast<float*>(ws + L.dq_off) : nullptr;
  float* nlse2 = has_q ? reinterpret_cast<float*>(ws + L.lse2_off) : nullptr;
  float* nsd = has_q ? reinterpret_cast<float*>(ws + L.dvec_off) : nullptr;

  if (has_q) {
    BwdPreParams pp{};
    pp.o = o;
    pp.dout = dout;
    pp.lse = lse;
    pp.o_sb = st[12];
    pp.o_sh = st[13];
    pp.o_sn = st[14];
    pp.do_sb = st[16];
    pp.do_sh = st[17];
    pp.do_sn = st[18];
    pp.rows = (int64_t)B * Hq * nq_pad;
    pp.Hq = Hq;
    pp.Nq = Nq;
    pp.Nq_pad = nq_pad;
    pp.scale = scale;
    pp.nsd = nsd;
    pp.nlse2 = nlse2;
    pp.dq_acc = dq_acc;
    cudaError_t e = launch_bwd_pre(D, bf, pp, s);
    if (e != cudaSuccess) return fail_cuda(e);
  }
  if (has_k) {
    CUtensorMap mq, mk, mv, mdo, mdq;
    bool swq = false, swk = false, swv = false, swd = false;
    if (int rc = encode_map(&mk, dtype, k, D, Nk, Hkv, B, st[6], st[5], st[4], &swk)) return rc;
    if (int rc = encode_map(&mv, dtype, v, D, Nk, Hkv, B, st[10], st[9], st[8], &swv)) return rc;
    if (has_q) {
      if (int rc = encode_map(&mq, dtype, q, D, Nq, Hq, B, st[2], st[1], st[0], &swq)) return rc;
      if (int rc = encode_map(&mdo, dtype, dout, D, Nq, Hq, B, st[18], st[17], st[16], &swd)) return rc;
      if (int rc = encode_dq_map(&mdq, dq_acc, D, Nq, (int64_t)B * Hq)) return rc;
    } else {
      // No queries: every key's gradient is 0 and no Q / dO tile is loaded
      // or dQ box added; the key map stands in for the unused ones.
      mq = mk;
      mdo = mk;
      mdq = mk;
    }
    BwdParams p{};
    p.dk = dk;
    p.dv = dv;
    p.dk_sb = st[24];
    p.dk_sh = st[25];
    p.dk_sn = st[26];
    p.dv_sb = st[28];
    p.dv_sh = st[29];
    p.dv_sn = st[30];
    p.nlse2 = nlse2;
    p.nsd = nsd;
    p.Nq = Nq;
    p.Nk = Nk;
    p.Nq_pad = nq_pad;
    p.Hq = Hq;
    p.group = Hq / Hkv;
    p.win_left = window_left_of(window_left);
    p.win_right = window_right_of(window_right, causal);
    p.scale = scale;
    p.scale_log2 = scale * 1.4426950408889634f;
    p.status = status;
    p.hn_swapped = (swq ? 1 : 0) | (swk ? 2 : 0) | (swv ? 4 : 0) | (swd ? 8 : 0);
    // Grouped longest-first order (the kernel's bwd_cta_coords), as for the
    // forward launch: groups of G (KV head, batch) pairs, G the smallest power
    // of two whose CTAs fill the SMs once.
    const int64_t gx = (Nk + 127) / 128, pairs = (int64_t)Hkv * B;
    dim3 grid((unsigned)gx, (unsigned)Hkv, (unsigned)B);
    p.grid_x = (int)gx;
    p.grid_y = Hkv;
    p.sched_q = p.sched_rem = 0;
    if (gx * pairs > num_sms && gx * pairs <= 0x7fffffffLL) {
      int64_t G = 1;
      while (G * gx < num_sms && G < pairs) G *= 2;
      const int64_t groups = (pairs + G - 1) / G;
      p.sched_q = (int)(pairs / groups);
      p.sched_rem = (int)(pairs % groups);
      grid = dim3((unsigned)(gx * pairs), 1, 1);
    }
    cudaError_t e;
    switch (D) {
      case 32:
        e = bf ? launch_bwd_d32_1(mq, mk, mv, mdo, mdq, p, grid, s)
               : launch_bwd_d32_0(mq, mk, mv, mdo, mdq, p, grid, s);
        break;
      case 64:
        e = bf ? launch_bwd_d64_1(mq, mk, mv, mdo, mdq, p, grid, s)
               : launch_bwd_d64_0(mq, mk, mv, mdo, mdq, p, grid, s);
        break;
      default:
        e = bf ? launch_bwd_d128_1(mq, mk, mv, mdo, mdq, p, grid, s)
               : launch_bwd_d128_0(mq, mk, mv, mdo, mdq, p, grid, s);
    }
    if (e != cudaSuccess) return fail_cuda(e);
  }
  if (has_q) {
    BwdConvertParams cp{};
    cp.dq_acc = dq_acc;
    cp.dq = dq;
    cp.dq_sb = st[20];
    cp.dq_sh = st[21];
    cp.dq_sn = st[22];
    cp.rows = (int64_t)B * Hq * Nq;
    cp.Hq = Hq;
    cp.Nq = Nq;
    cudaError_t e = launch_bwd_convert(D, bf, cp, s);
    if (e != cudaSuccess) return fail_cuda(e);
  }
  return ETATTN_OK;
}

// Host mirror of packed offsets: 0, non-decreasing, ending at total, every
// length <= max_len.
// whole = false: the offsets of a run of sequences inside a packed batch
// (they start at or after 0 and end at or before the total).
bool seqlens_ok(const int32_t* cu, int num_seqs, int total, int max_len, bool whole = true) {
  if (whole ? (cu[0] != 0 || cu[num_seqs] != total) : (cu[0] < 0 || cu[num_seqs] > total)) return false;
  for (int s = 0; s < num_seqs; ++s) {
    const int64_t len = (int64_t)cu[s + 1] - cu[s];
    if (len < 0 || len > max_len) return false;
  }
  return true;
}

int varlen_impl(const void* q, const void* k, const void* v, void* o, float* lse, const int32_t* cu_seqlens_q,
                const int32_t* cu_seqlens_k, const int32_t* cu_seqlens_q_host, const int32_t* cu_seqlens_k_host,
                int num_seqs, int max_seqlen_q, int max_seqlen_k, int total_q, int total_k, int Hq, int Hkv, int D,
                int dtype, const int64_t* strides, int causal, int window_left, int window_right, float scale,
                void* stream, bool do_launch, const SplitArgs* split = nullptr, int num_global = 0,
                bool sub_range = false, int ks_force = -1) {
  if (dtype != ETATTN_F16 && dtype != ETATTN_BF16) return ETATTN_ERR_BAD_DTYPE;
  if (num_seqs < 0 || max_seqlen_q < 0 || max_seqlen_k < 0 || total_q < 0 || total_k < 0 || Hq < 0 ||
      !head_dim_ok(D))
    return ETATTN_ERR_BAD_SHAPE;
  if (max_seqlen_q > kMaxTokens || max_seqlen_k > kMaxTokens || num_seqs > kMaxGridYZ || Hq > kMaxGridYZ)
    return ETATTN_ERR_BAD_SHAPE;
  if (Hkv <= 0 || Hq % Hkv != 0) return ETATTN_ERR_BAD_HEADS;
  if (!std::isfinite(scale) || !(scale > 0.f)) return ETATTN_ERR_BAD_SCALE;
  if (strides == nullptr) return ETATTN_ERR_NULL_PTR;
  if (num_global < 0 || (num_global > 0 && split != nullptr)) return ETATTN_ERR_BAD_SHAPE;
  if (split != nullptr && (split->num_splits < 1 || split->num_splits > kMaxSplits)) return ETATTN_ERR_BAD_SHAPE;
  if (cu_seqlens_q_host && !seqlens_ok(cu_seqlens_q_host, num_seqs, total_q, max_seqlen_q, !sub_range))
    return ETATTN_ERR_BAD_SEQLENS;
  if (cu_seqlens_k_host && !seqlens_ok(cu_seqlens_k_host, num_seqs, total_k, max_seqlen_k, !sub_range))
    return ETATTN_ERR_BAD_SEQLENS;
  if (num_seqs == 0 || Hq == 0 || total_q == 0 || max_seqlen_q == 0) return ETATTN_OK;
  const bool has_keys = total_k > 0;
  if (!q || !o || !cu_seqlens_q || !cu_seqlens_k || (has_keys && (!k || !v))) return ETATTN_ERR_NULL_PTR;

  const int T = total_q, Tk = total_k;
  const View vq{q, 3, {T, Hq, D, 0}, {strides[0], strides[1], strides[2], 0}};
  const View vk{k, 3, {Tk, Hkv, D, 0}, {strides[3], strides[4], strides[5], 0}};
  const View vv{v, 3, {Tk, Hkv, D, 0}, {strides[6], strides[7], strides[8], 0}};
  const View vo{o, 3, {T, Hq, D, 0}, {strides[9], strides[10], strides[11], 0}};
  const View vl{lse, 2, {Hq, T, 0, 0}, {T, 1, 0, 0}};
  for (const View* t : {&vq, &vk, &vv, &vo})
    if (!strides_ok(*t, 2)) return ETATTN_ERR_BAD_STRIDE;
  for (const void* ptr : {q, (const void*)o})
    if (!aligned16(ptr)) return ETATTN_ERR_BAD_ALIGN;
  if (has_keys && (!aligned16(k) || !aligned16(v))) return ETATTN_ERR_BAD_ALIGN;
  if (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)) return ETATTN_ERR_BAD_ALIGN;
  if ((reinterpret_cast<uintptr_t>(cu_seqlens_q) & 3u) || (reinterpret_cast<uintptr_t>(cu_seqlens_k) & 3u))
    return ETATTN_ERR_BAD_ALIGN;
  for (const View* t : {&vq, &vk, &vv})
    if (overlaps(vo, 2, *t, 2) || (lse && overlaps(vl, 4, *t, 2))) return ETATTN_ERR_ALIAS;
  if (lse && overlaps(vl, 4, vo, 2)) return ETATTN_ERR_ALIAS;
  // Split-KV: as in fwd_impl, one partial state per (slice, query head,
  // token) row, at the row's lse index h * T + t.
  const int64_t rows = (int64_t)Hq * T;
  const bool splitting = split != nullptr && split->num_splits > 1 && has_keys;
  if (splitting) {
    const size_t need = splitkv_bytes(rows, D, split->num_splits);
    if (need == 0) return ETATTN_ERR_BAD_SHAPE;
    if (split->workspace == nullptr) return ETATTN_ERR_NULL_PTR;
    if (reinterpret_cast<uintptr_t>(split->workspace) % kWorkspaceAlign) return ETATTN_ERR_BAD_ALIGN;
    if (split->workspace_bytes < need) return ETATTN_ERR_BAD_SHAPE;
    const View vw{split->workspace, 1, {(int64_t)need, 0, 0, 0}, {1, 0, 0, 0}};
    for (const View* t : {&vq, &vk, &vv, &vo})
      if (overlaps(vw, 1, *t, 2)) return ETATTN_ERR_ALIAS;
    if (lse && overlaps(vw, 1, vl, 4)) return ETATTN_ERR_ALIAS;
  }
  if (!do_launch) return ETATTN_OK;

  int dev = 0;
  int* status = nullptr;
  int num_sms = 0;
  if (int rc = current_device(&dev, &status, &num_sms)) return rc;

  // Shared query and key offsets mean equal lengths in every sequence (see
  // fwd_impl for why the right bound does not matter).
  const bool general = cu_seqlens_k != cu_seqlens_q || window_left_of(window_left) != kUnboundedWindow || splitting ||
                       num_global > 0;
  const int qpack = qpack_of(general, Hq / Hkv, max_seqlen_q);

  CUtensorMap mq, mk, mv;
  bool swq = false, swk = false, swv = false;
  if (int rc = encode_map(&mq, dtype, q, D, T, Hq, 1, strides[0], strides[1], 0, &swq, qpack)) return rc;
  if (has_keys) {
    if (int rc = encode_map(&mk, dtype, k, D, Tk, Hkv, 1, strides[3], strides[4], 0, &swk)) return rc;
    if (int rc = encode_map(&mv, dtype, v, D, Tk, Hkv, 1, strides[6], strides[7], 0, &swv)) return rc;
  } else {
    mk = mq;  // unused: no sequence has a key (see fwd_impl)
    mv = mq;
    swk = swv = swq;
  }

  FwdParams p{};
  p.o = o;
  p.lse = lse;
  p.o_sb = 0;
  p.o_sh = strides[10];
  p.o_sn = strides[9];
  p.lse_sb = 0;
  p.lse_sh = T;
  p.cu_seqlens_q = cu_seqlens_q;
  p.cu_seqlens_k = cu_seqlens_k;
  p.Nq = p.Nk = 0;
  p.total_q = T;
  p.total_k = Tk;
  p.max_seqlen_q = max_seqlen_q;
  p.max_seqlen_k = max_seqlen_k;
  p.Hq = Hq;
  p.group = Hq / Hkv;
  p.win_left = window_left_of(window_left);
  p.win_right = window_right_of(window_right, causal);
  p.scale = scale;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.status = status;
  p.hn_swapped = (swq ? 1 : 0) | (swk ? 2 : 0) | (swv ? 4 : 0);
  p.qpack = qpack;
  p.num_global = has_keys ? std::min(num_global, kMaxTokens) : 0;
  p.win_right_causal = causal ? 0 : kUnboundedWindow;
  const int64_t key_tiles = ((int64_t)max_seqlen_k + 127) / 128;
  if (splitting) {
    uint8_t* ws = static_cast<uint8_t*>(split->workspace);
    p.part_o = reinterpret_cast<float*>(ws);
    p.part_lse = reinterpret_cast<float*>(ws + splitkv_lse_offset(rows, D, split->num_splits));
    p.part_stride = rows;
    p.num_splits = split->num_splits;
    p.split_tiles = (int)((key_tiles + split->num_splits - 1) / split->num_splits);
  }
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  // Without host copies of the offsets any sequence may be short.
  bool few = dtype == ETATTN_BF16;
  if (few && cu_seqlens_q_host != nullptr && cu_seqlens_k_host != nullptr) {
    few = false;
    for (int i = 0; i < num_seqs && !few; ++i)
      few = has_few_key_rows(cu_seqlens_q_host[i + 1] - cu_seqlens_q_host[i],
                             cu_seqlens_k_host[i + 1] - cu_seqlens_k_host[i], p.win_left, p.win_right,
                             p.win_right_causal, p.num_global);
  }
  cudaError_t e = launch(D, dtype, mq, mk, mv, p, (int64_t)max_seqlen_q * qpack, (unsigned)(Hq / qpack),
                         (unsigned)num_seqs, num_sms, general, few, st, key_tiles, ks_force);
  if (e != cudaSuccess) return fail_cuda(e);
  if (splitting) {
    CombineParams c{};
    c.part_o = p.part_o;
    c.part_lse = p.part_lse;
    c.rows = rows;
    c.num_splits = p.num_splits;
    c.o = o;
    c.lse = lse;
    c.o_sb = 0;
    c.o_sh = strides[10];
    c.o_sn = strides[9];
    c.Hq = Hq;
    c.Nq = 0;
    c.packed = 1;
    c.total = T;
    e = launch_combine(D, dtype == ETATTN_BF16, c, st);
    if (e != cudaSuccess) return fail_cuda(e);
  }
  return ETATTN_OK;
}

// ---------------------------------------------------------------- host-buffer pipeline
// The host-buffer calls cut the problem into chunks (whole sequences of a
// packed batch, whole batches, or runs of KV heads) and pipeline them over
// the current device's two copy streams: chunk c + 1's inputs travel to the
// device while chunk c's kernel runs on the caller's stream, and chunk c's
// outputs travel back meanwhile.  The streams and events are created on first
// use and kept; a mutex per device orders the enqueues of concurrent calls.
constexpr int kHostChunks = 8;

struct HostPipe {
  std::mutex mu;
  bool ready = false;
  cudaStream_t h2d = nullptr, d2h = nullptr;
  cudaEvent_t start = nullptr, end = nullptr;
  cudaEvent_t in[kHostChunks] = {}, out[kHostChunks] = {};
};
HostPipe g_host_pipes[64];

// Creates the device's copy streams and events once; the caller holds pipe.mu.
int host_pipe_ready(HostPipe& hp) {
  if (hp.ready) return ETATTN_OK;
  cudaError_t e = cudaStreamCreateWithFlags(&hp.h2d, cudaStreamNonBlocking);
  if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&hp.d2h, cudaStreamNonBlocking);
  if (e == cudaSuccess) e = cudaEventCreateWithFlags(&hp.start, cudaEventDisableTiming);
  if (e == cudaSuccess) e = cudaEventCreateWithFlags(&hp.end, cudaEventDisableTiming);
  for (int c = 0; c < kHostChunks && e == cudaSuccess; ++c) {
    e = cudaEventCreateWithFlags(&hp.in[c], cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&hp.out[c], cudaEventDisableTiming);
  }
  if (e != cudaSuccess) return fail_cuda(e);
  hp.ready = true;
  return ETATTN_OK;
}

// Cuts n items with prefix sums pre[0..n] (pre[0] = 0 after rebasing) into at
// most max_chunks runs of about equal weight: a run ends after the first item
// whose prefix reaches the next multiple of total / chunks.  bounds[0..k] get
// the item indices; returns k (0 when n == 0).
int plan_runs(const int64_t* pre, int n, int max_chunks, int32_t* bounds) {
  if (n <= 0) return 0;
  const int k_max = std::max(1, std::min(std::min(max_chunks, kHostChunks), n));
  const int64_t total = pre[n] - pre[0];
  int k = 0;
  bounds[0] = 0;
  for (int i = 0; i < n; ++i) {
    const int64_t done = pre[i + 1] - pre[0];
    // close the run at item i when it reaches its share (the last run takes the rest)
    if (i + 1 == n || (k + 1 < k_max && done * k_max >= (int64_t)(k + 1) * total && total > 0))
      bounds[++k] = i + 1;
  }
  return k;
}

// The key-split choice `launch` makes for a whole square call of Hq heads
// (one query row per head, no packing) over `seqs` sequences or batches of up
// to `len` tokens, for its chunks to take.
int key_split_of(int64_t len, int64_t Hq, int64_t seqs, int num_sms) {
  const int64_t blocks1 = (len + 127) / 128;
  return blocks1 >= 2 && 2 * blocks1 * Hq * seqs <= num_sms ? 1 : 0;
}

// Enqueues the start of a pipelined call: the copy streams wait for the work
// already on the caller's stream.
cudaError_t pipe_begin(HostPipe& hp, cudaStream_t s) {
  cudaError_t e = cudaEventRecord(hp.start, s);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(hp.h2d, hp.start, 0);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(hp.d2h, hp.start, 0);
  return e;
}

// The caller's stream waits for the last output copy, so that the call's
// completion is observed on it.
cudaError_t pipe_end(HostPipe& hp, cudaStream_t s) {
  cudaError_t e = cudaEventRecord(hp.end, hp.d2h);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(s, hp.end, 0);
  return e;
}

}  // namespace

extern "C" {

int attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv, int N,
             int D, int dtype, const int64_t* strides, int causal, float scale, void* stream) {
  return fwd_impl(q, k, v, o, lse, B, Hq, Hkv, N, N, D, dtype, strides, causal, -1, -1, scale, stream, true);
}

int attn_fwd_ex(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv, int Nq,
                int Nk, int D, int dtype, const int64_t* strides, int causal, int window_left, int window_right,
                float scale, void* stream) {
  return fwd_impl(q, k, v, o, lse, B, Hq, Hkv, Nq, Nk, D, dtype, strides, causal, window_left, window_right, scale,
                  stream, true);
}

int attn_fwd_splitkv(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv,
                     int Nq, int Nk, int D, int dtype, const int64_t* strides, int causal, int window_left,
                     int window_right, float scale, int num_splits, void* workspace, size_t workspace_bytes,
                     void* stream) {
  const SplitArgs sa{num_splits, workspace, workspace_bytes};
  return fwd_impl(q, k, v, o, lse, B, Hq, Hkv, Nq, Nk, D, dtype, strides, causal, window_left, window_right, scale,
                  stream, true, &sa);
}

int attn_fwd_global(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv,
                    int Nq, int Nk, int D, int dtype, const int64_t* strides, int causal, int window_left,
                    int window_right, int num_global, float scale, void* stream) {
  if (num_global < 0) return ETATTN_ERR_BAD_SHAPE;
  // The window already holds every key the causal mask allows: nothing to add.
  const bool window_is_everything = window_left_of(window_left) == kUnboundedWindow &&
                                    window_right_of(window_right, causal) == (causal ? 0 : kUnboundedWindow);
  return fwd_impl(q, k, v, o, lse, B, Hq, Hkv, Nq, Nk, D, dtype, strides, causal, window_left, window_right, scale,
                  stream, true, nullptr, window_is_everything ? 0 : num_global);
}

// For callers that cannot allocate device memory at call time: a runtime
// whose device memory is all held by its own pool and that offers the
// attention call no allocation hook, or a plugin that is handed only the
// tensors of the step.  They get the split-KV path with the library's own
// fixed scratch instead of a workspace argument.
int attn_fwd_splitkv_noalloc(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq,
                             int Hkv, int Nq, int Nk, int D, int dtype, const int64_t* strides, int causal,
                             int window_left, int window_right, float scale, int num_splits, void* stream) {
  if (B < 0 || Hq < 0 || Nq < 0 || !head_dim_ok(D)) return ETATTN_ERR_BAD_SHAPE;
  if (num_splits < 1 || num_splits > kMaxSplits) return ETATTN_ERR_BAD_SHAPE;
  const int64_t rows = (int64_t)B * Hq * Nq;
  // Only a call that splits (more than one slice over at least one key)
  // uses the scratch; without keys every row is empty and nothing is split.
  if (num_splits > 1 && rows > 0 && Nk > 0 &&
      (splitkv_bytes(rows, D, num_splits) == 0 || splitkv_bytes(rows, D, num_splits) > kNoAllocScratchBytes))
    return ETATTN_ERR_BAD_SHAPE;  // beyond the fixed scratch
  // Every other argument is checked before the first device query.
  if (int rc = fwd_impl(q, k, v, o, lse, B, Hq, Hkv, Nq, Nk, D, dtype, strides, causal, window_left, window_right,
                        scale, stream, false))
    return rc;
  if (B == 0 || Hq == 0 || Nq == 0) return ETATTN_OK;
  void* scratch = nullptr;
  if (int rc = noalloc_scratch(&scratch)) return rc;
  const SplitArgs sa{num_splits, scratch, kNoAllocScratchBytes};
  return fwd_impl(q, k, v, o, lse, B, Hq, Hkv, Nq, Nk, D, dtype, strides, causal, window_left, window_right, scale,
                  stream, true, &sa);
}

size_t attn_fwd_splitkv_workspace_size(int B, int Hq, int Nq, int D, int num_splits) {
  if (B < 0 || Hq < 0 || Nq < 0 || !head_dim_ok(D) || num_splits < 1 || num_splits > kMaxSplits) return 0;
  return splitkv_bytes((int64_t)B * Hq * Nq, D, num_splits);
}

int attn_fwd_splitkv_plan(int B, int Hq, int Hkv, int Nq, int Nk, int* num_splits) {
  if (num_splits == nullptr) return ETATTN_ERR_NULL_PTR;
  if (B < 0 || Hq < 0 || Nq < 0 || Nk < 0) return ETATTN_ERR_BAD_SHAPE;
  if (Hkv <= 0 || Hq % Hkv != 0) return ETATTN_ERR_BAD_HEADS;
  int dev = 0, num_sms = 0;
  int* status = nullptr;
  if (int rc = current_device(&dev, &status, &num_sms)) return rc;
  const int P = qpack_of(true, Hq / Hkv, Nq);  // split launches use the general build
  const int64_t units = (int64_t)B * (Hq / P) * (((int64_t)Nq * P + 127) / 128);
  *num_splits = plan_splits(units, ((int64_t)Nk + 127) / 128, num_sms);
  return ETATTN_OK;
}

int attn_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dout, void* dq,
             void* dk, void* dv, int B, int Hq, int Hkv, int Nq, int Nk, int D, int dtype, const int64_t* strides,
             int causal, int window_left, int window_right, float scale, void* workspace, size_t workspace_bytes,
             void* stream) {
  return bwd_impl(q, k, v, o, lse, dout, dq, dk, dv, B, Hq, Hkv, Nq, Nk, D, dtype, strides, causal, window_left,
                  window_right, scale, workspace, workspace_bytes, stream);
}

size_t attn_bwd_workspace_size(int B, int Hq, int Nq, int D) {
  if (B < 0 || Hq < 0 || Nq < 0 || !head_dim_ok(D)) return 0;
  if (B == 0 || Hq == 0 || Nq == 0) return 0;
  return bwd_layout(B, Hq, Nq, D).total;
}

int attn_fwd_varlen(const void* q, const void* k, const void* v, void* o, float* lse, const int32_t* cu_seqlens,
                    const int32_t* cu_seqlens_host, int num_seqs, int max_seqlen, int total_tokens, int Hq,
                    int Hkv, int D, int dtype, const int64_t* strides, int causal, float scale, void* stream) {
  return varlen_impl(q, k, v, o, lse, cu_seqlens, cu_seqlens, cu_seqlens_host, cu_seqlens_host, num_seqs, max_seqlen,
                     max_seqlen, total_tokens, total_tokens, Hq, Hkv, D, dtype, strides, causal, -1, -1, scale, stream,
                     true);
}

int attn_fwd_varlen_ex(const void* q, const void* k, const void* v, void* o, float* lse,
                       const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k, const int32_t* cu_seqlens_q_host,
                       const int32_t* cu_seqlens_k_host, int num_seqs, int max_seqlen_q, int max_seqlen_k,
                       int total_q, int total_k, int Hq, int Hkv, int D, int dtype, const int64_t* strides, int causal,
                       int window_left, int window_right, float scale, void* stream) {
  return varlen_impl(q, k, v, o, lse, cu_seqlens_q, cu_seqlens_k, cu_seqlens_q_host, cu_seqlens_k_host, num_seqs,
                     max_seqlen_q, max_seqlen_k, total_q, total_k, Hq, Hkv, D, dtype, strides, causal, window_left,
                     window_right, scale, stream, true);
}

int attn_fwd_varlen_splitkv(const void* q, const void* k, const void* v, void* o, float* lse,
                            const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k, const int32_t* cu_seqlens_q_host,
                            const int32_t* cu_seqlens_k_host, int num_seqs, int max_seqlen_q, int max_seqlen_k,
                            int total_q, int total_k, int Hq, int Hkv, int D, int dtype, const int64_t* strides,
                            int causal, int window_left, int window_right, float scale, int num_splits,
                            void* workspace, size_t workspace_bytes, void* stream) {
  const SplitArgs sa{num_splits, workspace, workspace_bytes};
  return varlen_impl(q, k, v, o, lse, cu_seqlens_q, cu_seqlens_k, cu_seqlens_q_host, cu_seqlens_k_host, num_seqs,
                     max_seqlen_q, max_seqlen_k, total_q, total_k, Hq, Hkv, D, dtype, strides, causal, window_left,
                     window_right, scale, stream, true, &sa);
}

size_t attn_fwd_varlen_splitkv_workspace_size(int total_q, int Hq, int D, int num_splits) {
  if (total_q < 0 || Hq < 0 || !head_dim_ok(D) || num_splits < 1 || num_splits > kMaxSplits) return 0;
  return splitkv_bytes((int64_t)total_q * Hq, D, num_splits);
}

int attn_fwd_varlen_splitkv_plan(int num_seqs, int Hq, int Hkv, int max_seqlen_q, int max_seqlen_k,
                                 int* num_splits) {
  // The batched planner's wave model with every sequence as long as the
  // longest: the grid has num_seqs sequences of max_seqlen_q query rows.
  return attn_fwd_splitkv_plan(num_seqs, Hq, Hkv, max_seqlen_q, max_seqlen_k, num_splits);
}

int attn_fwd_varlen_global(const void* q, const void* k, const void* v, void* o, float* lse,
                           const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k, const int32_t* cu_seqlens_q_host,
                           const int32_t* cu_seqlens_k_host, int num_seqs, int max_seqlen_q, int max_seqlen_k,
                           int total_q, int total_k, int Hq, int Hkv, int D, int dtype, const int64_t* strides,
                           int causal, int window_left, int window_right, int num_global, float scale, void* stream) {
  if (num_global < 0) return ETATTN_ERR_BAD_SHAPE;
  const bool window_is_everything = window_left_of(window_left) == kUnboundedWindow &&
                                    window_right_of(window_right, causal) == (causal ? 0 : kUnboundedWindow);
  return varlen_impl(q, k, v, o, lse, cu_seqlens_q, cu_seqlens_k, cu_seqlens_q_host, cu_seqlens_k_host, num_seqs,
                     max_seqlen_q, max_seqlen_k, total_q, total_k, Hq, Hkv, D, dtype, strides, causal, window_left,
                     window_right, scale, stream, true, nullptr, window_is_everything ? 0 : num_global);
}

int attn_fwd_varlen_host_plan(const int32_t* cu_seqlens_host, int num_seqs, int max_chunks,
                                         int32_t* seq_bounds) {
  if (cu_seqlens_host == nullptr || seq_bounds == nullptr) return -ETATTN_ERR_NULL_PTR;
  if (num_seqs < 0 || max_chunks < 1) return -ETATTN_ERR_BAD_SHAPE;
  std::vector<int64_t> pre((size_t)num_seqs + 1);
  for (int i = 0; i <= num_seqs; ++i) pre[i] = cu_seqlens_host[i];
  for (int i = 0; i < num_seqs; ++i)
    if (pre[i + 1] < pre[i]) return -ETATTN_ERR_BAD_SEQLENS;
  return plan_runs(pre.data(), num_seqs, max_chunks, seq_bounds);
}

int attn_fwd_host(const void* q_host, const void* k_host, const void* v_host, void* o_host, float* lse_host,
                  void* q_dev, void* k_dev, void* v_dev, void* o_dev, float* lse_dev, int B, int Hq, int Hkv, int N,
                  int D, int dtype, int causal, float scale, void* stream) {
  if ((lse_host == nullptr) != (lse_dev == nullptr)) return ETATTN_ERR_NULL_PTR;
  const int64_t st[16] = {(int64_t)Hq * N * D,  (int64_t)N * D, D, 1, (int64_t)Hkv * N * D, (int64_t)N * D, D, 1,
                          (int64_t)Hkv * N * D, (int64_t)N * D, D, 1, (int64_t)Hq * N * D,  (int64_t)N * D, D, 1};
  if (int rc = fwd_impl(q_dev, k_dev, v_dev, o_dev, lse_dev, B, Hq, Hkv, N, N, D, dtype, st, causal, -1, -1, scale,
                        stream, false))
    return rc;
  if (B == 0 || Hq == 0 || N == 0) return ETATTN_OK;
  if (!q_host || !k_host || !v_host || !o_host) return ETATTN_ERR_NULL_PTR;
  // Chunks: runs of whole batches, or of KV heads (with their query heads)
  // when there is one batch; each is contiguous in every buffer.
  const int g = Hq / Hkv;
  const bool by_batch = B > 1;
  const int units = by_batch ? B : Hkv;
  const int64_t q_unit = (by_batch ? (int64_t)Hq : g) * N * D * 2;  // bytes of one unit's Q (and O)
  const int64_t kv_unit = (by_batch ? (int64_t)Hkv : 1) * N * D * 2;
  const int64_t l_unit = (by_batch ? (int64_t)Hq : g) * N;          // lse entries of one unit
  std::vector<int64_t> pre((size_t)units + 1);
  for (int i = 0; i <= units; ++i) pre[i] = i;
  int32_t bounds[kHostChunks + 1];
  const int k = plan_runs(pre.data(), units, kHostChunks, bounds);
  int dev = 0, num_sms = 0;
  int* status = nullptr;
  if (int rc = current_device(&dev, &status, &num_sms)) return rc;
  const int ks = key_split_of(N, Hq, B, num_sms);
  HostPipe& hp = g_host_pipes[dev];
  std::lock_guard<std::mutex> lk(hp.mu);
  if (int rc = host_pipe_ready(hp)) return rc;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  auto at = [](const void* base, int64_t off) { return static_cast<const char*>(base) + off; };
  auto atw = [](void* base, int64_t off) { return static_cast<char*>(base) + off; };
  cudaError_t e = pipe_begin(hp, s);
  for (int c = 0; c < k && e == cudaSuccess; ++c) {
    const int u0 = bounds[c], nu = bounds[c + 1] - bounds[c];
    e = cudaMemcpyAsync(atw(q_dev, u0 * q_unit), at(q_host, u0 * q_unit), nu * q_unit, cudaMemcpyHostToDevice,
                        hp.h2d);
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(atw(k_dev, u0 * kv_unit), at(k_host, u0 * kv_unit), nu * kv_unit, cudaMemcpyHostToDevice,
                          hp.h2d);
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(atw(v_dev, u0 * kv_unit), at(v_host, u0 * kv_unit), nu * kv_unit, cudaMemcpyHostToDevice,
                          hp.h2d);
    if (e == cudaSuccess) e = cudaEventRecord(hp.in[c], hp.h2d);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(s, hp.in[c], 0);
    if (e != cudaSuccess) break;
    float* lse_c = lse_dev ? lse_dev + u0 * l_unit : nullptr;
    if (int rc = fwd_impl(at(q_dev, u0 * q_unit), at(k_dev, u0 * kv_unit), at(v_dev, u0 * kv_unit),
                          atw(o_dev, u0 * q_unit), lse_c, by_batch ? nu : 1, by_batch ? Hq : nu * g,
                          by_batch ? Hkv : nu, N, N, D, dtype, st, causal, -1, -1, scale, stream, true, nullptr, 0,
                          ks))
      return rc;
    e = cudaEventRecord(hp.out[c], s);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(hp.d2h, hp.out[c], 0);
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(atw(o_host, u0 * q_unit), at(o_dev, u0 * q_unit), nu * q_unit, cudaMemcpyDeviceToHost,
                          hp.d2h);
    if (e == cudaSuccess && lse_host)
      e = cudaMemcpyAsync(lse_host + u0 * l_unit, lse_dev + u0 * l_unit, nu * l_unit * sizeof(float),
                          cudaMemcpyDeviceToHost, hp.d2h);
  }
  if (e == cudaSuccess) e = pipe_end(hp, s);
  if (e != cudaSuccess) return fail_cuda(e);
  return ETATTN_OK;
}

int attn_fwd_varlen_host(const void* q_host, const void* k_host, const void* v_host, void* o_host, float* lse_host,
                         const int32_t* cu_seqlens_host, void* q_dev, void* k_dev, void* v_dev, void* o_dev,
                         float* lse_dev, int32_t* cu_seqlens_dev, int num_seqs, int max_seqlen, int total_tokens,
                         int Hq, int Hkv, int D, int dtype, int causal, float scale, void* stream) {
  if ((lse_host == nullptr) != (lse_dev == nullptr)) return ETATTN_ERR_NULL_PTR;
  if (cu_seqlens_host == nullptr) return ETATTN_ERR_NULL_PTR;
  const int64_t st[12] = {(int64_t)Hq * D, D, 1, (int64_t)Hkv * D, D, 1, (int64_t)Hkv * D, D, 1, (int64_t)Hq * D, D, 1};
  if (int rc = varlen_impl(q_dev, k_dev, v_dev, o_dev, lse_dev, cu_seqlens_dev, cu_seqlens_dev, cu_seqlens_host,
                           cu_seqlens_host, num_seqs, max_seqlen, max_seqlen, total_tokens, total_tokens, Hq, Hkv, D,
                           dtype, st, causal, -1, -1, scale, stream, false))
    return rc;
  if (num_seqs == 0 || Hq == 0 || total_tokens == 0 || max_seqlen == 0) return ETATTN_OK;
  if (!q_host || !k_host || !v_host || !o_host) return ETATTN_ERR_NULL_PTR;
  // Chunks: runs of whole sequences of about equal token counts; each chunk's
  // rows are contiguous in Q, K, V and O and form one column band of lse
  // [Hq, T].  A chunk's launch reads its own run of the offsets in place
  // (absolute token positions inside the whole buffers).
  const int64_t T = total_tokens;
  const int64_t q_tok = (int64_t)Hq * D * 2, kv_tok = (int64_t)Hkv * D * 2;  // bytes per token
  std::vector<int64_t> pre((size_t)num_seqs + 1);
  for (int i = 0; i <= num_seqs; ++i) pre[i] = cu_seqlens_host[i];
  int32_t bounds[kHostChunks + 1];
  const int k = plan_runs(pre.data(), num_seqs, kHostChunks, bounds);
  // Processing order: nothing overlaps the first run's upload, nor the last
  // run's kernel and download, so the run with the fewest tokens goes first
  // and, of the others, the one with the least causal work (sum of squared
  // lengths) last; the rest keep their order.
  int order[kHostChunks];
  {
    int first = 0, last = -1;
    for (int c = 1; c < k; ++c)
      if (pre[bounds[c + 1]] - pre[bounds[c]] < pre[bounds[first + 1]] - pre[bounds[first]]) first = c;
    double best = 0.0;
    for (int c = 0; c < k; ++c) {
      if (c == first) continue;
      double work = 0.0;
      for (int i = bounds[c]; i < bounds[c + 1]; ++i) work += (double)(pre[i + 1] - pre[i]) * (pre[i + 1] - pre[i]);
      if (last < 0 || work < best) {
        last = c;
        best = work;
      }
    }
    int n = 0;
    order[n++] = first;
    for (int c = 0; c < k; ++c)
      if (c != first && c != last) order[n++] = c;
    if (last >= 0) order[n++] = last;
  }
  int dev = 0, num_sms = 0;
  int* status = nullptr;
  if (int rc = current_device(&dev, &status, &num_sms)) return rc;
  const int ks = key_split_of(max_seqlen, Hq, num_seqs, num_sms);
  HostPipe& hp = g_host_pipes[dev];
  std::lock_guard<std::mutex> lk(hp.mu);
  if (int rc = host_pipe_ready(hp)) return rc;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  auto at = [](const void* base, int64_t off) { return static_cast<const char*>(base) + off; };
  auto atw = [](void* base, int64_t off) { return static_cast<char*>(base) + off; };
  cudaError_t e = pipe_begin(hp, s);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(cu_seqlens_dev, cu_seqlens_host, (size_t)(num_seqs + 1) * sizeof(int32_t),
                        cudaMemcpyHostToDevice, hp.h2d);
  for (int c = 0; c < k && e == cudaSuccess; ++c) {
    const int a = bounds[order[c]], b = bounds[order[c] + 1];
    const int64_t t0 = cu_seqlens_host[a], nt = (int64_t)cu_seqlens_host[b] - t0;
    int len_max = 0;
    for (int i = a; i < b; ++i) len_max = std::max(len_max, cu_seqlens_host[i + 1] - cu_seqlens_host[i]);
    if (nt > 0) {
      e = cudaMemcpyAsync(atw(q_dev, t0 * q_tok), at(q_host, t0 * q_tok), nt * q_tok, cudaMemcpyHostToDevice, hp.h2d);
      if (e == cudaSuccess)
        e = cudaMemcpyAsync(atw(k_dev, t0 * kv_tok), at(k_host, t0 * kv_tok), nt * kv_tok, cudaMemcpyHostToDevice,
                            hp.h2d);
      if (e == cudaSuccess)
        e = cudaMemcpyAsync(atw(v_dev, t0 * kv_tok), at(v_host, t0 * kv_tok), nt * kv_tok, cudaMemcpyHostToDevice,
                            hp.h2d);
    }
    if (e == cudaSuccess) e = cudaEventRecord(hp.in[c], hp.h2d);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(s, hp.in[c], 0);
    if (e != cudaSuccess) break;
    if (int rc = varlen_impl(q_dev, k_dev, v_dev, o_dev, lse_dev, cu_seqlens_dev + a, cu_seqlens_dev + a,
                             cu_seqlens_host + a, cu_seqlens_host + a, b - a, len_max, len_max, total_tokens,
                             total_tokens, Hq, Hkv, D, dtype, st, causal, -1, -1, scale, stream, true, nullptr, 0,
                             true, ks))
      return rc;
    e = cudaEventRecord(hp.out[c], s);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(hp.d2h, hp.out[c], 0);
    if (e == cudaSuccess && nt > 0)
      e = cudaMemcpyAsync(atw(o_host, t0 * q_tok), at(o_dev, t0 * q_tok), nt * q_tok, cudaMemcpyDeviceToHost, hp.d2h);
    if (e == cudaSuccess && nt > 0 && lse_host)
      e = cudaMemcpy2DAsync(lse_host + t0, (size_t)T * sizeof(float), lse_dev + t0, (size_t)T * sizeof(float),
                            (size_t)nt * sizeof(float), (size_t)Hq, cudaMemcpyDeviceToHost, hp.d2h);
  }
  if (e == cudaSuccess) e = pipe_end(hp, s);
  if (e != cudaSuccess) return fail_cuda(e);
  return ETATTN_OK;
}

const char* etattn_status_string(int code) {
  switch (code) {
    case ETATTN_OK: return "ok";
    case ETATTN_ERR_NULL_PTR: return "a required pointer is NULL";
    case ETATTN_ERR_BAD_DTYPE: return "unsupported dtype (expected F16 or BF16)";
    case ETATTN_ERR_BAD_SHAPE: return "bad shape (negative size, head dim not 32/64/128, or beyond limits)";
    case ETATTN_ERR_BAD_HEADS: return "bad head mapping (Hkv <= 0 or Hq not a multiple of Hkv)";
    case ETATTN_ERR_BAD_STRIDE: return "bad stride (d-stride must be 1; others positive multiples of 16 bytes)";
    case ETATTN_ERR_BAD_ALIGN: return "a base pointer is not 16-byte aligned";
    case ETATTN_ERR_ALIAS: return "an output overlaps an input or the other output";
    case ETATTN_ERR_BAD_SCALE: return "scale must be finite and > 0";
    case ETATTN_ERR_BAD_SEQLENS: return "bad cu_seqlens (must rise from 0 to the token total, lengths <= the max length)";
    case ETATTN_ERR_LAUNCH: return "a CUDA runtime call failed";
    case ETATTN_ERR_DEVICE: return "the device reported a failure (a bounded wait ran out)";
    case ETATTN_ERR_NO_DEVICE: return "no sm_103 CUDA device is current";
    default: return "unknown status";
  }
}

int etattn_last_cuda_error(void) { return t_last_cuda_error; }

int etattn_read_device_status(int* out, int clear, void* stream) {
  if (!out) return ETATTN_ERR_NULL_PTR;
  int dev = 0;
  int* status = nullptr;
  if (int rc = current_device(&dev, &status)) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return fail_cuda(e);
  int word = 0;
  e = cudaMemcpy(&word, status, sizeof(int), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return fail_cuda(e);
  if (clear && word != 0) {
    e = cudaMemset(status, 0, sizeof(int));
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return fail_cuda(e);
  }
  *out = word == kDevOk ? ETATTN_OK : word == kDevBadSeqlens ? ETATTN_ERR_BAD_SEQLENS : ETATTN_ERR_DEVICE;
  return ETATTN_OK;
}

int etattn_selftest_wait_timeout(int limit_us, void* stream) {
  if (limit_us < 1 || limit_us > 1000000) return ETATTN_ERR_BAD_SHAPE;
  int dev = 0;
  int* status = nullptr;
  if (int rc = current_device(&dev, &status)) return rc;
  wait_selftest_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>((unsigned long long)limit_us * 1000ull,
                                                                         status);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fail_cuda(e);
  return ETATTN_OK;
}

int etattn_version(void) { return 201; }

}  // extern "C"

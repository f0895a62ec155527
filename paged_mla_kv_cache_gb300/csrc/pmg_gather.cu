// Paged MLA KV-cache gather for GB300 (sm_103a).
//
// What it computes: "MLA cache gather scheduled per logical page"
// (prhub.com.cn, vllm PR #51739). For each request r, the entries of context
// tokens [start_r, start_r + len_r) are read through block_table row r out of a
// paged cache [num_blocks, block_size, entry] and written back to back into
// dst starting at row min(cu_seq_lens[r], T) (section "关键源码片段": the
// map_gather_page_task listing fixes the output placement and the page split,
// the test test_cp_gather_cache_mla_large_uneven_sequences fixes the per-token
// result). The write is a byte copy, an FP8 E4M3 dequant, or a widening cast
// (section "实现拆解" item 1: three gather kernels, raw copy, FP8 -> BF16
// upconvert and maybe-dequant).
//
// How this file does it (GB300-first, not the page's kernel):
//  * Work split. The page gives one CTA per logical page. Here a persistent
//    grid (a multiple of the SM count) splits the OUTPUT ROWS across CTAs, so a
//    300K-token request and a 17-token request cost each CTA the same bytes;
//    inside its rows a CTA walks page tasks in order. With a caller workspace,
//    each CTA takes a static head (a quarter of its rows, at least two ring
//    stages) and the rest is claimed in stage-sized items through an atomic
//    counter, which evens out CTAs whose memory traffic is served at
//    different speeds.
//  * Page-task mapper. The exclusive prefix sum of per-request page counts is
//    built in shared memory (by one warp for up to 256 requests, by the CTA
//    up to 4096; larger batches run as groups). A flat task id becomes (req,
//    logical_block, page_token_begin, page_token_end, output_token_begin) by a
//    binary search over that prefix: O(log R) where the page's mapper scans
//    all requests linearly.
//  * Broadcast. A scheduler warp resolves the tasks of the next work item one
//    per lane (map, one block-table read, bounds checks) into a shared-memory
//    segment queue while the current item's copies are in flight.
//  * Movement. Byte copies of 16-byte aligned rows use a TMA 1-D bulk ring
//    (cp.async.bulk global -> shared with an mbarrier, then shared -> global
//    bulk stores) driven by one thread. Converting gathers bulk-load source
//    rows into a ring that converter warps turn into 16-byte stores. Rows that
//    are not 16-byte aligned take SIMT loads and stores of 16, 8, 4, 2 or 1
//    bytes. The per-token entry point maps each output row through
//    token_to_seq; on the TMA kernels that is a mode of the scheduler warp,
//    which merges runs of adjacent source rows into bulk segments.
//  * Launch. Programmatic dependent launch: metadata is prefetched into L2
//    while the previous grid finishes. The TMA kernels plan and resolve their
//    first batch from it before that grid completes and confirm both by
//    reading every input used again afterwards (or skip the check under the
//    caller's early-metadata promise); the cache is read and dst written only
//    after it completes.
//  * Safety. 64-bit byte offsets everywhere; the logical block is checked
//    against block_table_stride and the physical id against num_blocks in
//    every path (the review section "评论区精华" reports both checks missing
//    and an int32 overflow of output_token_begin * entry_bytes). Bad pages are
//    skipped and reported in an error flag; nothing traps, and every wait on
//    an mbarrier is bounded in time.
//  * No tensor cores: the path is pure data movement, bound by HBM.

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>
#include <cstdlib>
#include <mutex>

#include "pmg.h"

namespace {

constexpr int kPlanThreads = 256;        // SIMT kernel / debug-plan CTA size
constexpr int kBulkThreads = 128;        // bulk kernel CTA size
constexpr int kMaxStages = 8;            // TMA ring depth per CTA: at most this many stages
constexpr int kMaxStageBytes = 48 * 1024;
constexpr int kUnroll = 4;               // SIMT units in flight per thread
constexpr int kMinRowsPerCta = 8;
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s per bounded wait

enum Conv : int {
  CONV_COPY = 0,
  CONV_E4M3_BF16 = 1,
  CONV_E4M3_F16 = 2,
  CONV_E4M3_F32 = 3,
  CONV_BF16_F32 = 4,
  CONV_F16_F32 = 5,
};

struct Params {
  const uint8_t* cache;
  int64_t blk_stride_b;   // bytes between blocks
  int64_t tok_stride_b;   // bytes between slots
  int64_t num_blocks;
  const int32_t* bt;
  int64_t bt_stride;      // elements
  const int32_t* cu;
  const int32_t* ss;      // may be null
  int32_t R;
  int32_t T;              // total_tokens clamped to INT32_MAX
  int32_t B;
  int32_t implied_end;    // cu has R entries; the last request ends at T
  int32_t row_src_bytes;  // entry_size * src element bytes
  int32_t row_dst_bytes;  // entry_size * dst element bytes
  uint8_t* dst;
  int64_t dst_stride_b;   // bytes between output rows
  const float* scale;     // may be null
  int32_t* err;           // may be null
  int32_t* sched;         // work-claim counter in the caller's workspace, or null (static split)
  const int32_t* carry_in;  // large batches: highest cu_seq_lens boundary of the groups before (or null)
  int32_t* carry_out;       // large batches: where this group's highest boundary goes for the next group
  int32_t early;          // plan and first block ids before the previous grid completes (caller's promise)
  int32_t spec;           // plan and first batch before the previous grid completes, checked after it
  int32_t spec_guess;     // speculative start of one request without seq_starts: assume cu = [0, T]
  int32_t prefetch_rows;  // rows of the pre-wait batch warmed in L2
  const int32_t* t2s;     // per-token gather: request of each output row (token mode)
  int32_t token_mode;     // 1: rows [0, T) map through t2s instead of the page plan
  int32_t sched_static_pct;  // dynamic mode: share of rows split statically up front
  int32_t sched_min_rows;    // dynamic mode only when rows per CTA reach this
  int32_t sched_head_stages; // dynamic mode: static share of at least this many ring stages per CTA
  int32_t sched_tilt_pct;    // static shares fall linearly with blockIdx: first (1 + t), last (1 - t) of even
  int32_t sched_tilt_pow;     // shape of the tilt: shares 1 + t (1 - (pow + 1) x^pow), x = blockIdx / grid
  // SIMT mover
  int32_t units_per_row;  // entry_size / elements per unit
  uint32_t upr_magic;     // fast division by units_per_row (fast_div)
  int32_t upr_shift;
  int32_t dense;          // src and dst rows are back to back: no row split
  // bulk mover
  int32_t stages;         // ring depth (<= kMaxStages)
  int32_t stage_bytes;    // bytes of one ring stage
  int32_t rows_per_stage;
  int32_t src_dense;
  int32_t dst_dense;
};

// ---------------------------------------------------------------------------
// Small device helpers
// ---------------------------------------------------------------------------

__device__ __forceinline__ void set_flag(const Params& p, int bits) {
  if (bits != 0 && p.err != nullptr) atomicOr(p.err, bits);
}

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Metadata (cu_seq_lens, seq_starts, block_table) is tiny and read by every
// CTA, and a serving loop reads the same arrays for every layer: keep it in L2
// (evict_last) while the entry stream goes through with evict_first.
__device__ __forceinline__ uint64_t evict_last_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// Loads of metadata are coherent at GPU scope (never served from a stale L1
// line): a speculative plan reads it before the previous grid is known to be
// done, and the check after the wait must see the final values.
__device__ __forceinline__ int32_t ld_meta(const int32_t* ptr, uint64_t pol) {
  int32_t v;
  asm volatile("ld.relaxed.gpu.global.L2::cache_hint.b32 %0, [%1], %2;" : "=r"(v) : "l"(ptr), "l"(pol));
  return v;
}

// Programmatic dependent launch: let the next kernel in the stream begin its
// launch now, and wait until the previous kernel's writes are visible before
// this grid reads any input. Both are no-ops for a normal launch.
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_entry() {
  pdl_trigger();
  pdl_wait();
}

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// first index i in [0, n) with a[i] > key, or n (a is non-decreasing)
__device__ __forceinline__ int upper_bound_i32(const int32_t* a, int n, int64_t key) {
  int lo = 0, hi = n;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (static_cast<int64_t>(a[mid]) <= key) lo = mid + 1; else hi = mid;
  }
  return lo;
}

// Division of a 32-bit unsigned n by a fixed d >= 1 with one multiply-high,
// an add and a shift: with l = ceil(log2 d) and m = floor(2^32 (2^l - d) / d) + 1,
// floor(n / d) = (mulhi(m, n) + n) >> l for every 32-bit n (the invariant-
// divisor method of Granlund and Montgomery, 1994). The host computes m and l.
__device__ __forceinline__ uint32_t fast_div(uint32_t n, uint32_t magic, int shift) {
  const uint64_t hi = __umulhi(magic, n);
  return static_cast<uint32_t>((hi + n) >> shift);
}

// ---------------------------------------------------------------------------
// Page plan: per-request output begins, starts and the page-count prefix
// ---------------------------------------------------------------------------

struct PlanView {
  int32_t* ob;  // [R + 1] clamped output begins; ob[R] = end of the last request
  int32_t* st;  // [R] source starts
  int32_t* P;   // [R + 1] exclusive prefix of page counts
};

__device__ __forceinline__ PlanView plan_view(uint8_t* base, const Params& p) {
  PlanView v;
  v.ob = reinterpret_cast<int32_t*>(base);
  v.st = v.ob + (p.R + 1);
  v.P = v.st + p.R;
  return v;
}

// Bytes of one plan in shared memory (ob, st and P back to back).
__device__ __forceinline__ size_t plan_bytes(const Params& p) {
  return (static_cast<size_t>(3) * p.R + 2) * sizeof(int32_t);
}

// Pages of request r: the logical blocks its source range [s, s + len) touches
// (0 for len == 0 or a negative start). With 0 <= s <= 2^31-1 and
// 1 <= len <= 2^31-1, s + len - 1 < 2^32, so 32-bit unsigned division is exact.
__device__ __forceinline__ int32_t request_pages(const PlanView& v, int r, int B) {
  const int32_t len = v.ob[r + 1] - v.ob[r];
  const int32_t s = v.st[r];
  if (len <= 0 || s < 0) return 0;
  const uint32_t ub = static_cast<uint32_t>(B);
  const uint32_t first = static_cast<uint32_t>(s) / ub;
  const uint32_t last = (static_cast<uint32_t>(s) + static_cast<uint32_t>(len) - 1u) / ub;
  return static_cast<int32_t>(last - first + 1u);
}

// Builds the plan. kWarp = false: all threads of the CTA take part (any R up
// to PMG_MAX_REQS_PLAN). kWarp = true: one warp builds it alone, with no
// CTA-wide barrier, for R <= kWarpPlanMaxReqs. Returns the number of page
// tasks. report_flags: this CTA reports the plan-level flag bits (one CTA per
// launch does, to keep atomics rare) and, for a group of a large batch, passes
// the highest boundary on to the next group.
//
// Output placement is the page's clamp: request r owns rows [c_r, c_{r+1})
// with c_r = min(cu[r], T) when c_{r+1} > c_r, and none otherwise. A request
// with rows whose first row lies below row 0 or below an earlier boundary
// (c_r < m_r, m_r = max(0, c_0, ..., c_r), the highest boundary so far) would
// overlap rows written before it, or run out of order: it is skipped
// (PMG_FLAG_CU_ORDER) and every other request is copied. The plan keeps
// ob[r] = m_r, which never decreases, so a binary search finds the request of
// any output row: a copied request has m_r = c_r and m_{r+1} = c_{r+1}; a
// request without rows has m_{r+1} = m_r; a skipped request keeps the rows
// [m_r, m_{r+1}) to itself (they stay untouched) and has kSkipStart as its
// start, so it has no pages.
constexpr int kWarpPlanMaxReqs = 256;
constexpr int32_t kSkipStart = INT32_MIN;

// Exclusive scan with max over the threads' values, in thread order; the
// first thread gets `init`.
template <bool kWarp>
__device__ __forceinline__ int32_t exclusive_max_scan(int32_t x, int32_t init, int32_t* warp_vals) {
  const int tid = kWarp ? static_cast<int>(threadIdx.x & 31) : static_cast<int>(threadIdx.x);
  const int lane = tid & 31;
  int32_t inc = x;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int32_t y = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc = max(inc, y);
  }
  int32_t exc = __shfl_up_sync(0xffffffffu, inc, 1);
  exc = lane == 0 ? init : max(exc, init);
  if constexpr (!kWarp) {
    const int warp = tid >> 5;
    const int nwarps = (static_cast<int>(blockDim.x) + 31) >> 5;
    if (lane == 31) warp_vals[warp] = inc;
    __syncthreads();
    if (warp == 0) {
      int32_t w = lane < nwarps ? warp_vals[lane] : INT32_MIN;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int32_t y = __shfl_up_sync(0xffffffffu, w, o);
        if (lane >= o) w = max(w, y);
      }
      if (lane < nwarps) warp_vals[lane] = w;
    }
    __syncthreads();
    if (warp > 0) exc = max(exc, warp_vals[warp - 1]);
    __syncthreads();
  }
  return exc;
}

template <bool kWarp>
__device__ int build_plan(const Params& p, const PlanView& v, bool report_flags, int* flags_out = nullptr,
                          int32_t* raw_cu = nullptr) {
  __shared__ int32_t warp_sums[32];
  __shared__ int32_t total_pages;
  const int tid = kWarp ? static_cast<int>(threadIdx.x & 31) : static_cast<int>(threadIdx.x);
  const int nt = kWarp ? 32 : static_cast<int>(blockDim.x);
  const int R = p.R;
  const int64_t T = p.T;

  int bad_cu = 0, bad_start = 0;
  const uint64_t keep = evict_last_policy();
  const int32_t carry = (p.carry_in != nullptr) ? ld_meta(p.carry_in, keep) : 0;
  if constexpr (kWarp) {
    // One pass per 32 boundaries, in registers: lane l holds c_r (r = base +
    // l) and m_r; request r - 1 is decided from c_{r-1} and m_{r-1} of the
    // lane before (or of the previous pass).
    int32_t prev_c = 0, prev_m = max(carry, 0), prev_s = 0;
    for (int base = 0; base <= R; base += 32) {
      const int r = base + tid;
      const bool implied = p.implied_end && r == R;  // the last request ends at T
      const int32_t cur32 = (r <= R && !implied) ? ld_meta(p.cu + r, keep) : 0;
      const int32_t start = (r < R && p.ss != nullptr) ? ld_meta(p.ss + r, keep) : 0;
      if (raw_cu != nullptr && r <= R) raw_cu[r] = cur32;
      const int64_t c64 = implied ? T : static_cast<int64_t>(cur32);
      const int32_t c = r <= R ? static_cast<int32_t>(c64 < T ? c64 : T) : INT32_MIN;
      int32_t m = c;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int32_t y = __shfl_up_sync(0xffffffffu, m, o);
        if (tid >= o) m = max(m, y);
      }
      m = max(m, prev_m);
      const int32_t up_c = __shfl_up_sync(0xffffffffu, c, 1);
      const int32_t up_m = __shfl_up_sync(0xffffffffu, m, 1);
      const int32_t up_s = __shfl_up_sync(0xffffffffu, start, 1);
      const int32_t c_prev = tid == 0 ? prev_c : up_c;
      const int32_t m_prev = tid == 0 ? prev_m : up_m;
      const int32_t s_prev = tid == 0 ? prev_s : up_s;
      if (r >= 1 && r <= R) {
        // request r - 1 owns [c_prev, c) under the page's clamp
        const bool has_rows = c > c_prev;
        const bool skip = has_rows && c_prev < m_prev;
        bad_cu |= skip ? 1 : 0;
        bad_start |= (has_rows && !skip && s_prev < 0) ? 1 : 0;
        v.st[r - 1] = skip ? kSkipStart : s_prev;
      }
      if (r <= R) v.ob[r] = m;
      prev_c = __shfl_sync(0xffffffffu, c, 31);
      prev_m = __shfl_sync(0xffffffffu, m, 31);
      prev_s = __shfl_sync(0xffffffffu, start, 31);
    }
    __syncwarp();
  } else {
    // 1. the clamped boundaries c_r into ob and the starts into st; the loads
    // of an entry are issued together
    for (int r = tid; r <= R; r += nt) {
      const bool implied = p.implied_end && r == R;  // the last request ends at T
      const int32_t cur32 = implied ? 0 : ld_meta(p.cu + r, keep);
      const int32_t start = (r < R && p.ss != nullptr) ? ld_meta(p.ss + r, keep) : 0;
      if (raw_cu != nullptr) raw_cu[r] = cur32;
      const int64_t c = implied ? T : static_cast<int64_t>(cur32);
      v.ob[r] = static_cast<int32_t>(c < T ? c : T);
      if (r < R) v.st[r] = start;
    }
    __syncthreads();
    // 2. m_r = max(0, carried boundary, c_0..c_r) into P (scratch for now);
    // each thread owns a contiguous run of boundaries
    const int nb = R + 1;
    const int per_b = (nb + nt - 1) / nt;
    const int bb = min(tid * per_b, nb);
    const int be = min(bb + per_b, nb);
    int32_t run_max = INT32_MIN;
    for (int r = bb; r < be; ++r) run_max = max(run_max, v.ob[r]);
    int32_t m = exclusive_max_scan<false>(run_max, max(carry, 0), warp_sums);
    for (int r = bb; r < be; ++r) {
      m = max(m, v.ob[r]);
      v.P[r] = m;
    }
    __syncthreads();
    // 3. per request: skip the ones with rows below an earlier boundary; flag
    // negative starts of the others
    for (int r = tid; r < R; r += nt) {
      const int32_t c = v.ob[r];
      const bool has_rows = v.ob[r + 1] > c;
      if (has_rows && c < v.P[r]) {
        bad_cu = 1;
        v.st[r] = kSkipStart;
      } else if (has_rows && v.st[r] < 0) {
        bad_start = 1;
      }
    }
    __syncthreads();
    for (int r = bb; r < be; ++r) v.ob[r] = v.P[r];
    __syncthreads();
  }
  if (report_flags && tid == 0 && p.carry_out != nullptr) *p.carry_out = v.ob[R];
  const int per = (R + nt - 1) / nt;
  const int rb = min(tid * per, R);
  const int re = min(rb + per, R);

  // exclusive scan of page counts: each thread owns a contiguous run of requests
  int32_t local = 0;
  for (int r = rb; r < re; ++r) local += request_pages(v, r, p.B);
  const int lane = tid & 31;
  int32_t x = local;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int32_t y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  int32_t base, total;
  if (kWarp) {
    total = __shfl_sync(0xffffffffu, x, 31);
    base = x - local;
  } else {
    const int warp = tid >> 5;
    const int nwarps = (nt + 31) >> 5;
    if (lane == 31) warp_sums[warp] = x;
    __syncthreads();
    if (warp == 0) {
      int32_t w = lane < nwarps ? warp_sums[lane] : 0;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int32_t y = __shfl_up_sync(0xffffffffu, w, o);
        if (lane >= o) w += y;
      }
      if (lane < nwarps) warp_sums[lane] = w;
      if (lane == nwarps - 1) total_pages = w;
    }
    __syncthreads();
    base = (warp > 0 ? warp_sums[warp - 1] : 0) + x - local;
    total = total_pages;
  }
  for (int r = rb; r < re; ++r) {
    v.P[r] = base;
    base += request_pages(v, r, p.B);
  }
  if (tid == 0) v.P[R] = total;
  int flags = 0;
  if (kWarp) {
    __syncwarp();
    flags = (__any_sync(0xffffffffu, bad_cu) ? PMG_FLAG_CU_ORDER : 0) |
            (__any_sync(0xffffffffu, bad_start) ? PMG_FLAG_SEQ_START : 0);
  } else {
    flags = (__syncthreads_or(bad_cu) ? PMG_FLAG_CU_ORDER : 0) | (__syncthreads_or(bad_start) ? PMG_FLAG_SEQ_START : 0);
  }
  if (report_flags && tid == 0) set_flag(p, flags);
  if (flags_out != nullptr) *flags_out = flags;
  return total;
}

// The plan of a single request without seq_starts whose cu_seq_lens is
// [0, T] (or [0] with the implied end): the usual form of a one-request call,
// written without reading anything. The speculative start uses it as its
// guess; the check after the previous grid completes reads cu_seq_lens and
// compares it with raw_cu, so a call whose cu_seq_lens differs replans from
// the real values.
__device__ __forceinline__ int32_t guess_single_plan(const Params& p, const PlanView& v, int32_t* raw_cu) {
  if ((threadIdx.x & 31) == 0) {
    v.ob[0] = 0;
    v.ob[1] = p.T;
    v.st[0] = 0;
    v.P[0] = 0;
    v.P[1] = static_cast<int32_t>((static_cast<uint32_t>(p.T) + static_cast<uint32_t>(p.B) - 1u) /
                                  static_cast<uint32_t>(p.B));
    raw_cu[0] = 0;
    raw_cu[1] = p.implied_end ? 0 : p.T;
  }
  __syncwarp();
  return v.P[1];
}

// Before the previous grid is known to be done, a kernel may not read its
// inputs, but it may warm L2 with them: a prefetch is not a read into
// registers, and L2 is the point of coherence for later loads. The CTAs of
// the launch share the lines out, one prefetch per line (every CTA reads the
// same cu_seq_lens and seq_starts lines, and a line requested by hundreds of
// CTAs at once is a hot spot), block tables up to 4 MB.
__device__ __forceinline__ void prefetch_lines(const void* ptr, int64_t bytes, int64_t first_idx, int64_t step) {
  if (ptr == nullptr || bytes <= 0) return;
  const uintptr_t first = reinterpret_cast<uintptr_t>(ptr) & ~static_cast<uintptr_t>(127);
  const uintptr_t last = (reinterpret_cast<uintptr_t>(ptr) + static_cast<uintptr_t>(bytes) - 1) & ~static_cast<uintptr_t>(127);
  const int64_t lines = static_cast<int64_t>((last - first) / 128) + 1;
  for (int64_t i = first_idx; i < lines; i += step)
    asm volatile("prefetch.global.L2::evict_last [%0];" ::"l"(first + static_cast<uintptr_t>(i) * 128));
}

__device__ __forceinline__ void prefetch_metadata(const Params& p) {
  const int64_t R = p.R;
  if (p.token_mode) {
    // token_to_seq spread over the grid; cu_seq_lens and the block table while small
    prefetch_lines(p.t2s, static_cast<int64_t>(p.T) * 4, static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x,
                   static_cast<int64_t>(gridDim.x) * blockDim.x);
    if ((R + 1) * 4 <= (64ll << 10))
      prefetch_lines(p.cu, (R + 1) * 4, static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x,
                     static_cast<int64_t>(gridDim.x) * blockDim.x);
    const int64_t tb = R * p.bt_stride * 4;
    if (tb <= (4ll << 20))
      prefetch_lines(p.bt, tb, static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x,
                     static_cast<int64_t>(gridDim.x) * blockDim.x);
    return;
  }
  // one prefetch per line across the grid: the lines are shared by every CTA
  const int64_t gtid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t gthreads = static_cast<int64_t>(gridDim.x) * blockDim.x;
  const int64_t cu_n = p.implied_end ? R : R + 1;
  prefetch_lines(p.cu, cu_n * 4, gtid, gthreads);
  prefetch_lines(p.ss, R * 4, gtid, gthreads);
  const int64_t bt_bytes = R * p.bt_stride * 4;
  if (bt_bytes <= (4ll << 20))
    prefetch_lines(p.bt, bt_bytes, static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x,
                   static_cast<int64_t>(gridDim.x) * blockDim.x);
}

struct PageTask {
  int32_t req;
  int64_t logical_block;
  int32_t begin;  // page_token_begin (relative to the page start)
  int32_t end;    // page_token_end (exclusive)
  int32_t out;    // output_token_begin
};

// Flat task id -> page task: binary search over the page-count prefix, then
// the page's clipping of [start, start + len) to logical block lb.
__device__ __forceinline__ PageTask map_task(const PlanView& v, int R, int B, int32_t t) {
  const int r = upper_bound_i32(v.P, R + 1, t) - 1;
  const uint32_t j = static_cast<uint32_t>(t - v.P[r]);
  const int64_t s = v.st[r];
  const int64_t len = static_cast<int64_t>(v.ob[r + 1]) - v.ob[r];
  const uint32_t lb = static_cast<uint32_t>(s) / static_cast<uint32_t>(B) + j;  // s >= 0 for any request with pages
  const int64_t page_begin = static_cast<int64_t>(lb) * B;
  const int64_t cb = s > page_begin ? s : page_begin;
  const int64_t ce = (s + len) < (page_begin + B) ? (s + len) : (page_begin + B);
  PageTask k;
  k.req = r;
  k.logical_block = lb;
  k.begin = static_cast<int32_t>(cb - page_begin);
  k.end = static_cast<int32_t>(ce - page_begin);
  k.out = static_cast<int32_t>(v.ob[r] + (cb - s));
  return k;
}

// First task whose rows reach output row `row` (row inside [ob[0], ob[R])).
__device__ __forceinline__ int32_t first_task_for_row(const PlanView& v, int R, int B, uint32_t row) {
  const int r = upper_bound_i32(v.ob, R + 1, static_cast<int64_t>(row)) - 1;
  const int32_t s = v.st[r];
  if (s < 0) return v.P[r];  // no task in r; the next request's tasks follow
  const uint32_t pos = static_cast<uint32_t>(s) + (row - static_cast<uint32_t>(v.ob[r]));
  return v.P[r] + static_cast<int32_t>(pos / static_cast<uint32_t>(B) - static_cast<uint32_t>(s) / static_cast<uint32_t>(B));
}

// The CTA's share of output rows [row0, row1) and its first task id.
struct CtaRange {
  int32_t row0, row1, t0;
};

__device__ __forceinline__ CtaRange cta_range(const PlanView& v, int R, int B, int32_t num_tasks) {
  CtaRange c;
  // balanced split of [lo, hi): the first `rem` CTAs take one row more
  const uint32_t lo = static_cast<uint32_t>(v.ob[0]);
  const uint32_t rows = static_cast<uint32_t>(v.ob[R]) - lo;
  const uint32_t per = rows / gridDim.x;
  const uint32_t rem = rows - per * gridDim.x;
  const uint32_t b = blockIdx.x;
  c.row0 = static_cast<int32_t>(lo + b * per + (b < rem ? b : rem));
  c.row1 = c.row0 + static_cast<int32_t>(per + (b < rem ? 1u : 0u));
  c.t0 = num_tasks;
  if (c.row0 >= c.row1 || num_tasks <= 0) return c;
  c.t0 = first_task_for_row(v, R, B, static_cast<uint32_t>(c.row0));
  return c;
}

// A clipped, bounds-checked page task: rows [dst_row0, dst_row0 + nrows) of
// dst come from consecutive slots of one physical block.
struct Segment {
  int64_t src;     // byte offset into the cache
  int64_t dst;     // byte offset into dst
  int32_t nrows;   // 0 = nothing to copy
  int32_t pad;
};

// What a speculative resolution read and would have reported.
struct SpecRead {
  int bits;      // flag bits it would set
  int64_t idx;   // block-table element it read, or -1
  int32_t phys;  // the value read there
};

// Resolves task t for a CTA owning rows [row0, row1). Returns false when the
// task starts at or past row1 (tasks are ordered by output row, so every
// later task does too). With rec, flag bits and the block-table read are
// recorded there instead of reported.
__device__ __forceinline__ bool resolve_segment(const Params& p, const PlanView& v, int32_t t, int32_t num_tasks,
                                                int32_t row0, int32_t row1, Segment& seg, SpecRead* rec = nullptr) {
  seg.nrows = 0;
  seg.src = 0;
  seg.dst = 0;
  if (t >= num_tasks) return false;
  const PageTask k = map_task(v, p.R, p.B, t);
  if (k.out >= row1) return false;
  const int64_t lo = k.out > row0 ? k.out : row0;
  const int64_t task_end = static_cast<int64_t>(k.out) + (k.end - k.begin);
  const int64_t hi = task_end < row1 ? task_end : row1;
  if (hi <= lo) return true;
  if (k.logical_block >= p.bt_stride) {
    if (rec != nullptr) rec->bits |= PMG_FLAG_LOGICAL_BLOCK;
    else set_flag(p, PMG_FLAG_LOGICAL_BLOCK);
    return true;
  }
  const int64_t idx = static_cast<int64_t>(k.req) * p.bt_stride + k.logical_block;
  const int64_t phys = ld_meta(p.bt + idx, evict_last_policy());
  if (rec != nullptr) {
    rec->idx = idx;
    rec->phys = static_cast<int32_t>(phys);
  }
  if (phys < 0 || phys >= p.num_blocks) {
    if (rec != nullptr) rec->bits |= PMG_FLAG_PHYS_BLOCK;
    else set_flag(p, PMG_FLAG_PHYS_BLOCK);
    return true;
  }
  const int64_t slot = k.begin + (lo - k.out);
  seg.src = phys * p.blk_stride_b + slot * p.tok_stride_b;
  seg.dst = lo * p.dst_stride_b;
  seg.nrows = static_cast<int32_t>(hi - lo);
  return true;
}

// ---------------------------------------------------------------------------
// TMA bulk path (byte copy, 16-byte aligned rows)
// ---------------------------------------------------------------------------

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Waits for the given phase parity; gives up after kWaitLimitNs.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  uint32_t spins = 0;
  while (!mbar_try_wait(bar, parity)) {
    if ((++spins & 255u) == 0 && global_ns() - t0 > kWaitLimitNs) return false;
  }
  return true;
}

__device__ __forceinline__ uint64_t evict_first_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

__device__ __forceinline__ void bulk_load(void* smem_dst, const void* gsrc, uint32_t bytes, uint64_t* bar,
                                          uint64_t pol) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;"
      ::"r"(smem_addr(smem_dst)), "l"(gsrc), "r"(bytes), "r"(smem_addr(bar)), "l"(pol)
      : "memory");
}

__device__ __forceinline__ void bulk_store(void* gdst, const void* smem_src, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(gdst), "r"(smem_addr(smem_src)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }

__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// Wait until at most n committed bulk-store groups still read shared memory.
__device__ __forceinline__ void bulk_wait_read_upto(int n) {
  static_assert(kMaxStages == 8, "update the cases below");
  switch (n) {
    case 0: asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); break;
    case 1: asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory"); break;
    case 2: asm volatile("cp.async.bulk.wait_group.read 2;" ::: "memory"); break;
    case 3: asm volatile("cp.async.bulk.wait_group.read 3;" ::: "memory"); break;
    case 4: asm volatile("cp.async.bulk.wait_group.read 4;" ::: "memory"); break;
    case 5: asm volatile("cp.async.bulk.wait_group.read 5;" ::: "memory"); break;
    case 6: asm volatile("cp.async.bulk.wait_group.read 6;" ::: "memory"); break;
    default: asm volatile("cp.async.bulk.wait_group.read 7;" ::: "memory"); break;
  }
}

struct Chunk {
  int64_t src;
  int64_t dst;
  int32_t nrows;
  int32_t tentative;  // from the speculative first batch: store only once it is confirmed
};

// Walks a segment table chunk by chunk (at most rows_per_stage rows each).
struct ChunkIter {
  int seg;
  int32_t row;
  __device__ __forceinline__ bool next(const Segment* segs, int nseg, int32_t rows_per_stage, const Params& p,
                                       Chunk& c) {
    while (seg < nseg && row >= segs[seg].nrows) {
      ++seg;
      row = 0;
    }
    if (seg >= nseg) return false;
    const Segment& s = segs[seg];
    const int32_t n = min(rows_per_stage, s.nrows - row);
    c.src = s.src + static_cast<int64_t>(row) * p.tok_stride_b;
    c.dst = s.dst + static_cast<int64_t>(row) * p.dst_stride_b;
    c.nrows = n;
    row += n;
    return true;
  }
};

__device__ __forceinline__ bool mbar_test_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

// ---------------------------------------------------------------------------
// Work items. Without a workspace, CTA c owns one balanced share of the output
// rows (static). With a workspace, item c < G is CTA c's static first share (a
// rows; a quarter of all rows together by default) and items >= G (d rows
// each) are claimed in order through an atomic counter, so CTAs that get their
// data faster take more of the rest; the CTA making a launch's last claim
// resets the counter for the next call.
// ---------------------------------------------------------------------------

// Largest grid for which tilted static shares are computed (the numerator of
// tilted_prefix stays exact in 64 bits); larger grids split evenly.
constexpr uint32_t kTiltMaxGrid = 2048;

struct Items {
  uint32_t lo, hi;  // output rows [lo, hi)
  uint32_t a, d;    // static share and dynamic item size
  uint32_t n;       // number of items
  uint32_t tilt;    // percent: static shares tilted towards low blockIdx (0: even)
  uint32_t tilt_pow;
  bool dynamic;
};

// Dynamic mode needs a workspace and enough rows per CTA for the claims to
// pay off. Each CTA's static share is sched_static_pct % of its rows, but at
// least sched_head_stages ring stages (or all of its rows): the static item
// starts the moment the launch may read the cache, while a claimed item waits
// for its claim, so a CTA needs a static head start covering that latency
// (four stages for a page gather, two in token mode; the host sets them from
// measurements). Dynamic items are
// about rows / (64 G) rows and never smaller than one ring stage: small items
// even out the CTAs' finishing times (single-300K 0.975 -> 0.988), but an item
// must carry more data than the claim and block-table round trips that fetch
// it (half-stage items lost 10% on single-60K). Token mode resolves an item
// through three dependent round trips instead of one and keeps items four
// times larger (rows / (16 G)).
__device__ __forceinline__ Items make_items(const PlanView& v, const Params& p) {
  Items it;
  it.lo = p.token_mode ? 0u : static_cast<uint32_t>(v.ob[0]);
  it.hi = p.token_mode ? static_cast<uint32_t>(p.T) : static_cast<uint32_t>(v.ob[p.R]);
  const uint32_t rows = it.hi - it.lo;
  const uint32_t G = gridDim.x;
  const bool big = rows / G >= static_cast<uint32_t>(p.sched_min_rows);
  const uint32_t rps = static_cast<uint32_t>(p.rows_per_stage > 0 ? p.rows_per_stage : 1);
  const uint32_t hs = static_cast<uint32_t>(p.sched_head_stages) * rps;
  it.dynamic = p.sched != nullptr && big;
  if (it.dynamic) {
    it.a = static_cast<uint32_t>(static_cast<uint64_t>(rows) * static_cast<uint32_t>(p.sched_static_pct) / 100u / G);
    const uint32_t head = hs < rows / G ? hs : rows / G;
    if (it.a < head) it.a = head;
    const uint32_t d = rows / ((p.token_mode ? 16u : 64u) * G);
    it.d = d > rps ? d : rps;
    const uint32_t rest = rows - G * it.a;
    it.n = G + (rest + it.d - 1u) / it.d;
  } else {
    it.a = it.d = 0;
    it.n = G;
  }
  // The tilt only where claims cannot even out the finishing times: fewer
  // dynamic items than CTAs, or a static split of at most the head plus one
  // stage per CTA (the late CTAs' lag is a few microseconds whatever the
  // launch's length, so longer static launches keep even shares). And only
  // where CTAs hold enough rows for their start-up not to dominate. Shares
  // stay >= 0 (F increasing) while tilt * pow <= 100.
  const bool few = it.dynamic ? it.n - G < G : rows / G < hs + rps;
  it.tilt_pow = p.sched_tilt_pow >= 1 && p.sched_tilt_pow <= 4 ? static_cast<uint32_t>(p.sched_tilt_pow) : 1u;
  const uint32_t tmax = 100u / it.tilt_pow;
  const uint32_t t = static_cast<uint32_t>(p.sched_tilt_pct);
  it.tilt = (G <= kTiltMaxGrid && big && few) ? (t < tmax ? t : tmax) : 0u;
  return it;
}

// Rows before CTA k when `total` rows are split over G CTAs with shares
// 1 + t (1 - (q + 1) x^q) of the even share (x = k / G, t = tilt / 100,
// q = pow in 1..4): about total * F(k / G) with F(x) = x + t (x - x^(q+1)).
// q = 1 falls linearly from 1 + t to 1 - t; larger q keep the shares near
// 1 + t longer and drop them towards the last CTAs. The numerator
// k (100 G^q + tilt (G^q - k^q)) is exact in 64 bits for G <= 2048 and grows
// with k; scaling it in single precision keeps that order (rounding is
// monotone), k = G gives the total, and CTA k's end and CTA k + 1's start are
// the same call: the ranges are contiguous, in order and cover every row once.
__device__ __forceinline__ uint32_t tilted_prefix(uint32_t total, uint32_t k, uint32_t G, uint32_t tilt,
                                                  uint32_t pw) {
  if (k >= G) return total;
  uint64_t gq = G, kq = k;
  for (uint32_t i = 1; i < pw; ++i) {
    gq *= G;
    kq *= k;
  }
  const uint64_t num = static_cast<uint64_t>(k) * (gq * 100u + static_cast<uint64_t>(tilt) * (gq - kq));
  const float scale = static_cast<float>(total) / (static_cast<float>(gq) * static_cast<float>(G) * 100.0f);
  const float x = static_cast<float>(num) * scale;
  const uint32_t v = x >= static_cast<float>(total) ? total : static_cast<uint32_t>(x);
  return v < total ? v : total;
}

__device__ __forceinline__ void item_rows(const Items& it, uint32_t k, uint32_t& r0, uint32_t& r1) {
  const uint32_t G = gridDim.x;
  if (it.tilt != 0u && k < G) {
    // CTAs start in blockIdx order as the previous grid's CTAs leave: the
    // late ones get less of the static rows
    const uint32_t total = it.dynamic ? G * it.a : it.hi - it.lo;
    r0 = it.lo + tilted_prefix(total, k, G, it.tilt, it.tilt_pow);
    r1 = it.lo + tilted_prefix(total, k + 1u, G, it.tilt, it.tilt_pow);
  } else if (!it.dynamic) {
    const uint32_t rows = it.hi - it.lo;
    const uint32_t per = rows / G;
    const uint32_t rem = rows - per * G;
    r0 = it.lo + k * per + (k < rem ? k : rem);
    r1 = r0 + per + (k < rem ? 1u : 0u);
  } else if (k < G) {
    r0 = it.lo + k * it.a;
    r1 = r0 + it.a;
  } else {
    r0 = it.lo + G * it.a + (k - G) * it.d;
    r1 = r0 + it.d < it.hi ? r0 + it.d : it.hi;
  }
}

// Per-token gather: output token t reads request b = t2s[t] at context position
// t - cu[b]; every index is checked before use. One lane resolves the tokens
// t_first + 32 j (j < N, those below t_end) with the loads of each step issued
// together: t2s, then cu, then the block table. src[j] is the source byte
// offset of the row, or -1 (flag bits in `bits`; tokens at or past t_end set none).
constexpr int kTokGroup = 4;

// What the resolution of one token read (for the speculative start's check).
struct TokRead {
  int32_t b;    // token_to_seq[t] as read
  int32_t c0;   // cu_seq_lens[b] and [b + 1], when b was in range
  int32_t c1;
  int32_t phys; // the block-table entry read, at idx (or idx = -1)
  int64_t idx;
};

template <int N>
__device__ __forceinline__ void resolve_tokens(const Params& p, uint32_t t_first, uint32_t t_end, int64_t (&src)[N],
                                               int& bits, TokRead (&rec)[N]) {
  const uint64_t keep = evict_last_policy();
  int32_t b[N];
#pragma unroll
  for (int j = 0; j < N; ++j) {
    const uint32_t t = t_first + 32u * j;
    src[j] = -1;
    b[j] = t < t_end ? ld_meta(p.t2s + t, keep) : -1;
    rec[j] = TokRead{b[j], 0, 0, 0, -1};
    if (t < t_end && (b[j] < 0 || b[j] >= p.R)) {
      bits |= PMG_FLAG_TOKEN;
      b[j] = -1;
    }
  }
  int32_t c0[N], c1[N];
#pragma unroll
  for (int j = 0; j < N; ++j) {
    c0[j] = b[j] >= 0 ? ld_meta(p.cu + b[j], keep) : 0;
    c1[j] = b[j] >= 0 ? ld_meta(p.cu + b[j] + 1, keep) : 0;
    rec[j].c0 = c0[j];
    rec[j].c1 = c1[j];
  }
  int32_t phys[N];
  uint32_t off[N];
#pragma unroll
  for (int j = 0; j < N; ++j) {
    const int64_t t = static_cast<int64_t>(t_first) + 32 * j;
    phys[j] = -1;
    off[j] = 0;
    if (b[j] < 0) continue;
    if (t < c0[j] || t >= c1[j]) {
      bits |= PMG_FLAG_TOKEN;
      b[j] = -1;
      continue;
    }
    const uint32_t pos = static_cast<uint32_t>(t - c0[j]);
    const uint32_t lb = pos / static_cast<uint32_t>(p.B);
    off[j] = pos - lb * static_cast<uint32_t>(p.B);
    if (static_cast<int64_t>(lb) >= p.bt_stride) {
      bits |= PMG_FLAG_LOGICAL_BLOCK;
      b[j] = -1;
      continue;
    }
    rec[j].idx = static_cast<int64_t>(b[j]) * p.bt_stride + lb;
    phys[j] = ld_meta(p.bt + rec[j].idx, keep);
    rec[j].phys = phys[j];
  }
#pragma unroll
  for (int j = 0; j < N; ++j) {
    if (b[j] < 0) continue;
    if (phys[j] < 0 || phys[j] >= p.num_blocks) {
      bits |= PMG_FLAG_PHYS_BLOCK;
      continue;
    }
    src[j] = static_cast<int64_t>(phys[j]) * p.blk_stride_b + static_cast<int64_t>(off[j]) * p.tok_stride_b;
  }
}

// Whether the inputs of tokens t_first + 32 j (j < N, below t_end) still hold
// what rec recorded. The loads go to the recorded addresses and are all
// issued before any comparison.
template <int N>
__device__ __forceinline__ bool tokens_unchanged(const Params& p, uint32_t t_first, uint32_t t_end,
                                                 const TokRead (&rec)[N]) {
  const uint64_t keep = evict_last_policy();
  int32_t b[N], c0[N], c1[N], ph[N];
#pragma unroll
  for (int j = 0; j < N; ++j) {
    const uint32_t t = t_first + 32u * j;
    const bool in = rec[j].b >= 0 && rec[j].b < p.R;
    b[j] = t < t_end ? ld_meta(p.t2s + t, keep) : rec[j].b;
    c0[j] = (t < t_end && in) ? ld_meta(p.cu + rec[j].b, keep) : rec[j].c0;
    c1[j] = (t < t_end && in) ? ld_meta(p.cu + rec[j].b + 1, keep) : rec[j].c1;
    ph[j] = (t < t_end && rec[j].idx >= 0) ? ld_meta(p.bt + rec[j].idx, keep) : rec[j].phys;
  }
  bool same = true;
#pragma unroll
  for (int j = 0; j < N; ++j)
    same = same && b[j] == rec[j].b && c0[j] == rec[j].c0 && c1[j] == rec[j].c1 && ph[j] == rec[j].phys;
  return same;
}

// Segment batches handed from the scheduler warp to the producer thread.
constexpr int kSegBufs = 2;
constexpr int kSegCap = 32;

struct SegQueue {
  Segment seg[kSegBufs][kSegCap];
  int32_t count[kSegBufs];  // -1: no more work
  uint64_t full[kSegBufs];
  uint64_t empty[kSegBufs];
  int32_t tentative;  // batch 0 is the speculative first batch
  int32_t verdict;    // for it: 0 pending, 1 confirmed, 2 withdrawn
  // The batch published before the previous grid completes, handed to a warp
  // that warms L2 with its rows (the scheduler warp goes on to its check):
  // pf_state 0 pending, 1 pf_seg holds pf_n segments, 2 nothing to warm.
  Segment pf_seg[kSegCap];
  int32_t pf_n;
  int32_t pf_state;
};

__device__ __forceinline__ void segq_init(SegQueue& q) {
  for (int b = 0; b < kSegBufs; ++b) {
    mbar_init(&q.full[b], 1);
    mbar_init(&q.empty[b], 1);
  }
  q.tentative = 0;
  q.verdict = 0;
  q.pf_state = 0;
}

// Scheduler warp: hands the batch just published in slot b to the warming warp.
__device__ __forceinline__ void hand_off_prefetch(SegQueue& q, int b) {
  const int lane = threadIdx.x & 31;
  const int n = q.count[b];
  if (lane < n) q.pf_seg[lane] = q.seg[b][lane];
  if (lane == 0) q.pf_n = n;
  __syncwarp();
  if (lane == 0) {
    __threadfence_block();
    *reinterpret_cast<volatile int32_t*>(&q.pf_state) = 1;
  }
}

// Scheduler warp, after the wait: nothing (more) will be handed off.
__device__ __forceinline__ void pf_release(SegQueue& q) {
  if ((threadIdx.x & 31) == 0 && *reinterpret_cast<volatile int32_t*>(&q.pf_state) == 0)
    *reinterpret_cast<volatile int32_t*>(&q.pf_state) = 2;
}

// Verdict on the speculative first batch: 1 confirmed, 0 withdrawn, -1 the
// bounded wait for it ran out.
__device__ __forceinline__ int spec_verdict(const SegQueue& q) {
  const volatile int32_t* vp = &q.verdict;
  int32_t v = *vp;
  if (v == 0) {
    const uint64_t t0 = global_ns();
    while ((v = *vp) == 0) {
      if (global_ns() - t0 > kWaitLimitNs) return -1;
    }
  }
  return v == 1 ? 1 : 0;
}

// Warms L2 (and the address translation) with the source rows of a batch
// published before the wait, at most cap rows in segment order, the lines
// spread over the warp's lanes. A prefetch reads nothing into registers: if
// the previous grid still writes those rows, the loads after the wait read
// them as they are then, and rows of a withdrawn batch are only wasted
// bandwidth. Every address is inside a row the batch's checks accepted.
__device__ __forceinline__ void prefetch_rows(const Params& p, const Segment* segs, int n, int32_t cap) {
  const int lane = threadIdx.x & 31;
  const uint32_t rb = static_cast<uint32_t>(p.row_src_bytes);
  const uint32_t lpr = (rb + 127u) / 128u;  // lines a row touches from its start
  for (int i = 0; i < n && cap > 0; ++i) {
    const Segment sg = segs[i];
    const int32_t rows = sg.nrows < cap ? sg.nrows : cap;
    cap -= rows;
    const uint32_t units = static_cast<uint32_t>(rows) * lpr;
    for (uint32_t u = static_cast<uint32_t>(lane); u < units; u += 32u) {
      const uint32_t row = u / lpr;
      const uint32_t line = u - row * lpr;
      const uint32_t off = line * 128u < rb ? line * 128u : rb - 1u;
      const uint8_t* a = p.cache + sg.src + static_cast<int64_t>(row) * p.tok_stride_b + off;
      asm volatile("prefetch.global.L2 [%0];" ::"l"(a));
    }
  }
}

// The warming warp (a warp with nothing to do before the wait): waits, within
// the bounded time, for the scheduler's hand-off and prefetches up to
// p.prefetch_rows rows of the handed batch. Issuing the prefetches here keeps
// them off the scheduler warp, whose check after the wait gates the first
// stores.
__device__ __forceinline__ void prefetch_helper(const Params& p, const SegQueue& q) {
  const volatile int32_t* sp = &q.pf_state;
  int32_t st = *sp;
  if (st == 0) {
    const uint64_t t0 = global_ns();
    while ((st = *sp) == 0) {
      if (global_ns() - t0 > kWaitLimitNs) return;
    }
  }
  __threadfence_block();
  if (st == 1 && p.prefetch_rows > 0) prefetch_rows(p, q.pf_seg, q.pf_n, p.prefetch_rows);
}

// The check of a speculative start (uses is 0): publishes the first batch
// marked tentative when `publish`, waits for the previous grid, then reads
// again every input the speculative plan sv read (cu_seq_lens as kept in
// raw_cu, seq_starts) and, for a published batch, the block-table entry each
// lane read, all in one round trip, and compares. Returns whether everything
// still holds; for a published batch the verdict goes to the producer.
__device__ __forceinline__ bool spec_confirm(const Params& p, const PlanView& sv, const int32_t* raw_cu, SegQueue& q,
                                             const Segment& seg, int n, const SpecRead& rd, bool publish,
                                             uint32_t& uses) {
  const int lane = threadIdx.x & 31;
  if (publish) {
    q.seg[0][lane] = seg;
    if (lane == 0) {
      q.count[0] = n;
      q.tentative = 1;
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&q.full[0]);
    uses = 1;
    hand_off_prefetch(q, 0);
  }
  pdl_wait();
  pf_release(q);
  const uint64_t keep = evict_last_policy();
  const int32_t phys_now = (publish && rd.idx >= 0) ? ld_meta(p.bt + rd.idx, keep) : 0;
  bool same = !publish || rd.idx < 0 || phys_now == rd.phys;
  for (int base = 0; base <= p.R; base += 128) {
    int32_t c[4], st[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int r = base + 32 * j + lane;
      const bool implied = p.implied_end && r == p.R;
      c[j] = (r <= p.R && !implied) ? ld_meta(p.cu + r, keep) : 0;
      st[j] = (r < p.R && p.ss != nullptr) ? ld_meta(p.ss + r, keep) : 0;
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int r = base + 32 * j + lane;
      if (r <= p.R) same = same && c[j] == raw_cu[r];
      if (r < p.R) same = same && st[j] == sv.st[r];
    }
  }
  const bool valid = __all_sync(0xffffffffu, same);
  if (publish && lane == 0) *reinterpret_cast<volatile int32_t*>(&q.verdict) = valid ? 1 : 2;
  return valid;
}

// Publishes the 32 tokens t0 + lane (row source offset src, -1 for none) as
// one batch: consecutive lanes whose source rows are one slot apart form one
// segment. Returns the number of segments (0: nothing to publish) or -1 when
// the bounded wait for a free batch ran out.
__device__ __forceinline__ int publish_tokens(const Params& p, SegQueue& q, uint32_t& uses, uint32_t t0,
                                              int64_t src) {
  const int lane = threadIdx.x & 31;
  const int64_t prev = __shfl_up_sync(0xffffffffu, src, 1);
  const bool valid = src >= 0;
  const bool cont = lane > 0 && valid && prev >= 0 && src == prev + p.tok_stride_b;
  const bool start = valid && !cont;
  const uint32_t starts = __ballot_sync(0xffffffffu, start);
  const uint32_t breaks = __ballot_sync(0xffffffffu, !cont);
  const int n = __popc(starts);
  if (n == 0) return 0;
  const int b = static_cast<int>(uses % kSegBufs);
  if (uses >= kSegBufs && !mbar_wait_bounded(&q.empty[b], ((uses / kSegBufs) - 1u) & 1u)) return -1;
  if (start) {
    // the segment runs to the next lane that starts one or is empty
    const uint32_t after = lane == 31 ? 0u : (breaks & (0xffffffffu << (lane + 1)));
    const int next = after ? __ffs(after) - 1 : 32;
    Segment seg;
    seg.src = src;
    seg.dst = static_cast<int64_t>(t0 + static_cast<uint32_t>(lane)) * p.dst_stride_b;
    seg.nrows = next - lane;
    seg.pad = 0;
    q.seg[b][__popc(starts & ((1u << lane) - 1u))] = seg;
  }
  if (lane == 0) q.count[b] = n;
  __syncwarp();
  if (lane == 0) mbar_arrive(&q.full[b]);
  ++uses;
  return n;
}

// The scheduler warp: takes items (its static one, then claimed ones) and
// resolves each into batches of up to 32 segments, one task per lane (map,
// block-table read, bounds checks). Returns false on a timeout.
//
// Speculative start (p.spec, warp plans only): before the previous grid is
// known to be done, the warp plans into the spare area sv (keeping the raw
// cu_seq_lens values it read) and resolves the first batch of its static item,
// reporting nothing, and publishes that batch marked tentative, so that the
// producer can start its loads the moment the wait returns (loads only read
// the cache, at addresses checked in bounds). After the wait it reads every
// input the plan and the batch used again, in one round trip, and compares:
// if all agree, the plan and the batch are what they would have been after the
// wait, the batch is confirmed and sv becomes the plan; otherwise the batch is
// withdrawn (its chunks are dropped unstored) and the warp plans again into v
// and resolves the item from the start. A kernel that starts after other work
// runs its code cold in the instruction caches, so the check is a short loop
// rather than a second run of the plan. The per-token mode does the same with
// its first 32 tokens, checking every input they read.
__device__ bool run_scheduler(const Params& p, const PlanView& v, const PlanView& sv, int32_t num_tasks,
                              SegQueue& q) {
  const int lane = threadIdx.x & 31;
  uint32_t uses = 0;
  uint32_t k = blockIdx.x;
  PlanView pv = v;           // the plan in use
  bool spec_first = false;   // pv is the speculative plan; its first batch is still to be checked
  int32_t* raw_cu = nullptr;
  bool tok_spec = false;     // token mode: the first group of the static item is to be checked
  if (p.spec && p.token_mode) {
    tok_spec = true;
  } else if (p.spec) {
    raw_cu = sv.P + (p.R + 1);
    int plan_flags = 0;
    const int32_t sn = (p.spec_guess && p.R == 1 && p.ss == nullptr && p.T > 0) ? guess_single_plan(p, sv, raw_cu)
                                                                  : build_plan<true>(p, sv, false, &plan_flags, raw_cu);
    if (sn > 0 && plan_flags == 0) {
      // the main loop resolves the first batch from this plan and checks both
      pv = sv;
      num_tasks = sn;
      spec_first = true;
    } else {
      pdl_wait();
      pf_release(q);
      num_tasks = build_plan<true>(p, v, blockIdx.x == 0);
    }
  }
  if (!p.spec && !p.early) pf_release(q);
  // the work items live in shared memory (only this warp reads them): fewer
  // registers held across the loop
  __shared__ Items its;
  bool have = false;
  if (num_tasks > 0) {
    const Items t = make_items(pv, p);
    if (lane == 0) its = t;
    __syncwarp();
    have = k < t.n;
  }
  // with early metadata or a speculative start the workspace (claim counter)
  // is touched only after the previous grid is done: wait after the first
  // published batch
  bool waited = p.early == 0 && !spec_first && !tok_spec;
  while (have) {
    // claim the next item now; its latency overlaps this item's resolution
    uint32_t claimed = 0;
    if (its.dynamic && lane == 0 && waited) claimed = gridDim.x + atomicAdd(reinterpret_cast<unsigned*>(p.sched), 1u);
    uint32_t r0, r1;
    item_rows(its, k, r0, r1);
    bool replan = false;
    if (r0 < r1 && p.token_mode) {
      // 32 tokens per batch, one per lane, kTokGroup batches resolved together
      for (uint32_t g0 = r0; g0 < r1; g0 += 32u * kTokGroup) {
        int64_t srcs[kTokGroup];
        TokRead rec[kTokGroup];
        int bits = 0;
        resolve_tokens<kTokGroup>(p, g0 + static_cast<uint32_t>(lane), r1, srcs, bits, rec);
        int first = 0;  // batches of this group already published
        if (tok_spec) {
          // speculative start: the group's first batch goes out tentatively
          // (unless the group would report a flag); after the wait every input
          // the group read is read again in one round trip and compared
          tok_spec = false;
          waited = true;
          const bool publish = __all_sync(0xffffffffu, bits == 0) && __any_sync(0xffffffffu, srcs[0] >= 0);
          if (publish) {
            if (lane == 0) q.tentative = 1;
            (void)publish_tokens(p, q, uses, g0, srcs[0]);  // the first batch: no wait
            __syncwarp();
            if (uses == 1) hand_off_prefetch(q, 0);
          }
          pdl_wait();
          pf_release(q);
          const bool valid = __all_sync(0xffffffffu, tokens_unchanged<kTokGroup>(p, g0 + static_cast<uint32_t>(lane),
                                                                                   r1, rec));
          if (publish && lane == 0) *reinterpret_cast<volatile int32_t*>(&q.verdict) = valid ? 1 : 2;
          if (its.dynamic && lane == 0) claimed = gridDim.x + atomicAdd(reinterpret_cast<unsigned*>(p.sched), 1u);
          if (!valid) {
            // inputs changed: resolve the group again (the tentative batch is withdrawn)
            g0 -= 32u * kTokGroup;
            continue;
          }
          if (publish) first = 1;
        }
        if (bits != 0) set_flag(p, bits);
#pragma unroll
        for (int j = 0; j < kTokGroup; ++j) {
          if (j < first) continue;
          if (uses >= kSegBufs && !waited) {
            // Before the wait only the free batches may be filled: waiting
            // for the producer to free one would mean waiting for the
            // previous grid through a bounded wait. The wait (and this
            // item's claim) comes first.
            pdl_wait();
            pf_release(q);
            waited = true;
            if (its.dynamic && lane == 0) claimed = gridDim.x + atomicAdd(reinterpret_cast<unsigned*>(p.sched), 1u);
          }
          if (publish_tokens(p, q, uses, g0 + 32u * j, srcs[j]) < 0) return false;
        }
      }
    } else if (r0 < r1 && !p.token_mode) {
      int32_t t = first_task_for_row(pv, p.R, p.B, r0);
      for (;;) {
        Segment seg;
        SpecRead rd{0, -1, 0};
        const bool act = resolve_segment(p, pv, t + lane, num_tasks, static_cast<int32_t>(r0),
                                         static_cast<int32_t>(r1), seg, spec_first ? &rd : nullptr);
        const int n = __popc(__ballot_sync(0xffffffffu, act));
        if (spec_first) {
          // the first batch of a speculative start: published tentatively
          // (unless it would report a flag), then checked after the wait
          spec_first = false;
          waited = true;
          const bool publish = n > 0 && __all_sync(0xffffffffu, rd.bits == 0);
          if (!spec_confirm(p, sv, raw_cu, q, seg, n, rd, publish, uses)) {
            replan = true;
            break;
          }
          if (its.dynamic && lane == 0) claimed = gridDim.x + atomicAdd(reinterpret_cast<unsigned*>(p.sched), 1u);
          if (!publish) continue;  // the plan holds: resolve this batch again, reporting
          if (n < kSegCap) break;
          t += kSegCap;
          continue;
        }
        if (n == 0) break;
        if (uses >= kSegBufs && !waited) {
          // as in token mode: no wait on the producer before the wait
          pdl_wait();
          pf_release(q);
          waited = true;
          if (its.dynamic && lane == 0) claimed = gridDim.x + atomicAdd(reinterpret_cast<unsigned*>(p.sched), 1u);
        }
        const int b = static_cast<int>(uses % kSegBufs);
        if (uses >= kSegBufs && !mbar_wait_bounded(&q.empty[b], ((uses / kSegBufs) - 1u) & 1u)) return false;
        q.seg[b][lane] = seg;
        if (lane == 0) q.count[b] = n;
        __syncwarp();
        if (lane == 0) mbar_arrive(&q.full[b]);
        ++uses;
        if (!waited && uses == 1) hand_off_prefetch(q, b);  // early metadata
        if (n < kSegCap) break;
        t += kSegCap;
      }
    }
    tok_spec = false;  // an empty static item leaves nothing to check
    if (spec_first && !replan) {
      // the static item gave no batch to check: check the plan alone
      spec_first = false;
      waited = true;
      if (!spec_confirm(p, sv, raw_cu, q, Segment{}, 0, SpecRead{0, -1, 0}, false, uses)) replan = true;
      else if (its.dynamic && lane == 0) claimed = gridDim.x + atomicAdd(reinterpret_cast<unsigned*>(p.sched), 1u);
    }
    if (replan) {
      // the inputs changed under the speculative plan: plan again and start
      // over from the static item (no claim was made yet)
      num_tasks = build_plan<true>(p, v, blockIdx.x == 0);
      pv = v;
      k = blockIdx.x;
      have = false;
      if (num_tasks > 0) {
        const Items t = make_items(pv, p);
        __syncwarp();
        if (lane == 0) its = t;
        __syncwarp();
        have = k < t.n;
      }
      continue;
    }
    if (!waited) {
      pdl_wait();
      pf_release(q);
      waited = true;
      if (its.dynamic && lane == 0) claimed = gridDim.x + atomicAdd(reinterpret_cast<unsigned*>(p.sched), 1u);
    }
    if (its.dynamic) {
      k = __shfl_sync(0xffffffffu, claimed, 0);
      have = k < its.n;
      // Every CTA claims until a claim fails, so a launch makes exactly n
      // claims in all (n - G that succeed, one failing claim per CTA). The CTA
      // holding the n-th claim is the last to touch the counter: it resets
      // the workspace for the next call.
      if (lane == 0 && k - gridDim.x == its.n - 1u) atomicExch(reinterpret_cast<unsigned*>(p.sched), 0u);
    } else {
      have = false;
    }
  }
  if (!waited) pdl_wait();
  pf_release(q);
  const int b = static_cast<int>(uses % kSegBufs);
  if (uses >= kSegBufs && !mbar_wait_bounded(&q.empty[b], ((uses / kSegBufs) - 1u) & 1u)) return false;
  if (lane == 0) q.count[b] = -1;
  __syncwarp();
  if (lane == 0) mbar_arrive(&q.full[b]);
  return true;
}

// Producer-side reader of the segment batches, chunk by chunk.
struct SegReader {
  uint32_t uses;
  int cur;
  int n;
  ChunkIter it;
  bool end;
  int32_t tentative;
  // 1: a chunk; 0: none ready yet (only when block is false); -1: no more work;
  // -2: a bounded wait ran out
  __device__ __forceinline__ int next(SegQueue& q, const Params& p, Chunk& c, bool block) {
    for (;;) {
      if (cur >= 0) {
        if (it.next(q.seg[cur], n, p.rows_per_stage, p, c)) {
          c.tentative = tentative;
          return 1;
        }
        mbar_arrive(&q.empty[cur]);  // chunk descriptors are copied out: the batch is free
        ++uses;
        cur = -1;
      }
      if (end) return -1;
      const int b = static_cast<int>(uses % kSegBufs);
      const uint32_t par = (uses / kSegBufs) & 1u;
      if (!block) {
        if (!mbar_test_wait(&q.full[b], par)) return 0;
      } else if (!mbar_wait_bounded(&q.full[b], par)) {
        end = true;
        return -2;
      }
      n = q.count[b];
      if (n < 0) {
        end = true;
        return -1;
      }
      cur = b;
      it = ChunkIter{0, 0};
      tentative = (uses == 0 && q.tentative) ? 1 : 0;
    }
  }
};

__device__ __forceinline__ void issue_loads(const Params& p, const Chunk& c, uint8_t* buf, uint64_t* bar,
                                            uint64_t pol) {
  const uint32_t row_bytes = static_cast<uint32_t>(p.row_src_bytes);
  const uint32_t bytes = static_cast<uint32_t>(c.nrows) * row_bytes;
  mbar_arrive_expect_tx(bar, bytes);
  if (p.src_dense) {
    bulk_load(buf, p.cache + c.src, bytes, bar, pol);
  } else {
    for (int32_t i = 0; i < c.nrows; ++i)
      bulk_load(buf + static_cast<size_t>(i) * row_bytes, p.cache + c.src + i * p.tok_stride_b, row_bytes, bar, pol);
  }
}

// Byte copy: warp 0 lane 0 loads chunks into a ring of p.stages stages (at most kMaxStages) and
// stores each landed stage straight back out; warp 1 schedules.
__global__ void __launch_bounds__(kBulkThreads) gather_bulk_kernel(const __grid_constant__ Params p) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ __align__(8) uint64_t full_bar[kMaxStages];
  __shared__ Chunk stage_chunk[kMaxStages];
  __shared__ __align__(8) SegQueue q;

  // layout: [stages][plan][speculative plan]; stage buffers first keeps them 128-byte aligned
  uint8_t* stage_base = smem;
  const PlanView v = plan_view(smem + static_cast<size_t>(p.stages) * p.stage_bytes, p);
  // the speculative plan's area follows the plan (allocated only with p.spec)
  const PlanView sv = plan_view(smem + static_cast<size_t>(p.stages) * p.stage_bytes + plan_bytes(p), p);

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  // nothing before the PDL wait reads an input: barrier set-up, L2 prefetch
  if (tid == 0) {
    for (int s = 0; s < p.stages; ++s) mbar_init(&full_bar[s], 1);
    segq_init(q);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  prefetch_metadata(p);
  pdl_trigger();
  // With early metadata or speculation the scheduler warp plans and resolves
  // its first batch while the previous grid may still run; every read of the
  // cache, scale or workspace and every write of dst comes after the wait.
  const bool early = p.early != 0 || p.spec != 0;
  if (!early) pdl_wait();
  __syncthreads();
  // small batches: the scheduler warp plans alone; large ones: the whole CTA;
  // the per-token gather needs no plan
  const bool warp_plan = p.R <= kWarpPlanMaxReqs || p.token_mode;
  int32_t num_tasks = 0;
  if (!warp_plan) {
    num_tasks = build_plan<false>(p, v, blockIdx.x == 0);
    if (num_tasks <= 0) return;
  }

  if (warp == 1) {
    if (p.token_mode) num_tasks = 1;
    else if (warp_plan && !p.spec) num_tasks = build_plan<true>(p, v, blockIdx.x == 0);
    if (!run_scheduler(p, v, sv, num_tasks, q)) set_flag(p, PMG_FLAG_TIMEOUT);
  } else if (warp == 2) {
    if (early) prefetch_helper(p, q);
  } else if (tid == 0) {
    if (early) pdl_wait();
    const uint64_t pol = evict_first_policy();
    const uint32_t row_bytes = static_cast<uint32_t>(p.row_src_bytes);
    const uint32_t S = static_cast<uint32_t>(p.stages);
    SegReader rd{0, -1, 0, ChunkIter{0, 0}, false, 0};
    uint32_t loads = 0, stores = 0;
    bool gen_done = false;
    bool ok = true;
    for (;;) {
      // keep up to p.stages chunks loading ahead of the stores
      while (!gen_done && loads - stores < S) {
        Chunk c;
        const int r = rd.next(q, p, c, loads == stores);
        if (r == 0) break;
        if (r < 0) {
          gen_done = true;
          if (r == -2) ok = false;
          break;
        }
        const int s = static_cast<int>(loads % S);
        if (loads >= S) {
          // the store that last used stage s must have finished reading it
          bulk_wait_read_upto(static_cast<int>(stores - 1 - (loads - S)));
        }
        stage_chunk[s] = c;
        issue_loads(p, c, stage_base + static_cast<size_t>(s) * p.stage_bytes, &full_bar[s], pol);
        ++loads;
      }
      if (stores == loads) {
        if (gen_done) break;
        continue;
      }
      const int s = static_cast<int>(stores % S);
      if (!mbar_wait_bounded(&full_bar[s], (stores / S) & 1u)) {
        ok = false;
        break;
      }
      const Chunk c = stage_chunk[s];
      if (c.tentative) {
        const int vr = spec_verdict(q);
        if (vr != 1) {
          // withdrawn (or no verdict in time): drop the chunk; an empty group
          // keeps the count of bulk groups in step with `stores`
          if (vr < 0) set_flag(p, PMG_FLAG_TIMEOUT);
          bulk_commit();
          ++stores;
          continue;
        }
      }
      const uint8_t* buf = stage_base + static_cast<size_t>(s) * p.stage_bytes;
      if (p.dst_dense) {
        bulk_store(p.dst + c.dst, buf, static_cast<uint32_t>(c.nrows) * row_bytes);
      } else {
        for (int32_t i = 0; i < c.nrows; ++i)
          bulk_store(p.dst + c.dst + i * p.dst_stride_b, buf + static_cast<size_t>(i) * row_bytes, row_bytes);
      }
      bulk_commit();
      ++stores;
    }
    if (!ok) {
      // a wait ran out: report, give the loads in flight a bounded chance to
      // land, then stop
      set_flag(p, PMG_FLAG_TIMEOUT);
      for (uint32_t k = stores + 1; k < loads; ++k)
        (void)mbar_wait_bounded(&full_bar[k % S], (k / S) & 1u);
    }
    bulk_wait_all();
  }
  __syncthreads();
}

// ---------------------------------------------------------------------------
// SIMT path: converts and layouts the bulk path does not take
// ---------------------------------------------------------------------------

// Raw storage of one access: BYTES bytes in whole 32-bit words (or a sub-word).
template <int BYTES>
struct Raw {
  static constexpr int kWords = BYTES >= 4 ? BYTES / 4 : 1;
  uint32_t w[kWords];
};

template <int BYTES>
__device__ __forceinline__ void load_raw(const uint8_t* src, Raw<BYTES>& r) {
  if constexpr (BYTES == 16) {
    const uint4 x = __ldcs(reinterpret_cast<const uint4*>(src));
    r.w[0] = x.x; r.w[1] = x.y; r.w[2] = x.z; r.w[3] = x.w;
  } else if constexpr (BYTES == 8) {
    const uint2 x = __ldcs(reinterpret_cast<const uint2*>(src));
    r.w[0] = x.x; r.w[1] = x.y;
  } else if constexpr (BYTES == 4) {
    r.w[0] = __ldcs(reinterpret_cast<const unsigned int*>(src));
  } else if constexpr (BYTES == 2) {
    r.w[0] = __ldcs(reinterpret_cast<const unsigned short*>(src));
  } else {
    static_assert(BYTES == 1, "unit size");
    r.w[0] = __ldcs(reinterpret_cast<const unsigned char*>(src));
  }
}

template <int BYTES>
__device__ __forceinline__ void store_raw(uint8_t* dst, const Raw<BYTES>& r) {
  if constexpr (BYTES >= 16) {
#pragma unroll
    for (int i = 0; i < BYTES / 16; ++i)
      *reinterpret_cast<uint4*>(dst + 16 * i) = make_uint4(r.w[4 * i], r.w[4 * i + 1], r.w[4 * i + 2], r.w[4 * i + 3]);
  } else if constexpr (BYTES == 8) {
    *reinterpret_cast<uint2*>(dst) = make_uint2(r.w[0], r.w[1]);
  } else if constexpr (BYTES == 4) {
    *reinterpret_cast<uint32_t*>(dst) = r.w[0];
  } else if constexpr (BYTES == 2) {
    *reinterpret_cast<uint16_t*>(dst) = static_cast<uint16_t>(r.w[0]);
  } else {
    static_assert(BYTES == 1, "unit size");
    *dst = static_cast<uint8_t>(r.w[0]);
  }
}

template <int CONV>
struct ConvTraits;
template <> struct ConvTraits<CONV_COPY> { static constexpr int es = 1, ed = 1; };
template <> struct ConvTraits<CONV_E4M3_BF16> { static constexpr int es = 1, ed = 2; };
template <> struct ConvTraits<CONV_E4M3_F16> { static constexpr int es = 1, ed = 2; };
template <> struct ConvTraits<CONV_E4M3_F32> { static constexpr int es = 1, ed = 4; };
template <> struct ConvTraits<CONV_BF16_F32> { static constexpr int es = 2, ed = 4; };
template <> struct ConvTraits<CONV_F16_F32> { static constexpr int es = 2, ed = 4; };

// two e4m3 codes (low 16 bits of `pair`) -> two exact fp32 values
__device__ __forceinline__ float2 e4m3x2_to_f32x2(uint32_t pair) {
  const __half2_raw h = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(pair & 0xFFFFu), __NV_E4M3);
  __half2 hh;
  hh = h;
  return __half22float2(hh);
}

__device__ __forceinline__ uint32_t pack_out2(float a, float b, int conv) {
  if (conv == CONV_E4M3_BF16) {
    const __nv_bfloat162 o = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<const uint32_t*>(&o);
  } else {
    const __half2 o = __floats2half2_rn(a, b);
    return *reinterpret_cast<const uint32_t*>(&o);
  }
}

// Converts N elements held in `in` into `out`.
template <int CONV, int N>
__device__ __forceinline__ void convert_unit(const Raw<N * ConvTraits<CONV>::es>& in,
                                             Raw<N * ConvTraits<CONV>::ed>& out, float scale) {
  if constexpr (CONV == CONV_COPY) {
#pragma unroll
    for (int i = 0; i < Raw<N>::kWords; ++i) out.w[i] = in.w[i];
  } else if constexpr (CONV == CONV_E4M3_BF16 || CONV == CONV_E4M3_F16 || CONV == CONV_E4M3_F32) {
    if constexpr (N == 1) {
      const float2 f = e4m3x2_to_f32x2(in.w[0]);
      const float y = __fmul_rn(f.x, scale);
      if constexpr (CONV == CONV_E4M3_F32) {
        out.w[0] = __float_as_uint(y);
      } else if constexpr (CONV == CONV_E4M3_BF16) {
        out.w[0] = __bfloat16_as_ushort(__float2bfloat16_rn(y));
      } else {
        out.w[0] = __half_as_ushort(__float2half_rn(y));
      }
    } else {
#pragma unroll
      for (int i = 0; i < N / 4; ++i) {
        const uint32_t w = in.w[i];
        const float2 lo = e4m3x2_to_f32x2(w);
        const float2 hi = e4m3x2_to_f32x2(w >> 16);
        const float a = __fmul_rn(lo.x, scale), b = __fmul_rn(lo.y, scale);
        const float c = __fmul_rn(hi.x, scale), d = __fmul_rn(hi.y, scale);
        if constexpr (CONV == CONV_E4M3_F32) {
          out.w[4 * i + 0] = __float_as_uint(a);
          out.w[4 * i + 1] = __float_as_uint(b);
          out.w[4 * i + 2] = __float_as_uint(c);
          out.w[4 * i + 3] = __float_as_uint(d);
        } else {
          out.w[2 * i + 0] = pack_out2(a, b, CONV);
          out.w[2 * i + 1] = pack_out2(c, d, CONV);
        }
      }
    }
  } else {
    // bf16 / fp16 -> fp32, exact
    if constexpr (N == 1) {
      const uint32_t h = in.w[0] & 0xFFFFu;
      if constexpr (CONV == CONV_BF16_F32) {
        out.w[0] = h << 16;
      } else {
        out.w[0] = __float_as_uint(__half2float(__ushort_as_half(static_cast<unsigned short>(h))));
      }
    } else {
#pragma unroll
      for (int i = 0; i < N / 2; ++i) {
        const uint32_t w = in.w[i];
        if constexpr (CONV == CONV_BF16_F32) {
          out.w[2 * i + 0] = w << 16;
          out.w[2 * i + 1] = w & 0xFFFF0000u;
        } else {
          out.w[2 * i + 0] = __float_as_uint(__half2float(__ushort_as_half(static_cast<unsigned short>(w & 0xFFFFu))));
          out.w[2 * i + 1] = __float_as_uint(__half2float(__ushort_as_half(static_cast<unsigned short>(w >> 16))));
        }
      }
    }
  }
}

// Bytes [d, d + 16) of the 32 bytes (a, b), d in 0..15 (little-endian words).
__device__ __forceinline__ uint4 bytes_from(const uint4& a, const uint4& b, uint32_t d) {
  const uint32_t sh = (d & 3u) * 8u;
  uint32_t c0, c1, c2, c3, c4;
  switch (d >> 2) {
    case 0: c0 = a.x; c1 = a.y; c2 = a.z; c3 = a.w; c4 = b.x; break;
    case 1: c0 = a.y; c1 = a.z; c2 = a.w; c3 = b.x; c4 = b.y; break;
    case 2: c0 = a.z; c1 = a.w; c2 = b.x; c3 = b.y; c4 = b.z; break;
    default: c0 = a.w; c1 = b.x; c2 = b.y; c3 = b.z; c4 = b.w; break;
  }
  return make_uint4(__funnelshift_r(c0, c1, sh), __funnelshift_r(c1, c2, sh), __funnelshift_r(c2, c3, sh),
                    __funnelshift_r(c3, c4, sh));
}

// Realigning byte copy of a segment table (the SIMT kernel with N = 0): unit
// (row, j) is the j-th 16-byte-aligned word of the destination row, of
// `words` per row (enough for any alignment of the row start). The word's
// bytes of the row come from at most two aligned 16-byte source words; only
// those holding bytes of the row are read. Whole words leave with one 16-byte
// store; the partial first and last words of a row are written byte by byte,
// so no byte outside the row is written.
__device__ __forceinline__ void realign_units(const Params& p, const Segment* segs, const int64_t* unit_prefix,
                                              int64_t total, uint32_t words) {
  const int32_t rb = p.row_src_bytes;
  int cur = 0;
  for (int64_t g0 = threadIdx.x; g0 < total; g0 += static_cast<int64_t>(kUnroll) * kPlanThreads) {
    uint4 lo[kUnroll], hi[kUnroll];
    uint8_t* wd[kUnroll];
    uint32_t b0[kUnroll], b1[kUnroll], dl[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int64_t g = g0 + static_cast<int64_t>(u) * kPlanThreads;
      wd[u] = nullptr;
      b0[u] = b1[u] = dl[u] = 0;
      lo[u] = hi[u] = make_uint4(0u, 0u, 0u, 0u);
      if (g < total) {
        while (unit_prefix[cur + 1] <= g) ++cur;
        const Segment& sg = segs[cur];
        const uint32_t local = static_cast<uint32_t>(g - unit_prefix[cur]);
        const uint32_t row = fast_div(local, p.upr_magic, p.upr_shift);
        const uint32_t j = local - row * words;
        const uint8_t* src = p.cache + sg.src + static_cast<int64_t>(row) * p.tok_stride_b;
        uint8_t* dst = p.dst + sg.dst + static_cast<int64_t>(row) * p.dst_stride_b;
        const int32_t mis = static_cast<int32_t>(reinterpret_cast<uintptr_t>(dst) & 15u);
        // the word holds row bytes [w0, w0 + 16) (w0 < 0 for the first word)
        const int32_t w0 = 16 * static_cast<int32_t>(j) - mis;
        const int32_t first = w0 > 0 ? w0 : 0;
        const int32_t end = w0 + 16 < rb ? w0 + 16 : rb;
        if (first < end) {
          const uintptr_t s0 = reinterpret_cast<uintptr_t>(src);
          const uintptr_t a = s0 + static_cast<uintptr_t>(static_cast<intptr_t>(w0));  // source of row byte w0
          const uintptr_t base = a & ~static_cast<uintptr_t>(15);
          if (s0 + static_cast<uintptr_t>(first) < base + 16u)
            lo[u] = __ldcs(reinterpret_cast<const uint4*>(base));
          if (s0 + static_cast<uintptr_t>(end - 1) >= base + 16u)
            hi[u] = __ldcs(reinterpret_cast<const uint4*>(base + 16u));
          wd[u] = dst - mis + 16 * static_cast<int64_t>(j);
          b0[u] = static_cast<uint32_t>(first - w0);
          b1[u] = static_cast<uint32_t>(end - w0);
          dl[u] = static_cast<uint32_t>(a - base);
        }
      }
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      if (wd[u] == nullptr) continue;
      const uint4 w = bytes_from(lo[u], hi[u], dl[u]);
      if (b0[u] == 0 && b1[u] == 16) {
        *reinterpret_cast<uint4*>(wd[u]) = w;
      } else {
        for (uint32_t k = b0[u]; k < b1[u]; ++k) {
          const uint32_t x = k < 4 ? w.x : (k < 8 ? w.y : (k < 12 ? w.z : w.w));
          wd[u][k] = static_cast<uint8_t>(x >> (8u * (k & 3u)));
        }
      }
    }
  }
}

// Realigning converting gather (the SIMT kernel with N = 0 and a conversion):
// unit (row, j) is the j-th 16-byte-aligned word of the destination row,
// 16 / ed elements starting at element e0 (negative for a row's first word
// when the row starts inside a word). Their source bytes (at most 8) come from
// at most two aligned 16-byte source words, read only where they hold bytes of
// the row's elements; the elements are converted as one TMA-converter unit;
// whole words leave with one 16-byte store, the partial first and last words
// of a row element by element.
template <int CONV>
__device__ __forceinline__ void realign_convert_units(const Params& p, const Segment* segs,
                                                      const int64_t* unit_prefix, int64_t total, uint32_t words,
                                                      float scale) {
  constexpr int es = ConvTraits<CONV>::es;
  constexpr int ed = ConvTraits<CONV>::ed;
  constexpr int n = 16 / ed;   // elements per destination word
  constexpr int kIn = n * es;  // their source bytes
  static_assert(kIn == 4 || kIn == 8, "source bytes per word");
  const int32_t E = p.row_dst_bytes / ed;
  int cur = 0;
  for (int64_t g0 = threadIdx.x; g0 < total; g0 += static_cast<int64_t>(kUnroll) * kPlanThreads) {
    uint4 lo[kUnroll], hi[kUnroll];
    uint8_t* wd[kUnroll];
    int32_t f0[kUnroll], f1[kUnroll];
    uint32_t dl[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int64_t g = g0 + static_cast<int64_t>(u) * kPlanThreads;
      wd[u] = nullptr;
      f0[u] = f1[u] = 0;
      dl[u] = 0;
      lo[u] = hi[u] = make_uint4(0u, 0u, 0u, 0u);
      if (g < total) {
        while (unit_prefix[cur + 1] <= g) ++cur;
        const Segment& sg = segs[cur];
        const uint32_t local = static_cast<uint32_t>(g - unit_prefix[cur]);
        const uint32_t row = fast_div(local, p.upr_magic, p.upr_shift);
        const uint32_t j = local - row * words;
        const uint8_t* src = p.cache + sg.src + static_cast<int64_t>(row) * p.tok_stride_b;
        uint8_t* dst = p.dst + sg.dst + static_cast<int64_t>(row) * p.dst_stride_b;
        const int32_t mis = static_cast<int32_t>(reinterpret_cast<uintptr_t>(dst) & 15u);  // a multiple of ed
        const int32_t e0 = (16 * static_cast<int32_t>(j) - mis) / ed;
        const int32_t first = e0 > 0 ? e0 : 0;
        const int32_t end = e0 + n < E ? e0 + n : E;
        if (first < end) {
          const uintptr_t s0 = reinterpret_cast<uintptr_t>(src);
          const uintptr_t a = s0 + static_cast<uintptr_t>(static_cast<intptr_t>(e0) * es);  // element e0's source
          const uintptr_t base = a & ~static_cast<uintptr_t>(15);
          if (s0 + static_cast<uintptr_t>(first * es) < base + 16u)
            lo[u] = __ldcs(reinterpret_cast<const uint4*>(base));
          if (s0 + static_cast<uintptr_t>(end * es - 1) >= base + 16u)
            hi[u] = __ldcs(reinterpret_cast<const uint4*>(base + 16u));
          wd[u] = dst - mis + 16 * static_cast<int64_t>(j);
          f0[u] = first - e0;
          f1[u] = end - e0;
          dl[u] = static_cast<uint32_t>(a - base);
        }
      }
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      if (wd[u] == nullptr) continue;
      const uint4 w = bytes_from(lo[u], hi[u], dl[u]);
      Raw<kIn> in;
      in.w[0] = w.x;
      if constexpr (kIn == 8) in.w[1] = w.y;
      Raw<16> out;
      convert_unit<CONV, n>(in, out, scale);
      if (f0[u] == 0 && f1[u] == n) {
        store_raw<16>(wd[u], out);
      } else {
        for (int32_t k = f0[u] * ed; k < f1[u] * ed; ++k)
          wd[u][k] = static_cast<uint8_t>(out.w[k >> 2] >> (8 * (k & 3)));
      }
    }
  }
}

template <int CONV, int N>
__global__ void __launch_bounds__(kPlanThreads) gather_simt_kernel(const __grid_constant__ Params p) {
  constexpr int kInBytes = N * ConvTraits<CONV>::es;
  constexpr int kOutBytes = N * ConvTraits<CONV>::ed;
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ Segment segs[kPlanThreads];
  __shared__ int64_t unit_prefix[kPlanThreads + 1];
  __shared__ int64_t warp_units[kPlanThreads / 32];

  const PlanView v = plan_view(smem, p);
  prefetch_metadata(p);
  pdl_entry();
  const int32_t num_tasks = build_plan<false>(p, v, blockIdx.x == 0);
  if (num_tasks <= 0) return;
  const CtaRange range = cta_range(v, p.R, p.B, num_tasks);
  if (range.row0 >= range.row1) return;

  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  float scale = 1.0f;
  if (CONV == CONV_E4M3_BF16 || CONV == CONV_E4M3_F16 || CONV == CONV_E4M3_F32) {
    if (p.scale != nullptr) scale = __ldg(p.scale);
  }
  const uint32_t upr = static_cast<uint32_t>(p.units_per_row);

  for (int32_t tb = range.t0;; tb += kPlanThreads) {
    Segment seg;
    const bool active = resolve_segment(p, v, tb + tid, num_tasks, range.row0, range.row1, seg);
    segs[tid] = seg;
    // exclusive scan of units per segment
    const int64_t my_units = static_cast<int64_t>(seg.nrows) * upr;
    int64_t x = my_units;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int64_t y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) warp_units[warp] = x;
    const int nseg = __syncthreads_count(active);
    if (warp == 0) {
      int64_t w = lane < kPlanThreads / 32 ? warp_units[lane] : 0;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int64_t y = __shfl_up_sync(0xffffffffu, w, o);
        if (lane >= o) w += y;
      }
      if (lane < kPlanThreads / 32) warp_units[lane] = w;
    }
    __syncthreads();
    unit_prefix[tid] = (warp > 0 ? warp_units[warp - 1] : 0) + x - my_units;
    if (tid == 0) unit_prefix[kPlanThreads] = warp_units[kPlanThreads / 32 - 1];
    __syncthreads();

    const int64_t total = unit_prefix[kPlanThreads];
    int cur = 0;
    if constexpr (N == 0 && CONV == CONV_COPY) {
      realign_units(p, segs, unit_prefix, total, upr);
    } else if constexpr (N == 0) {
      realign_convert_units<CONV>(p, segs, unit_prefix, total, upr, scale);
    } else {
    for (int64_t g0 = tid; g0 < total; g0 += static_cast<int64_t>(kUnroll) * kPlanThreads) {
      Raw<kInBytes> in[kUnroll];
      uint8_t* dptr[kUnroll];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int64_t g = g0 + static_cast<int64_t>(u) * kPlanThreads;
        dptr[u] = nullptr;
        if (g < total) {
          while (unit_prefix[cur + 1] <= g) ++cur;
          const Segment& s = segs[cur];
          const int64_t local = g - unit_prefix[cur];
          int64_t so, dof;
          if (p.dense) {
            so = s.src + local * kInBytes;
            dof = s.dst + local * kOutBytes;
          } else {
            const uint32_t row = fast_div(static_cast<uint32_t>(local), p.upr_magic, p.upr_shift);
            const uint32_t col = static_cast<uint32_t>(local) - row * upr;
            so = s.src + static_cast<int64_t>(row) * p.tok_stride_b + static_cast<int64_t>(col) * kInBytes;
            dof = s.dst + static_cast<int64_t>(row) * p.dst_stride_b + static_cast<int64_t>(col) * kOutBytes;
          }
          load_raw<kInBytes>(p.cache + so, in[u]);
          dptr[u] = p.dst + dof;
        }
      }
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        if (dptr[u] != nullptr) {
          Raw<kOutBytes> out;
          convert_unit<CONV, N>(in[u], out, scale);
          store_raw<kOutBytes>(dptr[u], out);
        }
      }
    }
    }
    const bool last = nseg < kPlanThreads;
    __syncthreads();
    if (last) break;
  }
}

// ---------------------------------------------------------------------------
// TMA-in converting path: bulk loads of source rows into a shared-memory ring,
// converter warps turn each landed stage into destination elements and store
// them with one coalesced 16-byte store per thread.
// ---------------------------------------------------------------------------

constexpr int kCvtWarps = 4;                        // converter warps
constexpr int kCvtThreads = 32 * (kCvtWarps + 2);   // + producer warp + scheduler warp

template <int BYTES>
__device__ __forceinline__ void load_smem(const uint8_t* src, Raw<BYTES>& r) {
  if constexpr (BYTES == 8) {
    const uint2 x = *reinterpret_cast<const uint2*>(src);
    r.w[0] = x.x; r.w[1] = x.y;
  } else {
    static_assert(BYTES == 4, "unit size");
    r.w[0] = *reinterpret_cast<const uint32_t*>(src);
  }
}

template <int CONV, int N>
__global__ void __launch_bounds__(kCvtThreads) gather_tma_convert_kernel(const __grid_constant__ Params p) {
  constexpr int kInBytes = N * ConvTraits<CONV>::es;
  constexpr int kOutBytes = N * ConvTraits<CONV>::ed;
  static_assert(kOutBytes == 16, "one 16-byte store per unit");
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ __align__(8) uint64_t full_bar[kMaxStages];
  __shared__ __align__(8) uint64_t empty_bar[kMaxStages];
  __shared__ Chunk stage_chunk[kMaxStages];
  __shared__ __align__(8) SegQueue q;

  uint8_t* stage_base = smem;
  const PlanView v = plan_view(smem + static_cast<size_t>(p.stages) * p.stage_bytes, p);
  // the speculative plan's area follows the plan (allocated only with p.spec)
  const PlanView sv = plan_view(smem + static_cast<size_t>(p.stages) * p.stage_bytes + plan_bytes(p), p);
  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  // nothing before the PDL wait reads an input: barrier set-up, L2 prefetch
  if (tid == 0) {
    for (int s = 0; s < p.stages; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], kCvtWarps);
    }
    segq_init(q);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  prefetch_metadata(p);
  pdl_trigger();
  // With early metadata or speculation the scheduler warp plans and resolves
  // its first batch while the previous grid may still run; every read of the
  // cache, scale or workspace and every write of dst comes after the wait.
  const bool early = p.early != 0 || p.spec != 0;
  if (!early) pdl_wait();
  __syncthreads();
  // small batches: the scheduler warp plans alone; large ones: the whole CTA;
  // the per-token gather needs no plan
  const bool warp_plan = p.R <= kWarpPlanMaxReqs || p.token_mode;
  int32_t num_tasks = 0;
  if (!warp_plan) {
    num_tasks = build_plan<false>(p, v, blockIdx.x == 0);
    if (num_tasks <= 0) return;
  }

  if (warp == kCvtWarps + 1) {
    if (p.token_mode) num_tasks = 1;
    else if (warp_plan && !p.spec) num_tasks = build_plan<true>(p, v, blockIdx.x == 0);
    if (!run_scheduler(p, v, sv, num_tasks, q)) set_flag(p, PMG_FLAG_TIMEOUT);
  } else if (warp == kCvtWarps) {
    // producer: one lane issues the bulk loads, up to p.stages chunks ahead
    if (lane == 0) {
      if (early) pdl_wait();
      const uint64_t pol = evict_first_policy();
      const uint32_t S = static_cast<uint32_t>(p.stages);
      SegReader rd{0, -1, 0, ChunkIter{0, 0}, false, 0};
      for (uint32_t g = 0;; ++g) {
        Chunk c;
        const int r = rd.next(q, p, c, true);
        const int s = static_cast<int>(g % S);
        const uint32_t use = g / S;
        if (use > 0 && !mbar_wait_bounded(&empty_bar[s], (use - 1) & 1u)) {
          set_flag(p, PMG_FLAG_TIMEOUT);
          break;
        }
        if (r <= 0) {
          // no more work: an empty chunk tells the converters to stop
          if (r == -2) set_flag(p, PMG_FLAG_TIMEOUT);
          stage_chunk[s].nrows = 0;
          mbar_arrive(&full_bar[s]);
          break;
        }
        stage_chunk[s] = c;
        issue_loads(p, c, stage_base + static_cast<size_t>(s) * p.stage_bytes, &full_bar[s], pol);
      }
    }
  } else {
    // converters: every landed stage, unit u = (row, col) of the chunk
    if (early) {
      if (warp == 0) prefetch_helper(p, q);
      pdl_wait();
    }
    float scale = 1.0f;
    if (CONV == CONV_E4M3_BF16 || CONV == CONV_E4M3_F16 || CONV == CONV_E4M3_F32) {
      if (p.scale != nullptr) scale = __ldg(p.scale);
    }
    const uint32_t upr = static_cast<uint32_t>(p.units_per_row);
    const uint32_t S = static_cast<uint32_t>(p.stages);
    for (uint32_t g = 0;; ++g) {
      const int s = static_cast<int>(g % S);
      if (!mbar_wait_bounded(&full_bar[s], (g / S) & 1u)) {
        set_flag(p, PMG_FLAG_TIMEOUT);
        break;
      }
      const Chunk c = stage_chunk[s];
      if (c.nrows == 0) break;
      if (c.tentative) {
        const int vr = spec_verdict(q);
        if (vr != 1) {
          // withdrawn (or no verdict in time): drop the chunk unconverted
          if (vr < 0 && tid == 0) set_flag(p, PMG_FLAG_TIMEOUT);
          __syncwarp();
          if (lane == 0) mbar_arrive(&empty_bar[s]);
          continue;
        }
      }
      const uint8_t* in = stage_base + static_cast<size_t>(s) * p.stage_bytes;
      const uint32_t units = static_cast<uint32_t>(c.nrows) * upr;
      uint8_t* out = p.dst + c.dst;
      for (uint32_t u = tid; u < units; u += kCvtWarps * 32) {
        Raw<kInBytes> x;
        load_smem<kInBytes>(in + static_cast<size_t>(u) * kInBytes, x);
        Raw<kOutBytes> y;
        convert_unit<CONV, N>(x, y, scale);
        int64_t off;
        if (p.dense) {
          off = static_cast<int64_t>(u) * kOutBytes;
        } else {
          const uint32_t row = fast_div(u, p.upr_magic, p.upr_shift);
          off = static_cast<int64_t>(row) * p.dst_stride_b + static_cast<int64_t>(u - row * upr) * kOutBytes;
        }
        store_raw<kOutBytes>(out + off, y);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty_bar[s]);
    }
  }
  __syncthreads();
}

// ---------------------------------------------------------------------------
// Per-token indexed gather ("indexer kernels take shape arguments at run time",
// vllm PR #56153, section "关键源码片段": _cp_gather_indexer_quant_cache_kernel).
// Output row t reads request b = token_to_seq[t] at context position
// t - cu_seq_lens[b]. One warp takes 32 consecutive tokens: each lane resolves
// its token (request id, row range, block-table column, block id, all masked),
// then the warp moves the 32 rows as a flat run of vector units, each lane
// fetching the row base of its unit from the owning lane by shuffle. Small
// calls use tiles of 16 or 8 tokens so that every resident warp has work.
// ---------------------------------------------------------------------------

struct TokParams {
  const uint8_t* cache;
  int64_t blk_stride_b;
  int64_t tok_stride_b;
  int64_t num_blocks;
  const int32_t* bt;
  int64_t bt_stride;
  const int32_t* t2s;
  const int32_t* cu;
  int64_t T;  // num_tokens (<= INT32_MAX)
  int32_t R;
  int32_t B;
  uint8_t* dst;
  int64_t dst_stride_b;
  const float* scale;
  int32_t* err;
  int32_t units_per_row;
  uint32_t upr_magic;
  int32_t upr_shift;
  int32_t tile_rows;  // tokens per warp tile: 8, 16 or 32
};

constexpr int kTokThreads = 256;

template <int CONV, int N>
__global__ void __launch_bounds__(kTokThreads) gather_tokens_kernel(const __grid_constant__ TokParams p) {
  constexpr int kInBytes = N * ConvTraits<CONV>::es;
  constexpr int kOutBytes = N * ConvTraits<CONV>::ed;
  pdl_entry();
  const int lane = threadIdx.x & 31;
  const int64_t warps = static_cast<int64_t>(gridDim.x) * (kTokThreads / 32);
  float scale = 1.0f;
  if (CONV == CONV_E4M3_BF16 || CONV == CONV_E4M3_F16 || CONV == CONV_E4M3_F32) {
    if (p.scale != nullptr) scale = __ldg(p.scale);
  }
  const uint64_t keep = evict_last_policy();
  const uint32_t upr = static_cast<uint32_t>(p.units_per_row);
  int bits = 0;
  const int64_t tr = p.tile_rows;
  for (int64_t tile = static_cast<int64_t>(blockIdx.x) * (kTokThreads / 32) + (threadIdx.x >> 5); tile * tr < p.T;
       tile += warps) {
    const int64_t t = tile * tr + lane;
    int64_t src = -1;
    if (lane < tr && t < p.T) {
      const int32_t b = __ldg(p.t2s + t);
      if (b < 0 || b >= p.R) {
        bits |= PMG_FLAG_TOKEN;
      } else {
        const int64_t c0 = ld_meta(p.cu + b, keep);
        const int64_t c1 = ld_meta(p.cu + b + 1, keep);
        if (t < c0 || t >= c1) {
          bits |= PMG_FLAG_TOKEN;
        } else {
          const uint32_t pos = static_cast<uint32_t>(t - c0);
          const uint32_t lb = pos / static_cast<uint32_t>(p.B);
          const uint32_t off = pos - lb * static_cast<uint32_t>(p.B);
          if (static_cast<int64_t>(lb) >= p.bt_stride) {
            bits |= PMG_FLAG_LOGICAL_BLOCK;
          } else {
            const int64_t phys = ld_meta(p.bt + static_cast<int64_t>(b) * p.bt_stride + lb, keep);
            if (phys < 0 || phys >= p.num_blocks) {
              bits |= PMG_FLAG_PHYS_BLOCK;
            } else {
              src = phys * p.blk_stride_b + static_cast<int64_t>(off) * p.tok_stride_b;
            }
          }
        }
      }
    }
    const int64_t dst_row = t * p.dst_stride_b;
    const int64_t left = p.T - tile * tr;
    const uint32_t nrows = static_cast<uint32_t>(left < tr ? left : tr);
    const uint32_t total = nrows * upr;
    for (uint32_t base = 0; base < total; base += 32u * kUnroll) {
      Raw<kInBytes> in[kUnroll];
      int64_t dofs[kUnroll];
      bool ok[kUnroll];
#pragma unroll
      for (int k = 0; k < kUnroll; ++k) {
        const uint32_t u = base + static_cast<uint32_t>(k) * 32u + lane;
        const uint32_t row = u < total ? fast_div(u, p.upr_magic, p.upr_shift) : 0u;
        const int64_t s = __shfl_sync(0xffffffffu, src, static_cast<int>(row));
        const int64_t d = __shfl_sync(0xffffffffu, dst_row, static_cast<int>(row));
        ok[k] = u < total && s >= 0;
        dofs[k] = 0;
        if (ok[k]) {
          const uint32_t col = u - row * upr;
          load_raw<kInBytes>(p.cache + s + static_cast<int64_t>(col) * kInBytes, in[k]);
          dofs[k] = d + static_cast<int64_t>(col) * kOutBytes;
        }
      }
#pragma unroll
      for (int k = 0; k < kUnroll; ++k) {
        if (ok[k]) {
          Raw<kOutBytes> out;
          convert_unit<CONV, N>(in[k], out, scale);
          store_raw<kOutBytes>(p.dst + dofs[k], out);
        }
      }
    }
  }
  bits = __reduce_or_sync(0xffffffffu, bits);
  if (lane == 0 && bits != 0 && p.err != nullptr) atomicOr(p.err, bits);
}

// ---------------------------------------------------------------------------
// Large batches (more requests than one launch plans in shared memory) run as
// consecutive launches over groups of requests. A group's plan needs the
// highest cu_seq_lens boundary of the groups before it (a request is skipped
// when its rows start below it): each group's first CTA leaves that value in
// one of two workspace slots for the next group, which reads it only after the
// group before has completed; a final one-thread launch clears the slots.
// ---------------------------------------------------------------------------

constexpr int kCarrySlot = 2;  // workspace ints 2 and 3
static_assert(kCarrySlot + 2 <= PMG_WORKSPACE_INTS, "the carried boundaries must fit the workspace");

__global__ void clear_carry_kernel(int32_t* ws) {
  pdl_entry();
  if (threadIdx.x < 2) ws[kCarrySlot + threadIdx.x] = 0;
}

// ---------------------------------------------------------------------------
// Debug plan: the mapper alone
// ---------------------------------------------------------------------------

__global__ void __launch_bounds__(kPlanThreads) debug_plan_kernel(const __grid_constant__ Params p, int32_t* tasks_out,
                                                                  int64_t max_tasks, int64_t* num_tasks_out) {
  extern __shared__ __align__(128) uint8_t smem[];
  const PlanView v = plan_view(smem, p);
  const int32_t n = build_plan<false>(p, v, true);
  const int32_t num = n < 0 ? 0 : n;
  if (threadIdx.x == 0) *num_tasks_out = num;
  const int64_t lim = num < max_tasks ? num : max_tasks;
  for (int64_t t = threadIdx.x; t < lim; t += blockDim.x) {
    const PageTask k = map_task(v, p.R, p.B, static_cast<int32_t>(t));
    int32_t* o = tasks_out + t * 5;
    o[0] = k.req;
    o[1] = static_cast<int32_t>(k.logical_block);
    o[2] = k.begin;
    o[3] = k.end;
    o[4] = k.out;
  }
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------

int elem_bytes(int dt) {
  switch (dt) {
    case PMG_BF16: return 2;
    case PMG_FP16: return 2;
    case PMG_FP32: return 4;
    case PMG_FP8_E4M3: return 1;
    case PMG_U8: return 1;
    default: return 0;
  }
}

// -1 for an unsupported pair
int conv_of(int src, int dst) {
  if (elem_bytes(src) == 0 || elem_bytes(dst) == 0) return -1;
  if (src == dst) return CONV_COPY;
  if (src == PMG_FP8_E4M3) {
    if (dst == PMG_BF16) return CONV_E4M3_BF16;
    if (dst == PMG_FP16) return CONV_E4M3_F16;
    if (dst == PMG_FP32) return CONV_E4M3_F32;
  }
  if (dst == PMG_FP32) {
    if (src == PMG_BF16) return CONV_BF16_F32;
    if (src == PMG_FP16) return CONV_F16_F32;
  }
  return -1;
}

// An integer tuning variable from the environment, clamped to [lo, hi].
int env_int(const char* name, int dflt, int lo, int hi) {
  const char* e = std::getenv(name);
  int v = e ? std::atoi(e) : dflt;
  return v < lo ? lo : (v > hi ? hi : v);
}

// Target bytes of one stage of the byte-copy TMA ring (three stages by
// default). A page gather over back-to-back source rows moves each chunk with
// one copy: 32 KB stages, two CTAs per SM. Padded source rows take one copy per
// row, all issued by the CTA's one producer thread, and the per-token mode
// resolves its rows through three dependent reads per batch: both do better
// with 22 KB stages, which fit three CTAs (three producers and schedulers) per
// SM. Measured: single-300K 1.008 -> 1.010, single-60K 0.926 -> 0.931,
// skew-64 raw (padded) 0.961 -> 0.983, per-token single-60K 0.86 -> 0.93 of
// the copy peak, against four 24 KB stages. PMG_BULK_STAGE_KB (8..48)
// overrides both for tuning sweeps; it changes only the chunking, never the
// result.
int bulk_stage_target_bytes(bool one_copy_per_chunk) {
  static const int env = [] {
    const char* e = std::getenv("PMG_BULK_STAGE_KB");
    if (e == nullptr) return 0;
    int kb = std::atoi(e);
    if (kb < 8) kb = 8;
    if (kb > kMaxStageBytes / 1024) kb = kMaxStageBytes / 1024;
    return kb * 1024;
  }();
  if (env > 0) return env;
  return (one_copy_per_chunk ? 32 : 22) * 1024;
}

// Ring of the converting kernel. Its registers allow four CTAs per SM; what
// decides is the source bytes in flight per SM and how the ring's stages fall
// against the work split. Measured on single fp8 -> bf16 requests and the
// named workloads (fractions of the copy peak):
// - launches of at most 128 rows per CTA (a static split: each CTA's head of
//   four stages covers its share) take two 18 KB stages of 32 rows: skew-8
//   0.875 -> 0.892, one 60,000-token request 0.968 -> 0.979, against three of
//   16 KB; longer launches lose with two stages (120,000 tokens 0.93);
// - longer launches over back-to-back rows take three 14 KB stages (120,000
//   tokens 0.940 -> 0.973, 300,000 0.989 -> 0.999);
// - longer launches over padded rows keep three 16 KB stages (skew-64 dequant
//   0.940; 0.929-0.938 with 4 x 12, 3 x 14, 3 x 18 or 2 x 18 KB);
// - the per-token mode four of 12 KB (its scheduler's dependent reads favour
//   it: 0.93 against 0.92).
// rows_per_cta < 0 means not known yet (the host half of a call, before the
// grid is sized). PMG_CVT_STAGE_KB (4..48) and PMG_CVT_STAGES (2..8) override
// every case for tuning sweeps.
constexpr int64_t kCvtSmallRows = 128;
constexpr int kCvtCtasPerSm = 4;
struct CvtRing {
  int stages;
  int kb;
};
CvtRing cvt_ring(bool token_mode, bool dense_rows, int64_t rows_per_cta) {
  static const int env_kb = [] {
    const char* e = std::getenv("PMG_CVT_STAGE_KB");
    if (e == nullptr) return 0;
    int kb = std::atoi(e);
    if (kb < 4) kb = 4;
    if (kb > kMaxStageBytes / 1024) kb = kMaxStageBytes / 1024;
    return kb;
  }();
  static const int env_stages = env_int("PMG_CVT_STAGES", 0, 0, kMaxStages);
  CvtRing r;
  if (token_mode) r = {4, 12};
  else if (rows_per_cta >= 0 && rows_per_cta <= kCvtSmallRows) r = {2, 18};
  else if (dense_rows) r = {3, 14};
  else r = {3, 16};
  if (env_kb > 0) r.kb = env_kb;
  if (env_stages >= 2) r.stages = env_stages;
  return r;
}

// Dynamic scheduling knobs (PMG_SCHED_STATIC_PCT, PMG_SCHED_MIN_ROWS) for
// tuning sweeps; they change only the work split, never the result.
int sched_static_pct() {
  static const int v = env_int("PMG_SCHED_STATIC_PCT", 25, 0, 100);
  return v;
}
// Ring stages' worth of rows of the pre-wait batch prefetched into L2
// (PMG_PREFETCH_STAGES, 0..8). A full ring (4) measured best: single-300K
// 0.987 -> 1.002 of the copy peak, skew-64 dequant 0.902 -> 0.924; 8 loses
// on the padded raw rows.
int prefetch_stages() {
  static const int v = env_int("PMG_PREFETCH_STAGES", 4, 0, kMaxStages);
  return v;
}

// The realigning byte copy for rows that are not 16-byte aligned
// (PMG_REALIGN=0 keeps them on the narrow-unit SIMT kernels, for A/B runs).
bool use_realign() {
  static const int v = env_int("PMG_REALIGN", 1, 0, 1);
  return v != 0;
}

// Speculative start of the TMA paths (PMG_SPEC=0 turns it off).
bool use_spec() {
  static const int v = env_int("PMG_SPEC", 1, 0, 1);
  return v != 0;
}

// One request without seq_starts: the speculative plan assumes cu = [0, T]
// instead of reading it (PMG_SPEC_GUESS=0 reads it, for A/B runs).
bool use_spec_guess() {
  static const int v = env_int("PMG_SPEC_GUESS", 1, 0, 1);
  return v != 0;
}

int sched_min_rows() {
  static const int v = env_int("PMG_SCHED_MIN_ROWS", 32, 1, 1 << 30);
  return v;
}
// Static head of the dynamic split, in ring stages per CTA: a page gather's
// CTAs start with at least four stages of their own rows before they claim
// (single-60K 0.936 -> 0.974 of peak; the large workloads unchanged), the
// per-token mode with two (its claims cost less than its idle head: four
// stages lost 8% on skew-8). PMG_SCHED_HEAD_STAGES overrides both.
int sched_head_stages(bool token_mode) {
  static const int v = env_int("PMG_SCHED_HEAD_STAGES", 0, 0, 64);
  if (v >= 1) return v;
  return token_mode ? 2 : 4;
}

// Tilt of the static shares by blockIdx (make_items, tilted_prefix). A
// launch's CTAs start in blockIdx order as the previous grid's CTAs leave (the
// last eighth about 5 us after the first in steady state), and the late ones
// pay their start-up (plan, block-table and first data round trips) while the
// others already stream. The converting kernel takes a quartic tilt of 8%
// (shares 1.08 of even for most CTAs, falling to 0.68 for the last): skew-8
// 0.871 -> 0.892 of the copy peak with its two-stage ring (0.821 -> 0.870 with
// three 16 KB stages), one fp8 request of 45,657 tokens 0.910 -> 0.939; cubic
// 10% and quartic 6% measured within 0.3% of it, linear 20-30% lower. A call
// whose CTAs all start at once gains nothing from it: skew-8 after an L2 flush
// that leaves clean lines takes about 1.7 us longer on average (the page's
// write flush: no change). The byte-copy kernel keeps even shares (a tilt cost
// its static splits 1-3.5%). PMG_SCHED_TILT_PCT (0..100) and
// PMG_SCHED_TILT_POW (1..4) override both kernels for tuning sweeps.
int sched_tilt_pct(bool converter) {
  static const int v = env_int("PMG_SCHED_TILT_PCT", -1, -1, 100);
  if (v >= 0) return v;
  return converter ? 8 : 0;
}
int sched_tilt_pow() {
  static const int v = env_int("PMG_SCHED_TILT_POW", 4, 1, 4);
  return v;
}

// Ring depths (PMG_BULK_STAGES, PMG_CVT_STAGES: 2..8) for tuning sweeps.
int bulk_stages() {
  static const int v = env_int("PMG_BULK_STAGES", 3, 2, kMaxStages);
  return v;
}

// Elements per unit of the converting TMA path: one 16-byte store per unit.
int tma_convert_unit(int conv) {
  switch (conv) {
    case CONV_E4M3_BF16:
    case CONV_E4M3_F16: return 8;
    case CONV_E4M3_F32:
    case CONV_BF16_F32:
    case CONV_F16_F32: return 4;
    default: return 0;
  }
}

bool aligned(const void* ptr, int64_t a) { return (reinterpret_cast<uintptr_t>(ptr) % static_cast<uint64_t>(a)) == 0; }

int unit_candidates(int conv, int* out);

// Largest access unit (elements; bytes for a byte copy) that every source row
// start, row length and destination row start allow.
int pick_unit(int conv, int es, int ed, int32_t E, const void* cache, int64_t blk_b, int64_t tok_b, const void* dst,
              int64_t dst_b) {
  int cand[5];
  const int ncand = unit_candidates(conv, cand);
  for (int i = 0; i < ncand; ++i) {
    const int n = cand[i];
    const int64_t row_units_base = (conv == CONV_COPY) ? static_cast<int64_t>(E) * es : E;
    const int64_t in_b = (conv == CONV_COPY) ? n : static_cast<int64_t>(n) * es;
    const int64_t out_b = (conv == CONV_COPY) ? n : static_cast<int64_t>(n) * ed;
    const int64_t out_align = out_b > 16 ? 16 : out_b;
    if (row_units_base % n != 0) continue;
    if (!aligned(cache, in_b) || blk_b % in_b != 0 || tok_b % in_b != 0) continue;
    if (!aligned(dst, out_align) || dst_b % out_align != 0) continue;
    return n;
  }
  return 1;
}

struct Plan {
  int path;         // pmg_path
  int conv;
  int unit;         // elements per access for SIMT (bytes for CONV_COPY)
  Params prm;
};

// candidate units (elements per access; bytes for a byte copy)
int unit_candidates(int conv, int* out) {
  switch (conv) {
    case CONV_COPY: out[0] = 16; out[1] = 8; out[2] = 4; out[3] = 2; out[4] = 1; return 5;
    case CONV_E4M3_BF16:
    case CONV_E4M3_F16:
    case CONV_E4M3_F32: out[0] = 16; out[1] = 4; out[2] = 1; return 3;
    default: out[0] = 8; out[1] = 2; out[2] = 1; return 3;
  }
}

// Ring of the converting kernel: stages of whole source rows.
void set_cvt_ring(Params& q, bool token_mode, int64_t rows_per_cta) {
  const CvtRing r = cvt_ring(token_mode, q.src_dense != 0, rows_per_cta);
  const int32_t rows = std::max(1, r.kb * 1024 / q.row_src_bytes);
  q.rows_per_stage = rows;
  q.stage_bytes = rows * q.row_src_bytes;
  q.stages = r.stages;
  q.prefetch_rows = prefetch_stages() * rows;
}

// Ring of the byte-copy kernel: stages of whole rows.
void set_bulk_ring(Params& q, bool one_copy_per_chunk) {
  const int32_t rows = std::max(1, bulk_stage_target_bytes(one_copy_per_chunk) / q.row_src_bytes);
  q.rows_per_stage = rows;
  q.stage_bytes = rows * q.row_src_bytes;
  q.stages = bulk_stages();
  q.prefetch_rows = prefetch_stages() * rows;
}

// Validation and path choice: the host half of every entry point. No CUDA call.
int make_plan(const void* cache, int64_t cbs, int64_t cts, int64_t num_blocks, const int32_t* bt, int64_t bt_stride,
              const int32_t* cu, const int32_t* ss, int32_t R, int64_t T, int32_t B, int32_t E, int32_t sdt,
              int32_t ddt, const float* scale, const void* dst, int64_t dts, int32_t* err, int32_t* workspace,
              uint32_t options, Plan& out) {
  out.path = PMG_PATH_NONE;
  out.unit = 0;
  const int conv = conv_of(sdt, ddt);
  if (conv < 0) return PMG_ERR_DTYPE;
  if (R < 0 || T < 0 || B < 1 || E < 1 || num_blocks < 0 || bt_stride < 0 || cbs < 0 || cts < 0 || dts < E)
    return PMG_ERR_ARG;
  if (options & ~(PMG_OPT_FORCE_SIMT | PMG_OPT_FORCE_SCALAR | PMG_OPT_IMPLIED_END | PMG_OPT_EARLY_METADATA))
    return PMG_ERR_ARG;
  if (R > PMG_MAX_REQS) return PMG_ERR_UNSUPPORTED;
  // more requests than one launch plans need the workspace (it carries the
  // highest cu_seq_lens boundary from one group of requests to the next)
  if (R > PMG_MAX_REQS_PLAN && workspace == nullptr) return PMG_ERR_UNSUPPORTED;
  const int es = elem_bytes(sdt), ed = elem_bytes(ddt);
  if (static_cast<int64_t>(E) * ed > INT32_MAX || static_cast<int64_t>(E) * es > INT32_MAX) return PMG_ERR_UNSUPPORTED;
  if (R == 0 || T == 0) {
    out.conv = conv;
    return PMG_OK;  // nothing to write: no launch
  }
  if (cache == nullptr || bt == nullptr || cu == nullptr || dst == nullptr) return PMG_ERR_NULL;
  if (!aligned(cache, es) || !aligned(dst, ed) || !aligned(bt, 4) || !aligned(cu, 4) ||
      (ss != nullptr && !aligned(ss, 4)) || (scale != nullptr && !aligned(scale, 4)) ||
      (err != nullptr && !aligned(err, 4)) || (workspace != nullptr && !aligned(workspace, 16)))
    return PMG_ERR_ALIGN;
  // strides in bytes must not overflow int64
  if (cbs > INT64_MAX / es / 2 || cts > INT64_MAX / es / 2 || dts > INT64_MAX / ed / 2) return PMG_ERR_ARG;

  Params& q = out.prm;
  q = Params{};
  q.cache = static_cast<const uint8_t*>(cache);
  q.blk_stride_b = cbs * es;
  q.tok_stride_b = cts * es;
  q.num_blocks = num_blocks;
  q.bt = bt;
  q.bt_stride = bt_stride;
  q.cu = cu;
  q.ss = ss;
  q.R = R;
  q.T = static_cast<int32_t>(T < INT32_MAX ? T : INT32_MAX);
  q.B = B;
  q.implied_end = (options & PMG_OPT_IMPLIED_END) ? 1 : 0;
  q.row_src_bytes = E * es;
  q.row_dst_bytes = E * ed;
  q.dst = static_cast<uint8_t*>(const_cast<void*>(dst));
  q.dst_stride_b = dts * ed;
  q.scale = scale;
  q.err = err;
  q.sched = workspace;
  // large batches read a verdict from the workspace first: no early start there
  q.early = ((options & PMG_OPT_EARLY_METADATA) && R <= PMG_MAX_REQS_PLAN) ? 1 : 0;
  // without the promise, small batches still plan before the wait and check
  // the plan after it (the TMA paths; the SIMT kernels ignore the field)
  q.spec = (!q.early && R <= kWarpPlanMaxReqs && use_spec()) ? 1 : 0;
  q.spec_guess = use_spec_guess() ? 1 : 0;
  q.sched_static_pct = sched_static_pct();
  q.sched_min_rows = sched_min_rows();
  q.sched_head_stages = sched_head_stages(false);
  q.sched_tilt_pow = sched_tilt_pow();
  out.conv = conv;

  int unit = pick_unit(conv, es, ed, E, cache, q.blk_stride_b, q.tok_stride_b, dst, q.dst_stride_b);
  if (options & PMG_OPT_FORCE_SCALAR) unit = (conv == CONV_COPY) ? es : 1;
  out.unit = unit;

  const bool forced = (options & (PMG_OPT_FORCE_SIMT | PMG_OPT_FORCE_SCALAR)) != 0;
  const bool bulk_ok = conv == CONV_COPY && unit == 16 && q.row_src_bytes <= kMaxStageBytes && !forced;
  // converting TMA path: source rows fit 16-byte bulk copies, output units are
  // 16-byte stores
  const int cu_unit = tma_convert_unit(conv);
  const bool tma_cvt_ok = conv != CONV_COPY && !forced && cu_unit > 0 && E % cu_unit == 0 &&
                          q.row_src_bytes % 16 == 0 && q.row_src_bytes <= kMaxStageBytes && aligned(cache, 16) &&
                          q.blk_stride_b % 16 == 0 && q.tok_stride_b % 16 == 0 && aligned(dst, 16) &&
                          q.dst_stride_b % 16 == 0;
  q.src_dense = q.tok_stride_b == q.row_src_bytes;
  q.dst_dense = q.dst_stride_b == q.row_dst_bytes;
  if (bulk_ok) {
    out.path = PMG_PATH_BULK;
    set_bulk_ring(q, q.src_dense != 0);
    q.sched_tilt_pct = sched_tilt_pct(false);
    out.unit = 0;
  } else {
    int64_t upr;
    if (tma_cvt_ok) {
      out.path = PMG_PATH_BULK;
      out.unit = cu_unit;
      upr = E / cu_unit;
      set_cvt_ring(q, false, -1);  // sized again at launch, from the grid
      q.sched_tilt_pct = sched_tilt_pct(true);
      q.dense = q.dst_dense;
    } else if (!forced && q.row_dst_bytes >= 16 && use_realign() &&
               (conv == CONV_COPY ? unit < 16 : cu_unit > 0)) {
      // rows not 16-byte aligned (or converting rows whose length is not a
      // whole number of converter units): whole 16-byte words of each
      // destination row, assembled from aligned source words (the SIMT
      // kernel's N = 0 movers)
      out.path = PMG_PATH_REALIGN;
      out.unit = 0;
      upr = (static_cast<int64_t>(q.row_dst_bytes) + 15 + 15) / 16;
      q.dense = 0;
    } else {
      const int64_t unit_elems = (conv == CONV_COPY) ? unit / es : unit;
      out.path = (unit_elems > 1) ? PMG_PATH_VECTOR : PMG_PATH_SCALAR;
      upr = (conv == CONV_COPY) ? static_cast<int64_t>(E) * es / unit : E / unit;
      q.dense = q.src_dense && q.dst_dense;
    }
    q.units_per_row = static_cast<int32_t>(upr);
    if (!q.dense) {
      // the row split divides 32-bit unit indices inside one page or stage
      if (static_cast<uint64_t>(B) * static_cast<uint64_t>(upr) >= (1ull << 32)) return PMG_ERR_UNSUPPORTED;
      uint32_t l = 0;
      while ((1ull << l) < static_cast<uint64_t>(upr)) ++l;
      const uint64_t m = (((1ull << l) - static_cast<uint64_t>(upr)) << 32) / static_cast<uint64_t>(upr) + 1;
      q.upr_magic = static_cast<uint32_t>(m);
      q.upr_shift = static_cast<int32_t>(l);
    }
  }
  return PMG_OK;
}

// --- per-device launch facts -------------------------------------------------

constexpr int kMaxDevices = 64;
std::mutex g_mu;
int g_sm_count[kMaxDevices];
bool g_attr_set[kMaxDevices];
int g_optin_smem[kMaxDevices];
bool g_plan_attr_set[kMaxDevices];

using KernelFn = void (*)(Params);

KernelFn simt_kernel_for(int conv, int unit) {
#define PMG_CASE(C, N) \
  if (conv == C && unit == N) return gather_simt_kernel<C, N>;
  PMG_CASE(CONV_COPY, 16) PMG_CASE(CONV_COPY, 8) PMG_CASE(CONV_COPY, 4) PMG_CASE(CONV_COPY, 2)
  PMG_CASE(CONV_COPY, 1) PMG_CASE(CONV_COPY, 0)
  PMG_CASE(CONV_E4M3_BF16, 16) PMG_CASE(CONV_E4M3_BF16, 4) PMG_CASE(CONV_E4M3_BF16, 1) PMG_CASE(CONV_E4M3_BF16, 0)
  PMG_CASE(CONV_E4M3_F16, 16) PMG_CASE(CONV_E4M3_F16, 4) PMG_CASE(CONV_E4M3_F16, 1) PMG_CASE(CONV_E4M3_F16, 0)
  PMG_CASE(CONV_E4M3_F32, 16) PMG_CASE(CONV_E4M3_F32, 4) PMG_CASE(CONV_E4M3_F32, 1) PMG_CASE(CONV_E4M3_F32, 0)
  PMG_CASE(CONV_BF16_F32, 8) PMG_CASE(CONV_BF16_F32, 2) PMG_CASE(CONV_BF16_F32, 1) PMG_CASE(CONV_BF16_F32, 0)
  PMG_CASE(CONV_F16_F32, 8) PMG_CASE(CONV_F16_F32, 2) PMG_CASE(CONV_F16_F32, 1) PMG_CASE(CONV_F16_F32, 0)
#undef PMG_CASE
  return nullptr;
}

using TokKernelFn = void (*)(TokParams);

TokKernelFn tokens_kernel_for(int conv, int unit) {
#define PMG_TCASE(C, N) \
  if (conv == C && unit == N) return gather_tokens_kernel<C, N>;
  PMG_TCASE(CONV_COPY, 16) PMG_TCASE(CONV_COPY, 8) PMG_TCASE(CONV_COPY, 4) PMG_TCASE(CONV_COPY, 2)
  PMG_TCASE(CONV_COPY, 1)
  PMG_TCASE(CONV_E4M3_BF16, 16) PMG_TCASE(CONV_E4M3_BF16, 4) PMG_TCASE(CONV_E4M3_BF16, 1)
  PMG_TCASE(CONV_E4M3_F16, 16) PMG_TCASE(CONV_E4M3_F16, 4) PMG_TCASE(CONV_E4M3_F16, 1)
  PMG_TCASE(CONV_E4M3_F32, 16) PMG_TCASE(CONV_E4M3_F32, 4) PMG_TCASE(CONV_E4M3_F32, 1)
  PMG_TCASE(CONV_BF16_F32, 8) PMG_TCASE(CONV_BF16_F32, 2) PMG_TCASE(CONV_BF16_F32, 1)
  PMG_TCASE(CONV_F16_F32, 8) PMG_TCASE(CONV_F16_F32, 2) PMG_TCASE(CONV_F16_F32, 1)
#undef PMG_TCASE
  return nullptr;
}

const KernelFn kAllSimt[] = {
    gather_simt_kernel<CONV_COPY, 16>,      gather_simt_kernel<CONV_COPY, 8>,      gather_simt_kernel<CONV_COPY, 4>,
    gather_simt_kernel<CONV_COPY, 2>,       gather_simt_kernel<CONV_COPY, 1>,      gather_simt_kernel<CONV_E4M3_BF16, 16>,
    gather_simt_kernel<CONV_E4M3_BF16, 4>,  gather_simt_kernel<CONV_E4M3_BF16, 1>, gather_simt_kernel<CONV_E4M3_F16, 16>,
    gather_simt_kernel<CONV_E4M3_F16, 4>,   gather_simt_kernel<CONV_E4M3_F16, 1>,  gather_simt_kernel<CONV_E4M3_F32, 16>,
    gather_simt_kernel<CONV_E4M3_F32, 4>,   gather_simt_kernel<CONV_E4M3_F32, 1>,  gather_simt_kernel<CONV_BF16_F32, 8>,
    gather_simt_kernel<CONV_BF16_F32, 2>,   gather_simt_kernel<CONV_BF16_F32, 1>,  gather_simt_kernel<CONV_F16_F32, 8>,
    gather_simt_kernel<CONV_F16_F32, 2>,    gather_simt_kernel<CONV_F16_F32, 1>,  gather_simt_kernel<CONV_COPY, 0>,
    gather_simt_kernel<CONV_E4M3_BF16, 0>,  gather_simt_kernel<CONV_E4M3_F16, 0>,  gather_simt_kernel<CONV_E4M3_F32, 0>,
    gather_simt_kernel<CONV_BF16_F32, 0>,   gather_simt_kernel<CONV_F16_F32, 0>,
};

KernelFn tma_convert_kernel_for(int conv) {
  switch (conv) {
    case CONV_E4M3_BF16: return gather_tma_convert_kernel<CONV_E4M3_BF16, 8>;
    case CONV_E4M3_F16: return gather_tma_convert_kernel<CONV_E4M3_F16, 8>;
    case CONV_E4M3_F32: return gather_tma_convert_kernel<CONV_E4M3_F32, 4>;
    case CONV_BF16_F32: return gather_tma_convert_kernel<CONV_BF16_F32, 4>;
    case CONV_F16_F32: return gather_tma_convert_kernel<CONV_F16_F32, 4>;
    default: return nullptr;
  }
}

const KernelFn kAllTmaConvert[] = {
    gather_tma_convert_kernel<CONV_E4M3_BF16, 8>, gather_tma_convert_kernel<CONV_E4M3_F16, 8>,
    gather_tma_convert_kernel<CONV_E4M3_F32, 4>,  gather_tma_convert_kernel<CONV_BF16_F32, 4>,
    gather_tma_convert_kernel<CONV_F16_F32, 4>,
};

// Raises a kernel's dynamic shared memory limit to what the device allows
// per block beyond the kernel's own static shared memory.
int allow_max_dyn_smem(KernelFn k, int optin) {
  cudaFuncAttributes fa;
  if (cudaFuncGetAttributes(&fa, k) != cudaSuccess) return PMG_ERR_CUDA;
  const int limit = optin - static_cast<int>(fa.sharedSizeBytes);
  if (limit <= 0) return PMG_ERR_CUDA;
  return cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, limit) == cudaSuccess ? PMG_OK
                                                                                                        : PMG_ERR_CUDA;
}

// SM count of the current device; raises the dynamic shared memory limit of
// every kernel once per device.
int device_setup(int* sm_count) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return PMG_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return PMG_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_attr_set[dev]) {
    int n = 0, optin = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return PMG_ERR_CUDA;
    if (cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess) return PMG_ERR_CUDA;
    if (allow_max_dyn_smem(reinterpret_cast<KernelFn>(gather_bulk_kernel), optin) != PMG_OK) return PMG_ERR_CUDA;
    for (KernelFn k : kAllSimt)
      if (allow_max_dyn_smem(k, optin) != PMG_OK) return PMG_ERR_CUDA;
    for (KernelFn k : kAllTmaConvert)
      if (allow_max_dyn_smem(k, optin) != PMG_OK) return PMG_ERR_CUDA;
    g_sm_count[dev] = n;
    g_optin_smem[dev] = optin;
    g_attr_set[dev] = true;
  }
  *sm_count = g_sm_count[dev];
  return PMG_OK;
}

// Whether launches carry the programmatic-dependent-launch attribute
// (PMG_PDL=0 turns it off). The kernels wait for the previous grid before
// reading any input, so the attribute only hides launch latency.
bool use_pdl() {
  static const bool v = [] {
    const char* e = std::getenv("PMG_PDL");
    return !(e && e[0] == '0');
  }();
  return v;
}

cudaError_t launch(KernelFn k, int64_t grid, int threads, size_t smem, cudaStream_t stream, const Params& q) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(static_cast<unsigned>(threads));
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = use_pdl() ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, k, q);
}

size_t host_plan_bytes(int R) { return (static_cast<size_t>(3) * R + 2) * sizeof(int32_t); }

// Resident CTAs per SM for (kernel, block size, dynamic shared memory),
// memoised per device so repeated calls skip the occupancy query.
int ctas_per_sm(KernelFn k, int threads, size_t smem, int* out) {
  struct Entry {
    int dev;
    KernelFn k;
    size_t smem;
    int n;
  };
  static Entry cache[64];
  static int used = 0;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return PMG_ERR_CUDA;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    for (int i = 0; i < used; ++i)
      if (cache[i].dev == dev && cache[i].k == k && cache[i].smem == smem) {
        *out = cache[i].n;
        return PMG_OK;
      }
  }
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k, threads, smem) != cudaSuccess) return PMG_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  if (used < 64) cache[used++] = Entry{dev, k, smem, n};
  *out = n;
  return PMG_OK;
}

int launch_one(const Plan& pl, cudaStream_t stream) {
  int sms = 0;
  const int st = device_setup(&sms);
  if (st != PMG_OK) return st;
  Params q = pl.prm;
  const int64_t max_by_rows = (static_cast<int64_t>(q.T) + kMinRowsPerCta - 1) / kMinRowsPerCta;
  if (pl.path == PMG_PATH_BULK) {
    const bool copy = pl.conv == CONV_COPY;
    if (!copy && !q.token_mode) {
      // the converter's ring depends on the rows each CTA will hold
      const int64_t ctas = std::max<int64_t>(1, std::min<int64_t>(static_cast<int64_t>(kCvtCtasPerSm) * sms,
                                                                  max_by_rows));
      set_cvt_ring(q, false, static_cast<int64_t>(q.T) / ctas);
    }
    KernelFn k = copy ? gather_bulk_kernel : tma_convert_kernel_for(pl.conv);
    if (k == nullptr) return PMG_ERR_UNSUPPORTED;
    const int threads = copy ? kBulkThreads : kCvtThreads;
    // the speculative area also keeps the R + 1 entries of cu_seq_lens it read
    const size_t plans = q.token_mode ? 0
                         : q.spec ? 2 * host_plan_bytes(q.R) + (static_cast<size_t>(q.R) + 1) * sizeof(int32_t)
                                  : host_plan_bytes(q.R);
    const size_t smem = static_cast<size_t>(q.stages) * q.stage_bytes + plans;
    int per_sm = 0;
    if (ctas_per_sm(k, threads, smem, &per_sm) != PMG_OK) return PMG_ERR_CUDA;
    if (per_sm < 1) return PMG_ERR_UNSUPPORTED;
    const int64_t grid = std::max<int64_t>(1, std::min<int64_t>(static_cast<int64_t>(per_sm) * sms, max_by_rows));
    if (launch(k, grid, threads, smem, stream, q) != cudaSuccess) return PMG_ERR_CUDA;
  } else {
    KernelFn k = simt_kernel_for(pl.conv, pl.unit);
    if (k == nullptr) return PMG_ERR_UNSUPPORTED;
    const size_t smem = host_plan_bytes(q.R);
    int per_sm = 0;
    if (ctas_per_sm(k, kPlanThreads, smem, &per_sm) != PMG_OK) return PMG_ERR_CUDA;
    if (per_sm < 1) return PMG_ERR_UNSUPPORTED;
    const int64_t grid = std::max<int64_t>(1, std::min<int64_t>(static_cast<int64_t>(per_sm) * sms, max_by_rows));
    if (launch(k, grid, kPlanThreads, smem, stream, q) != cudaSuccess) return PMG_ERR_CUDA;
  }
  return cudaGetLastError() == cudaSuccess ? PMG_OK : PMG_ERR_CUDA;
}

// One call: a single launch, or, beyond PMG_MAX_REQS_PLAN requests, one launch
// per group of requests (pointers into cu_seq_lens, seq_starts and the block
// table advance by the group; output rows come from the absolute cu values,
// so every group writes its own rows; group g reads the highest boundary so
// far from workspace slot (g - 1) % 2 and writes its own to slot g % 2), and
// the clearing of the two slots.
int launch_gather(const Plan& pl, cudaStream_t stream) {
  const Params& q = pl.prm;
  if (q.R <= PMG_MAX_REQS_PLAN) return launch_one(pl, stream);
  int sms = 0;
  int st = device_setup(&sms);
  if (st != PMG_OK) return st;
  int32_t* slots = q.sched + kCarrySlot;
  int64_t g_index = 0;
  for (int64_t r0 = 0; r0 < q.R; r0 += PMG_MAX_REQS_PLAN, ++g_index) {
    Plan g = pl;
    const int32_t rg = static_cast<int32_t>(std::min<int64_t>(PMG_MAX_REQS_PLAN, q.R - r0));
    g.prm.R = rg;
    g.prm.cu = q.cu + r0;
    g.prm.ss = q.ss ? q.ss + r0 : nullptr;
    g.prm.bt = q.bt + r0 * q.bt_stride;
    g.prm.implied_end = (q.implied_end && r0 + rg == q.R) ? 1 : 0;
    g.prm.carry_in = g_index == 0 ? nullptr : slots + ((g_index - 1) & 1);
    g.prm.carry_out = slots + (g_index & 1);
    st = launch_one(g, stream);
    if (st != PMG_OK) return st;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(1);
  cfg.blockDim = dim3(32);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = use_pdl() ? 1 : 0;
  if (cudaLaunchKernelEx(&cfg, clear_carry_kernel, q.sched) != cudaSuccess) return PMG_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? PMG_OK : PMG_ERR_CUDA;
}

}  // namespace

// ---------------------------------------------------------------------------
// Scratch for pmg_gather_noalloc.
//
// Some callers cannot call cudaMalloc: a serving engine that hands nearly all
// of HBM to its own KV-cache pool up front and lets nothing else allocate, a
// plugin inside a framework that owns every allocation, and latency-bound
// paths where cudaMalloc's implicit device synchronisation is not acceptable.
// For them the scheduling counter of the dynamic work split lives here: a
// file-scope device array that every GPU which loads this library holds until
// the process exits. Its size is fixed and small; the gather needs
// PMG_WORKSPACE_INTS of its ints whatever the input sizes.
// ---------------------------------------------------------------------------
constexpr int kNoAllocScratchInts = 64;  // 256 bytes
static_assert(PMG_WORKSPACE_INTS <= kNoAllocScratchInts, "the scheduling counter must fit the static scratch");
static __device__ __align__(256) int32_t g_noalloc_scratch[kNoAllocScratchInts];

namespace {

int32_t* g_noalloc_ptr[kMaxDevices];
bool g_noalloc_ready[kMaxDevices];

// Device address of g_noalloc_scratch on the current device. In host code the
// array's name is only a host-side stand-in, so the address is looked up once
// per device (with that device current) and cached.
int noalloc_scratch(int32_t** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return PMG_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return PMG_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_noalloc_ready[dev]) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || ptr == nullptr) return PMG_ERR_CUDA;
    g_noalloc_ptr[dev] = static_cast<int32_t*>(ptr);
    g_noalloc_ready[dev] = true;
  }
  *out = g_noalloc_ptr[dev];
  return PMG_OK;
}

}  // namespace

extern "C" {

int pmg_gather_noalloc(const void* cache, int64_t cache_block_stride, int64_t cache_token_stride, int64_t num_blocks,
                       const int32_t* block_table, int64_t block_table_stride, const int32_t* cu_seq_lens,
                       const int32_t* seq_starts, int32_t num_reqs, int64_t total_tokens, int32_t block_size,
                       int32_t entry_size, int32_t src_dtype, int32_t dst_dtype, const float* scale, void* dst,
                       int64_t dst_token_stride, int32_t* error_flag, void* stream) {
  // every check of pmg_gather first, on the host, with no CUDA call
  Plan pl;
  // the static scratch stands in for the workspace (its address is only known
  // after the CUDA set-up below; any 16-byte aligned non-null value passes the
  // host checks)
  int32_t* const placeholder = reinterpret_cast<int32_t*>(static_cast<uintptr_t>(256));
  int st = make_plan(cache, cache_block_stride, cache_token_stride, num_blocks, block_table, block_table_stride,
                     cu_seq_lens, seq_starts, num_reqs, total_tokens, block_size, entry_size, src_dtype, dst_dtype,
                     scale, dst, dst_token_stride, error_flag, placeholder, 0u, pl);
  if (st != PMG_OK) return st;
  if (pl.path == PMG_PATH_NONE) return PMG_OK;
  int32_t* scratch = nullptr;
  st = noalloc_scratch(&scratch);
  if (st != PMG_OK) return st;
  // The array keeps whatever the last call left; the claim counter must start
  // at zero, so clear it on this stream ahead of the launch.
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(scratch, 0, PMG_WORKSPACE_INTS * sizeof(int32_t), s) != cudaSuccess) return PMG_ERR_CUDA;
  pl.prm.sched = scratch;
  return launch_gather(pl, s);
}


int pmg_debug_noalloc_scratch(void** device_ptr, int64_t* num_ints) {
  if (device_ptr == nullptr || num_ints == nullptr) return PMG_ERR_NULL;
  int32_t* scratch = nullptr;
  const int st = noalloc_scratch(&scratch);
  if (st != PMG_OK) return st;
  *device_ptr = scratch;
  *num_ints = kNoAllocScratchInts;
  return PMG_OK;
}

int pmg_gather_ex(const void* cache, int64_t cache_block_stride, int64_t cache_token_stride, int64_t num_blocks,
                  const int32_t* block_table, int64_t block_table_stride, const int32_t* cu_seq_lens,
                  const int32_t* seq_starts, int32_t num_reqs, int64_t total_tokens, int32_t block_size,
                  int32_t entry_size, int32_t src_dtype, int32_t dst_dtype, const float* scale, void* dst,
                  int64_t dst_token_stride, int32_t* error_flag, int32_t* workspace, void* stream,
                  uint32_t options) {
  Plan pl;
  const int st = make_plan(cache, cache_block_stride, cache_token_stride, num_blocks, block_table, block_table_stride,
                           cu_seq_lens, seq_starts, num_reqs, total_tokens, block_size, entry_size, src_dtype,
                           dst_dtype, scale, dst, dst_token_stride, error_flag, workspace, options, pl);
  if (st != PMG_OK) return st;
  if (pl.path == PMG_PATH_NONE) return PMG_OK;
  return launch_gather(pl, static_cast<cudaStream_t>(stream));
}

int pmg_gather_tokens(const void* cache, int64_t cache_block_stride, int64_t cache_token_stride, int64_t num_blocks,
                      const int32_t* block_table, int64_t block_table_stride, const int32_t* token_to_seq,
                      const int32_t* cu_seq_lens, int32_t num_reqs, int64_t num_tokens, int32_t block_size,
                      int32_t entry_size, int32_t src_dtype, int32_t dst_dtype, const float* scale, void* dst,
                      int64_t dst_token_stride, int32_t* error_flag, int32_t* workspace, void* stream,
                      uint32_t options) {
  const int conv = conv_of(src_dtype, dst_dtype);
  if (conv < 0) return PMG_ERR_DTYPE;
  if (num_reqs < 0 || num_tokens < 0 || block_size < 1 || entry_size < 1 || num_blocks < 0 ||
      block_table_stride < 0 || cache_block_stride < 0 || cache_token_stride < 0 || dst_token_stride < entry_size)
    return PMG_ERR_ARG;
  if (options & ~(PMG_OPT_FORCE_SIMT | PMG_OPT_FORCE_SCALAR | PMG_OPT_EARLY_METADATA)) return PMG_ERR_ARG;
  const int es = elem_bytes(src_dtype), ed = elem_bytes(dst_dtype);
  if (static_cast<int64_t>(entry_size) * ed > INT32_MAX || num_tokens > INT32_MAX) return PMG_ERR_UNSUPPORTED;
  if (num_tokens == 0) return PMG_OK;
  if (token_to_seq == nullptr || dst == nullptr) return PMG_ERR_NULL;
  if (num_reqs > 0 && (cache == nullptr || block_table == nullptr || cu_seq_lens == nullptr)) return PMG_ERR_NULL;
  if (!aligned(cache, es) || !aligned(dst, ed) || !aligned(block_table, 4) || !aligned(token_to_seq, 4) ||
      !aligned(cu_seq_lens, 4) || (scale != nullptr && !aligned(scale, 4)) ||
      (error_flag != nullptr && !aligned(error_flag, 4)) || (workspace != nullptr && !aligned(workspace, 16)))
    return PMG_ERR_ALIGN;
  if (cache_block_stride > INT64_MAX / es / 2 || cache_token_stride > INT64_MAX / es / 2 ||
      dst_token_stride > INT64_MAX / ed / 2)
    return PMG_ERR_ARG;
  if (num_reqs > 0 && (options & (PMG_OPT_FORCE_SIMT | PMG_OPT_FORCE_SCALAR)) == 0) {
    // The TMA pipelines in token mode: the scheduler warp resolves 32 tokens
    // per batch and merges runs whose source rows are adjacent into segments.
    // The page plan's checks and path choice run with a single stand-in
    // request, since token mode plans nothing per request.
    Plan pl;
    const int st = make_plan(cache, cache_block_stride, cache_token_stride, num_blocks, block_table,
                             block_table_stride, cu_seq_lens, nullptr, 1, num_tokens, block_size, entry_size,
                             src_dtype, dst_dtype, scale, dst, dst_token_stride, error_flag, workspace,
                             options & PMG_OPT_EARLY_METADATA, pl);
    if (st == PMG_OK && pl.path == PMG_PATH_BULK) {
      pl.prm.R = num_reqs;
      pl.prm.t2s = token_to_seq;
      pl.prm.token_mode = 1;
      // the per-token mode's own ring sizes and static head
      if (pl.conv == CONV_COPY) set_bulk_ring(pl.prm, false);
      else set_cvt_ring(pl.prm, true, -1);
      pl.prm.sched_head_stages = sched_head_stages(true);
      return launch_one(pl, static_cast<cudaStream_t>(stream));
    }
  }
  TokParams q{};
  q.cache = static_cast<const uint8_t*>(cache);
  q.blk_stride_b = cache_block_stride * es;
  q.tok_stride_b = cache_token_stride * es;
  q.num_blocks = num_blocks;
  q.bt = block_table;
  q.bt_stride = block_table_stride;
  q.t2s = token_to_seq;
  q.cu = cu_seq_lens;
  q.T = num_tokens;
  q.R = num_reqs;
  q.B = block_size;
  q.dst = static_cast<uint8_t*>(dst);
  q.dst_stride_b = dst_token_stride * ed;
  q.scale = scale;
  q.err = error_flag;
  int unit = pick_unit(conv, es, ed, entry_size, cache, q.blk_stride_b, q.tok_stride_b, dst, q.dst_stride_b);
  if (options & PMG_OPT_FORCE_SCALAR) unit = (conv == CONV_COPY) ? es : 1;
  const int64_t upr = (conv == CONV_COPY) ? static_cast<int64_t>(entry_size) * es / unit : entry_size / unit;
  if (32ull * static_cast<uint64_t>(upr) >= (1ull << 32)) return PMG_ERR_UNSUPPORTED;
  q.units_per_row = static_cast<int32_t>(upr);
  uint32_t l = 0;
  while ((1ull << l) < static_cast<uint64_t>(upr)) ++l;
  q.upr_magic = static_cast<uint32_t>((((1ull << l) - static_cast<uint64_t>(upr)) << 32) / static_cast<uint64_t>(upr) + 1);
  q.upr_shift = static_cast<int32_t>(l);
  TokKernelFn k = tokens_kernel_for(conv, unit);
  if (k == nullptr) return PMG_ERR_UNSUPPORTED;
  int sms = 0;
  int st = device_setup(&sms);
  if (st != PMG_OK) return st;
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k, kTokThreads, 0) != cudaSuccess || per_sm < 1)
    return PMG_ERR_CUDA;
  // smaller tiles until there are at least four per resident warp
  const int64_t resident_warps = static_cast<int64_t>(per_sm) * sms * (kTokThreads / 32);
  int32_t tr = 32;
  while (tr > 8 && (num_tokens + tr - 1) / tr < 4 * resident_warps) tr /= 2;
  // PMG_TOKEN_TILE (8, 16 or 32) overrides the choice for tuning sweeps
  static const int tile_env = env_int("PMG_TOKEN_TILE", 0, 0, 32);
  if (tile_env == 8 || tile_env == 16 || tile_env == 32) tr = tile_env;
  q.tile_rows = tr;
  const int64_t tiles = (num_tokens + tr - 1) / tr;
  const int64_t need = (tiles + kTokThreads / 32 - 1) / (kTokThreads / 32);
  const int64_t grid = std::max<int64_t>(1, std::min<int64_t>(static_cast<int64_t>(per_sm) * sms, need));
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(kTokThreads);
  cfg.stream = static_cast<cudaStream_t>(stream);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = use_pdl() ? 1 : 0;
  if (cudaLaunchKernelEx(&cfg, k, q) != cudaSuccess) return PMG_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? PMG_OK : PMG_ERR_CUDA;
}

int pmg_gather(const void* cache, int64_t cache_block_stride, int64_t cache_token_stride, int64_t num_blocks,
               const int32_t* block_table, int64_t block_table_stride, const int32_t* cu_seq_lens,
               const int32_t* seq_starts, int32_t num_reqs, int64_t total_tokens, int32_t block_size,
               int32_t entry_size, int32_t src_dtype, int32_t dst_dtype, const float* scale, void* dst,
               int64_t dst_token_stride, int32_t* error_flag, void* stream) {
  return pmg_gather_ex(cache, cache_block_stride, cache_token_stride, num_blocks, block_table, block_table_stride,
                       cu_seq_lens, seq_starts, num_reqs, total_tokens, block_size, entry_size, src_dtype, dst_dtype,
                       scale, dst, dst_token_stride, error_flag, nullptr, stream, 0u);
}

int pmg_select_path(const void* cache, int64_t cache_block_stride, int64_t cache_token_stride, int64_t num_blocks,
                    const int32_t* block_table, int64_t block_table_stride, const int32_t* cu_seq_lens,
                    int32_t num_reqs, int64_t total_tokens, int32_t block_size, int32_t entry_size, int32_t src_dtype,
                    int32_t dst_dtype, const void* dst, int64_t dst_token_stride, uint32_t options, int32_t* path_out,
                    int32_t* unit_elems_out) {
  Plan pl;
  // the path does not depend on whether a workspace is given; a stand-in lets
  // large batches through the host checks
  int32_t* const placeholder = reinterpret_cast<int32_t*>(static_cast<uintptr_t>(256));
  const int st = make_plan(cache, cache_block_stride, cache_token_stride, num_blocks, block_table, block_table_stride,
                           cu_seq_lens, nullptr, num_reqs, total_tokens, block_size, entry_size, src_dtype, dst_dtype,
                           nullptr, dst, dst_token_stride, nullptr, placeholder, options, pl);
  if (st != PMG_OK) return st;
  if (path_out) *path_out = pl.path;
  if (unit_elems_out) {
    int u = pl.unit;
    // report elements, not bytes, for a byte copy
    if (pl.path != PMG_PATH_BULK && pl.path != PMG_PATH_NONE && pl.conv == CONV_COPY) u /= elem_bytes(src_dtype);
    *unit_elems_out = (pl.path == PMG_PATH_BULK || pl.path == PMG_PATH_NONE) ? 0 : u;
  }
  return PMG_OK;
}

int pmg_debug_plan(const int32_t* cu_seq_lens, const int32_t* seq_starts, int32_t num_reqs, int64_t total_tokens,
                   int32_t block_size, int32_t* tasks_out, int64_t max_tasks, int64_t* num_tasks_out,
                   int32_t* error_flag, void* stream, uint32_t options) {
  if (num_reqs < 0 || total_tokens < 0 || block_size < 1 || max_tasks < 0) return PMG_ERR_ARG;
  if (options & ~PMG_OPT_IMPLIED_END) return PMG_ERR_ARG;
  if (num_reqs > PMG_MAX_REQS_PLAN) return PMG_ERR_UNSUPPORTED;
  if (num_tasks_out == nullptr || (num_reqs > 0 && cu_seq_lens == nullptr) || (max_tasks > 0 && tasks_out == nullptr))
    return PMG_ERR_NULL;
  Params q{};
  q.cu = cu_seq_lens;
  q.ss = seq_starts;
  q.R = num_reqs;
  q.T = static_cast<int32_t>(total_tokens < INT32_MAX ? total_tokens : INT32_MAX);
  q.B = block_size;
  q.implied_end = (options & PMG_OPT_IMPLIED_END) ? 1 : 0;
  q.err = error_flag;
  int sms = 0;
  const int st = device_setup(&sms);
  if (st != PMG_OK) return st;
  {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return PMG_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_plan_attr_set[dev]) {
      cudaFuncAttributes fa;
      if (cudaFuncGetAttributes(&fa, debug_plan_kernel) != cudaSuccess) return PMG_ERR_CUDA;
      if (cudaFuncSetAttribute(debug_plan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               g_optin_smem[dev] - static_cast<int>(fa.sharedSizeBytes)) != cudaSuccess)
        return PMG_ERR_CUDA;
      g_plan_attr_set[dev] = true;
    }
  }
  debug_plan_kernel<<<1, kPlanThreads, host_plan_bytes(num_reqs), static_cast<cudaStream_t>(stream)>>>(
      q, tasks_out, max_tasks, num_tasks_out);
  return cudaGetLastError() == cudaSuccess ? PMG_OK : PMG_ERR_CUDA;
}

const char* pmg_status_string(int status) {
  switch (status) {
    case PMG_OK: return "PMG_OK: success";
    case PMG_ERR_NULL: return "PMG_ERR_NULL: a required pointer is NULL";
    case PMG_ERR_ARG: return "PMG_ERR_ARG: a size, stride or option is out of range";
    case PMG_ERR_DTYPE: return "PMG_ERR_DTYPE: unknown dtype or unsupported (src, dst) pair";
    case PMG_ERR_ALIGN: return "PMG_ERR_ALIGN: a pointer is not aligned to its element size";
    case PMG_ERR_UNSUPPORTED: return "PMG_ERR_UNSUPPORTED: request beyond this build's limits";
    case PMG_ERR_CUDA: return "PMG_ERR_CUDA: a CUDA runtime call or kernel launch failed";
    default: return "unknown pmg status";
  }
}

int pmg_version(void) { return 1; }

}  // extern "C"

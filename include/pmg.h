/*
 * pmg.h — C ABI of the GB300 paged MLA KV-cache gather.
 *
 * The operation is the one described in "MLA cache gather scheduled per
 * logical page" (prhub.com.cn, vllm PR #51739). The binding it documents is
 * ops.cp_gather_cache(src_cache, dst, block_table, cu_seq_lens, batch_size,
 * seq_starts) (section "关键源码片段", test
 * test_cp_gather_cache_mla_large_uneven_sequences). For every request r it
 * reads the cached-context entries of tokens [start_r, start_r + len_r) out of
 * a paged cache, through that request's block-table row, and writes them back
 * to back into a contiguous workspace starting at row min(cu_seq_lens[r], T).
 * The write is a byte copy, an FP8 E4M3 dequant (section "实现拆解" item 1:
 * the FP8 -> BF16 upconvert kernel), or a widening cast (the "maybe dequant"
 * kernel with kv_cache_dtype "auto").
 *
 * Conventions for every entry point:
 *  - Arrays are device memory unless stated otherwise; sizes, strides and
 *    dtypes are host values. The caller owns every pointer. The library keeps
 *    no per-call state and allocates no memory.
 *  - Strides are in ELEMENTS of the array they index; the last (entry)
 *    dimension has stride 1.
 *  - `stream` is a cudaStream_t passed as void* (NULL = the legacy default
 *    stream). Calls are asynchronous on that stream and never synchronise.
 *  - Kernels are launched with programmatic dependent launch. With up to 256
 *    requests (and for pmg_gather_tokens) the TMA paths read cu_seq_lens,
 *    seq_starts, token_to_seq and block_table once before the previous kernel
 *    in the stream has finished, plan from those values, and read every value
 *    they used again after it has finished; they use the early plan only if
 *    nothing changed. The result is always that of the inputs as they are
 *    when the previous kernel has finished. Nothing is written, and no cache,
 *    scale or workspace byte is read into a result, before that point.
 *  - Host-detected errors return a non-zero pmg_status synchronously; nothing
 *    is launched and no output is touched.
 *  - Data errors found on the device (values inside cu_seq_lens, seq_starts or
 *    block_table) are not host errors: the affected rows are skipped and left
 *    untouched, a PMG_FLAG_* bit is OR-ed into *error_flag (if non-NULL), and
 *    the call still returns PMG_OK. The caller reads the flag when it likes.
 */
#ifndef PMG_H_
#define PMG_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Element types. PMG_FP8_E4M3 is OCP E4M3 ("fn": bias 7, no infinities,
 * S.1111.111 is NaN). PMG_U8 is raw bytes. */
typedef enum pmg_dtype {
  PMG_BF16 = 0,
  PMG_FP16 = 1,
  PMG_FP32 = 2,
  PMG_FP8_E4M3 = 3,
  PMG_U8 = 4
} pmg_dtype;

typedef enum pmg_status {
  PMG_OK = 0,
  PMG_ERR_NULL = 1,        /* a required pointer is NULL */
  PMG_ERR_ARG = 2,         /* a size or stride is out of range */
  PMG_ERR_DTYPE = 3,       /* unknown dtype or unsupported (src, dst) pair */
  PMG_ERR_ALIGN = 4,       /* a pointer is not aligned to its element size */
  PMG_ERR_UNSUPPORTED = 5, /* valid request beyond this build's limits */
  PMG_ERR_CUDA = 6         /* a CUDA runtime call or the launch failed */
} pmg_status;

/* Bits OR-ed into *error_flag by the device. */
#define PMG_FLAG_LOGICAL_BLOCK 1 /* logical block >= block_table_stride: page skipped */
#define PMG_FLAG_PHYS_BLOCK 2    /* block_table entry outside [0, num_blocks): page skipped */
#define PMG_FLAG_SEQ_START 4     /* seq_starts[r] < 0 with len_r > 0: request skipped */
#define PMG_FLAG_CU_ORDER 8      /* a request's rows start below row 0 or an earlier cu boundary: request skipped */
#define PMG_FLAG_TIMEOUT 16      /* a bounded device wait ran out: output incomplete */
#define PMG_FLAG_TOKEN 32        /* pmg_gather_tokens: request id or row range of a token invalid: token skipped */

/* Requests one launch plans in shared memory. A call with more requests needs
 * a workspace (pmg_gather_ex, or pmg_gather_noalloc) and runs as one launch
 * per group of PMG_MAX_REQS_PLAN requests (each group passes the highest
 * cu_seq_lens boundary so far to the next through the workspace) and a final
 * one-thread launch; without a workspace it returns PMG_ERR_UNSUPPORTED.
 * pmg_debug_plan is limited to this many. */
#define PMG_MAX_REQS_PLAN 4096

/* Most requests one call accepts; more return PMG_ERR_UNSUPPORTED. */
#define PMG_MAX_REQS (1 << 20)

/* Options of pmg_gather_ex. */
#define PMG_OPT_FORCE_SIMT 1u      /* use the SIMT vector kernel even where TMA bulk applies */
#define PMG_OPT_FORCE_SCALAR 2u    /* use one-element units (the scalar-stride path) */
#define PMG_OPT_IMPLIED_END 4u     /* cu_seq_lens has num_reqs entries; the last request ends at total_tokens */
/* The caller promises that no kernel still running in the stream when this
 * call starts writes cu_seq_lens, seq_starts, block_table or error_flag. The
 * TMA paths then read them (plan and first block ids) while the previous grid
 * finishes, under programmatic dependent launch; the cache, the scale, the
 * workspace and dst are still touched only after the previous grid completes.
 * Ignored by the SIMT paths and for more than PMG_MAX_REQS_PLAN requests. */
#define PMG_OPT_EARLY_METADATA 8u

/* Data-movement paths (pmg_select_path). */
typedef enum pmg_path {
  PMG_PATH_NONE = 0,   /* nothing to do (no rows or no requests): no launch */
  PMG_PATH_BULK = 1,   /* TMA 1-D bulk loads of 16-B aligned source rows into a shared ring; byte copies
                          leave by bulk stores, converting gathers by 16-byte stores of converter warps */
  PMG_PATH_VECTOR = 2, /* SIMT loads/stores of several elements per thread */
  PMG_PATH_SCALAR = 3, /* SIMT, one element per access (any alignment) */
  PMG_PATH_REALIGN = 4 /* rows of at least 16 output bytes that the TMA paths cannot take (byte
                          copies whose rows are not 16-B aligned; converting gathers whose rows are
                          not 16-B aligned or not a whole number of converter units): each
                          16-B-aligned word of a destination row is assembled from the aligned
                          16-B source words holding its bytes (converted for a converting gather);
                          whole words by 16-B stores, the partial first and last words of a row
                          byte by byte */
} pmg_path;

/*
 * pmg_gather — the paged gather (the call of ops.cp_gather_cache in the
 * section "关键源码片段", with strides, dtypes, scale and stream made explicit).
 *
 *  cache               [num_blocks, block_size, >= entry_size] of src_dtype.
 *  cache_block_stride  elements between consecutive blocks (>= 0).
 *  cache_token_stride  elements between consecutive slots of a block (>= 0);
 *                      a value larger than entry_size is a padded row.
 *  num_blocks          physical blocks; a block id outside [0, num_blocks) is
 *                      a data error (PMG_FLAG_PHYS_BLOCK).
 *  block_table         int32 [num_reqs, block_table_stride]: row r maps logical
 *                      block i of request r (tokens [i*block_size,
 *                      (i+1)*block_size) of its context) to a physical block.
 *  cu_seq_lens         int32 [num_reqs + 1]: request r owns output rows
 *                      [min(cu[r], T), min(cu[r+1], T)); its length is
 *                      max(min(cu[r+1], T) - min(cu[r], T), 0), so a decrease
 *                      only gives a request no rows. A request with rows whose
 *                      first row min(cu[r], T) is below 0 or below an earlier
 *                      boundary min(cu[j], T), j < r (its rows would overlap
 *                      earlier rows or come out of order) is skipped and
 *                      PMG_FLAG_CU_ORDER is set; the other requests are copied.
 *  seq_starts          int32 [num_reqs] or NULL (all zero): the first context
 *                      token of request r to copy.
 *  num_reqs            0 <= num_reqs <= PMG_MAX_REQS_PLAN (pmg_gather) or
 *                      PMG_MAX_REQS (pmg_gather_ex with a workspace).
 *  total_tokens        T >= 0, rows of dst. Rows >= T are never written.
 *  block_size          tokens per block, >= 1.
 *  entry_size          elements per token entry, >= 1.
 *  src_dtype/dst_dtype same dtype: byte copy. PMG_FP8_E4M3 -> PMG_BF16,
 *                      PMG_FP16 or PMG_FP32: dst = round_to_nearest_even(
 *                      fp32(x) *fp32 scale). PMG_BF16 or PMG_FP16 -> PMG_FP32:
 *                      exact widening, no scale. Other pairs: PMG_ERR_DTYPE.
 *  scale               device fp32 scalar, or NULL for 1.0. Read only when the
 *                      source is PMG_FP8_E4M3 and the dtypes differ.
 *  dst                 [>= T, dst_token_stride] of dst_dtype.
 *  dst_token_stride    elements between output rows, >= entry_size.
 *  error_flag          device int32 or NULL; PMG_FLAG_* bits are OR-ed in.
 *  stream              cudaStream_t.
 * Returns a pmg_status. Only rows of valid pages are written; every other
 * element of dst (other rows, columns past entry_size) is left as it was.
 */
int pmg_gather(const void* cache, int64_t cache_block_stride, int64_t cache_token_stride, int64_t num_blocks,
               const int32_t* block_table, int64_t block_table_stride, const int32_t* cu_seq_lens,
               const int32_t* seq_starts, int32_t num_reqs, int64_t total_tokens, int32_t block_size,
               int32_t entry_size, int32_t src_dtype, int32_t dst_dtype, const float* scale, void* dst,
               int64_t dst_token_stride, int32_t* error_flag, void* stream);

/* Size of the scheduling workspace of pmg_gather_ex, in int32 elements. */
#define PMG_WORKSPACE_INTS 4

/*
 * pmg_gather_ex — pmg_gather with a scheduling workspace and PMG_OPT_* options
 * (workspace NULL and options 0 is exactly pmg_gather).
 *
 *  workspace  device int32 [PMG_WORKSPACE_INTS], 16-byte aligned, or NULL.
 *             With a workspace, the TMA paths split a quarter of the output
 *             rows evenly up front and hand out the rest in small pieces
 *             through an atomic counter, so CTAs
 *             whose memory traffic is served faster take more of the work
 *             (without one, every CTA gets one equal share). The caller zeroes
 *             it once before first use; every call that completes leaves it
 *             zeroed again. Calls that may run concurrently (different
 *             streams) need separate workspaces: two calls sharing one at the
 *             same time race. After a call that reported PMG_FLAG_TIMEOUT,
 *             zero it again. The SIMT paths ignore it.
 *  options    PMG_OPT_* bits. PMG_OPT_IMPLIED_END selects the page's other
 *             calling convention (map_gather_page_task with
 *             has_terminal_start = false, section "关键源码片段"): cu_seq_lens
 *             then holds num_reqs entries and request num_reqs-1 ends at
 *             total_tokens.
 */
int pmg_gather_ex(const void* cache, int64_t cache_block_stride, int64_t cache_token_stride, int64_t num_blocks,
                  const int32_t* block_table, int64_t block_table_stride, const int32_t* cu_seq_lens,
                  const int32_t* seq_starts, int32_t num_reqs, int64_t total_tokens, int32_t block_size,
                  int32_t entry_size, int32_t src_dtype, int32_t dst_dtype, const float* scale, void* dst,
                  int64_t dst_token_stride, int32_t* error_flag, int32_t* workspace, void* stream,
                  uint32_t options);

/*
 * pmg_gather_noalloc — pmg_gather with the dynamic work split of
 * pmg_gather_ex, for callers that cannot allocate device memory. The pages
 * have no counterpart of this entry point.
 *
 * Who needs it: callers that may not call cudaMalloc. A serving engine that
 * reserves nearly all of HBM for its own KV-cache pool at start-up leaves no
 * room for, and often forbids, allocations outside that pool; a caller on a
 * latency-bound path cannot afford cudaMalloc's implicit device
 * synchronisation; and a plugin inside a host framework that owns every
 * allocation may only use memory handed to it.
 *
 * The arguments, their meaning and the results are those of pmg_gather; the
 * caller still passes every input and output. Instead of a caller workspace,
 * the scheduling counter lives in a 256-byte static device array inside the
 * library, which every GPU that loads the library holds until the process
 * exits. The call needs PMG_WORKSPACE_INTS of those ints whatever the input
 * sizes; inputs beyond pmg_gather_ex's limits (num_reqs > PMG_MAX_REQS, ...)
 * are rejected with the same statuses (PMG_ERR_UNSUPPORTED, PMG_ERR_ARG, ...).
 * It calls no cudaMalloc, cudaFree or other allocating routine: before each
 * launch it clears the counter with cudaMemsetAsync on `stream`.
 *
 * The first call on a device looks up the array's device address
 * (cudaGetSymbolAddress) with that device current and caches it; make that
 * first call before any stream capture. Every call shares the one array: calls
 * that overlap on the GPU (different streams, or several host threads) race on
 * it and may produce wrong output; serialise them, or use pmg_gather_ex with a
 * workspace per stream.
 */

/*
 * pmg_debug_noalloc_scratch — test hook: the device address of the static
 * scratch pmg_gather_noalloc uses on the current device, and its size in
 * int32 elements. Like the first pmg_gather_noalloc call it performs the
 * one-time address lookup for the device. Tests use it to leave stale values
 * in the array and check that a call still starts from a cleared counter.
 * Writing to the array while a pmg_gather_noalloc call runs corrupts that call.
 */
int pmg_debug_noalloc_scratch(void** device_ptr, int64_t* num_ints);
int pmg_gather_noalloc(const void* cache, int64_t cache_block_stride, int64_t cache_token_stride,
                       int64_t num_blocks, const int32_t* block_table, int64_t block_table_stride,
                       const int32_t* cu_seq_lens, const int32_t* seq_starts, int32_t num_reqs,
                       int64_t total_tokens, int32_t block_size, int32_t entry_size, int32_t src_dtype,
                       int32_t dst_dtype, const float* scale, void* dst, int64_t dst_token_stride,
                       int32_t* error_flag, void* stream);

/*
 * pmg_gather_tokens — per-token indexed gather, the gather pattern of the
 * indexer kernel on the page "indexer kernels take shape arguments at run
 * time" (prhub.com.cn, vllm PR #56153, section "关键源码片段":
 * _cp_gather_indexer_quant_cache_kernel). Instead of deriving each output
 * row's request from cu_seq_lens, the caller names it:
 *
 *  token_to_seq   int32 [num_tokens], device: request of output row t.
 *  cu_seq_lens    int32 [num_reqs + 1], device: request b owns output rows
 *                 [cu[b], cu[b+1]); row t reads context position t - cu[b].
 *  num_tokens     rows of dst to produce, 0 <= num_tokens <= INT32_MAX.
 *  workspace      NULL, or PMG_WORKSPACE_INTS zeroed int32 on the device
 *                 (16-byte aligned), as in pmg_gather_ex: it lets the TMA
 *                 path balance rows across CTAs dynamically.
 *  options        bitwise OR of PMG_OPT_FORCE_SIMT, PMG_OPT_FORCE_SCALAR and
 *                 PMG_OPT_EARLY_METADATA (read for token_to_seq as well).
 *                 Without a FORCE option, rows whose 16-byte alignment fits
 *                 the TMA path (PMG_PATH_BULK of pmg_select_path) go through
 *                 it: consecutive tokens whose cache rows are adjacent travel
 *                 as one bulk copy. Otherwise a SIMT kernel copies each row.
 * Every other argument is as in pmg_gather (there is no seq_starts). Output
 * row t = convert(cache[block_table[b, p / block_size], p % block_size]) with
 * b = token_to_seq[t], p = t - cu[b]. Every index is checked before use: a
 * request id outside [0, num_reqs) or a row outside [cu[b], cu[b+1]) skips the
 * row (PMG_FLAG_TOKEN), a column past the block-table row or a block id outside
 * [0, num_blocks) skips it too (PMG_FLAG_LOGICAL_BLOCK, PMG_FLAG_PHYS_BLOCK).
 * Skipped rows are left untouched. Shapes are runtime arguments only.
 */
int pmg_gather_tokens(const void* cache, int64_t cache_block_stride, int64_t cache_token_stride, int64_t num_blocks,
                      const int32_t* block_table, int64_t block_table_stride, const int32_t* token_to_seq,
                      const int32_t* cu_seq_lens, int32_t num_reqs, int64_t num_tokens, int32_t block_size,
                      int32_t entry_size, int32_t src_dtype, int32_t dst_dtype, const float* scale, void* dst,
                      int64_t dst_token_stride, int32_t* error_flag, int32_t* workspace, void* stream,
                      uint32_t options);

/*
 * pmg_select_path — host-only: validates the layout arguments of a gather the
 * way pmg_gather_ex does and reports the path and the elements moved per
 * access it would use. Makes no CUDA call. Pointers are only inspected for
 * alignment and NULL. *path_out receives a pmg_path, *unit_elems_out the
 * elements per access (0 for PMG_PATH_NONE, PMG_PATH_BULK and PMG_PATH_REALIGN).
 */
int pmg_select_path(const void* cache, int64_t cache_block_stride, int64_t cache_token_stride,
                    int64_t num_blocks, const int32_t* block_table, int64_t block_table_stride,
                    const int32_t* cu_seq_lens, int32_t num_reqs, int64_t total_tokens, int32_t block_size,
                    int32_t entry_size, int32_t src_dtype, int32_t dst_dtype, const void* dst,
                    int64_t dst_token_stride, uint32_t options, int32_t* path_out, int32_t* unit_elems_out);

/*
 * pmg_debug_plan — runs the device page-task mapper alone (section
 * "实现拆解" item 1 and the GatherPageTask / map_gather_page_task listing:
 * a flat task id -> (req, logical_block, page_token_begin, page_token_end,
 * output_token_begin)). Here the mapper is a prefix sum over per-request page
 * counts plus a binary search, the same device code the gather uses.
 *  tasks_out      device int32 [max_tasks, 5]: task t is written as
 *                 {req, logical_block, page_token_begin, page_token_end,
 *                 output_token_begin} for t < min(num_tasks, max_tasks).
 *  num_tasks_out  device int64 scalar: the number of tasks.
 *  error_flag     as in pmg_gather (PMG_FLAG_SEQ_START, PMG_FLAG_CU_ORDER).
 * A request with len 0, a negative start, or rows starting below an earlier
 * cu_seq_lens boundary (PMG_FLAG_CU_ORDER) has no task. The block table is
 * not read.
 */
int pmg_debug_plan(const int32_t* cu_seq_lens, const int32_t* seq_starts, int32_t num_reqs, int64_t total_tokens,
                   int32_t block_size, int32_t* tasks_out, int64_t max_tasks, int64_t* num_tasks_out,
                   int32_t* error_flag, void* stream, uint32_t options);

/* Static description of a status code. Never NULL. */
const char* pmg_status_string(int status);

/* ABI version of this library: 1. */
int pmg_version(void);

#ifdef __cplusplus
}
#endif

#endif /* PMG_H_ */

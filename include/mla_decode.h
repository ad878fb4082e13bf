/*
 * mla_decode.h -- C ABI of the GB300 (sm_103a) MLA speculative-verify decode library
 * (libmla_verify_sm103.so).
 *
 * Operation (sglang PR #33650 "[Kimi-K3] Allow DSPARK verify on cutedsl_mla
 * (fold_sq)": the isolated MLA decode of the "Which decode backend?" section, MQA
 * with one latent KV head; the fold rule of its "Why" paragraph; the split-KV
 * reduction of its GPU-timeline section):
 *
 *   For request b with ctx = seq_lens[b] cached keys (its q = q_lens[b] verify
 *   tokens included), verify token i in [0, q) and query head h in [0, H):
 *     key j in [0, ctx - q + i + 1) lives in cache row
 *       page_table[b * page_table_stride + j / 64] * 64 + j % 64,
 *     Khat_j = that row's 576 values (times kv_scale for an fp8 e4m3 cache),
 *     s_j = sm_scale * <Q[b, i, h, 0:576], Khat_j>,
 *     out[b, i, h, :] = sum_j softmax(s)_j * Khat_j[0:512]     (bf16),
 *     lse[b, i, h]    = ln sum_j exp(s_j)                     (fp32, natural log).
 *
 *   The q tokens of a request are folded into the tile rows (fold_sq): F is the
 *   largest divisor of q with H * F <= 128, and each group of F tokens x H heads
 *   reads the paged cache once instead of once per token. Folding and split-KV
 *   change the order of the arithmetic only, never the result.
 *
 * Layouts (row-major, dense, all device pointers 16-byte aligned):
 *   q          [sum(q_lens), H, 576] bf16, requests concatenated in batch order
 *   kv_cache   [num_pages, 64, 576]  bf16, or fp8 e4m3 (OCP "e4m3fn") codes
 *   page_table [batch, page_table_stride] int32 physical page ids
 *   seq_lens, q_lens [batch] int32 (device copies of the values given to the plan)
 *   out        [sum(q_lens), H, 512] bf16
 *   lse        [sum(q_lens), H] fp32 (may be NULL)
 *
 * Ownership: the caller owns and allocates every buffer. The library allocates
 * no memory, never synchronises the stream, and keeps no state between calls
 * apart from a thread-local error string (and the fixed device array behind
 * mla_decode_run_static_ws, declared below).
 *
 * Errors: every entry point returns an mla_status; on failure mla_last_error()
 * describes the cause. Arguments are checked on the host before any launch.
 * Device-side problems (a bounded wait that ran out, seq_lens/q_lens that differ
 * from the plan, a page id outside [0, num_pages)) never trap: the kernels stop
 * the affected work item and OR a code into *status_dev (if given), which the
 * caller reads after synchronising.
 */
#ifndef MLA_DECODE_H_
#define MLA_DECODE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MLA_OK = 0,
  MLA_ERR_INVALID_ARG = -1,   /* a null pointer, a bad size, q_len > seq_len, ... */
  MLA_ERR_UNSUPPORTED = -2,   /* H outside [1, 128], page size other than 64, no sm_103 device */
  MLA_ERR_BUFFER = -3,        /* plan buffer or workspace too small */
  MLA_ERR_CUDA = -4,          /* a CUDA runtime/driver call failed */
  MLA_ERR_PLAN = -5           /* plan bytes do not describe a plan of this library */
} mla_status;

typedef enum { MLA_KV_BF16 = 0, MLA_KV_FP8_E4M3 = 1 } mla_kv_dtype;

/* Bits OR-ed into *status_dev by the kernels. */
#define MLA_DEVICE_WAIT_TIMEOUT 0x1     /* a bounded mbarrier wait ran out */
#define MLA_DEVICE_PLAN_MISMATCH 0x2    /* seq_lens / q_lens on the device differ from the plan */
#define MLA_DEVICE_BAD_PAGE 0x4         /* a page id outside [0, num_pages) */

#define MLA_HEAD_DIM_QK 576
#define MLA_HEAD_DIM_V 512
#define MLA_PAGE_SIZE 64
#define MLA_MAX_HEADS 128

/* Test and tuning knobs of the planner (all 0 = automatic). */
typedef struct {
  int force_splits;        /* > 0: split every row tile's KV range into this many page-aligned parts */
  int max_rows_per_cta;    /* > 0: cap on packed rows per CTA tile (multiple of 16, <= the kernel's cap) */
  int min_pages_per_split; /* > 0: lower bound on pages per split unit */
  int force_fold;          /* > 0: use this fold factor F instead of the largest divisor rule
                              (must divide every q_len; F = 1 is the fold-less diagnostic mode) */
  int unit_pages;          /* > 0: cut every fold group's key range into pieces of this many pages
                              (the last one shorter) instead of the length the planner picks */
  int cta_pair;            /* > 0: with a bf16 cache whose fold groups all have 49..96 rows,
                              run each group on a cluster of two CTAs that split the page
                              columns (0: <= 48-row single-CTA tiles) */
  int pair_slots;          /* > 0: clusters of two CTAs the device runs at once (the planner's
                              dispatch model); 0: num_sms / 2 */
  int debug_skip_copy;     /* test of the device timeout path only, 0 in production: > 0 makes
                              the first work unit skip the copy of its page number
                              debug_skip_copy - 1 and shortens every bounded wait of the call to
                              ~2 ms, so the units that wait for that page report
                              MLA_DEVICE_WAIT_TIMEOUT and stop (no fault, no hang) */
} mla_plan_options;

/*
 * mla_decode_plan -- host-only split-KV work partition (flashinfer PR #5588,
 * "What was measured" table, "host plan" row: the plan is built from host-known
 * scalars only). Folds each request's tokens into groups of F tokens
 * (largest divisor of q with H*F <= 128), cuts each group's packed rows into CTA
 * row tiles, and cuts each row tile's key range [0, seq_len) into page-aligned
 * splits so that the units fill the num_sms SMs.
 *
 *   seq_lens_h, q_lens_h : host int32 [batch]
 *   num_heads            : H, 1..128
 *   page_size            : must be 64
 *   kv_dtype             : MLA_KV_BF16 or MLA_KV_FP8_E4M3
 *   num_sms              : SMs to fill (the device's multiProcessorCount)
 *   plan_buf             : caller-owned host buffer of plan_buf_bytes; may be NULL
 *                          to query the size
 *   plan_bytes_out       : receives the plan size in bytes (always, if non-NULL)
 *   workspace_bytes_out  : receives the device workspace size that mla_decode_run
 *                          needs for this plan (partial O and LSE of split units)
 *
 * Returns MLA_ERR_BUFFER (with the sizes filled in) when plan_buf is NULL or too small.
 * The caller copies the plan bytes to device memory (plan_dev) before mla_decode_run.
 * A changed page table needs no new plan; changed seq_lens or q_lens do.
 */
int mla_decode_plan(const int32_t* seq_lens_h, const int32_t* q_lens_h, int batch, int num_heads,
                    int page_size, int kv_dtype, int num_sms, void* plan_buf, size_t plan_buf_bytes,
                    size_t* plan_bytes_out, size_t* workspace_bytes_out);

/* mla_decode_plan with explicit planner knobs (opts may be NULL). */
int mla_decode_plan_ex(const int32_t* seq_lens_h, const int32_t* q_lens_h, int batch, int num_heads,
                       int page_size, int kv_dtype, int num_sms, const mla_plan_options* opts,
                       void* plan_buf, size_t plan_buf_bytes, size_t* plan_bytes_out,
                       size_t* workspace_bytes_out);

/* Work-unit and merge counts of a plan (host bytes), for launch sizing and tests. */
int mla_decode_plan_info(const void* plan_host, size_t plan_bytes, int* n_units, int* n_merge,
                         int* total_q, int* num_heads, int* kv_dtype);

/*
 * mla_decode_run -- enqueue the verify decode on `stream` (a cudaStream_t; NULL is
 * the legacy default stream). Launches the fused fold kernel (paged TMA loads of
 * the latent cache, Q*K^T and P*V on the tcgen05 tensor cores with TMEM
 * accumulators, online softmax) and, when the plan split any key range, the
 * log-sum-exp merge kernel as a programmatic dependent launch (flashinfer PR
 * #5588 "What was measured", "split rows" row: a separate reduce kernel beat an
 * in-kernel merge).
 *
 *   plan_dev / plan_host : the plan bytes in device and host memory (same contents)
 *   q, kv_cache, page_table, seq_lens, q_lens, out, lse : see the layouts above
 *   page_table_stride    : int32 entries per page_table row (>= pages of the longest request)
 *   num_pages            : pages in kv_cache (page ids must lie in [0, num_pages))
 *   sm_scale             : score scale (1/sqrt(192) for the Kimi-K3 / DeepSeek head sizes)
 *   kv_scale             : per-tensor dequantisation scale of an fp8 cache (ignored for bf16)
 *   workspace            : device scratch of at least the plan's workspace bytes (may be
 *                          NULL when that size is 0)
 *   status_dev           : optional device int32 the kernels OR MLA_DEVICE_* bits into
 *
 * Enqueue only: no allocation, no host synchronisation, no host reads of device
 * memory, so the call can be captured in a CUDA graph (the tensor maps are built on
 * the host and passed by value).
 */
int mla_decode_run(const void* plan_dev, const void* plan_host, size_t plan_bytes, const void* q,
                   const void* kv_cache, const int32_t* page_table, int page_table_stride,
                   int num_pages, const int32_t* seq_lens, const int32_t* q_lens, float sm_scale,
                   float kv_scale, void* out, float* lse, void* workspace, size_t workspace_bytes,
                   int32_t* status_dev, void* stream);

/*
 * mla_decode_run_static_ws -- mla_decode_run without a caller-supplied workspace.
 *
 * The pages have no counterpart for this entry point; it exists for callers that
 * cannot allocate device memory: code running where an allocation would synchronise
 * the device or break a real-time budget, plug-in hosts that hand out only the
 * input and output buffers and own every allocator, and runtimes with a fixed memory
 * plan. The split-KV partials go to a library-owned device array of
 * MLA_STATIC_WORKSPACE_BYTES (16 MiB), which every GPU that loads the library holds
 * until the process exits. The call itself allocates nothing (no cudaMalloc,
 * cudaFree or allocating library routine).
 *
 *   Arguments are those of mla_decode_run without workspace / workspace_bytes.
 *   A plan whose workspace exceeds the array (mla_decode_plan reports the size) is
 *   rejected with MLA_ERR_BUFFER before any launch; plan with fewer splits
 *   (mla_plan_options.force_splits) or use mla_decode_run with your own workspace.
 *   The first call on a device looks up the array's device address (with that device
 *   current) and caches it with the current context; make that first call before any
 *   stream capture. After a device reset the next call looks it up again.
 *   Every call in the process shares the one array per device and overwrites what the
 *   previous call left in it; nothing in it needs clearing. Calls whose kernels
 *   overlap on the GPU (for example on two concurrent streams) race on the array, so
 *   serialise them.
 */
#define MLA_STATIC_WORKSPACE_BYTES (16u << 20)
int mla_decode_run_static_ws(const void* plan_dev, const void* plan_host, size_t plan_bytes, const void* q,
                             const void* kv_cache, const int32_t* page_table, int page_table_stride, int num_pages,
                             const int32_t* seq_lens, const int32_t* q_lens, float sm_scale, float kv_scale, void* out,
                             float* lse, int32_t* status_dev, void* stream);

/*
 * mla_device_pair_slots -- how many clusters of two CTAs of the two-CTA decode kernel the
 * device runs at once (cudaOccupancyMaxActiveClusters). A plan for fold groups of 49..96
 * rows with a bf16 cache runs on such clusters; pass this number as
 * mla_plan_options.pair_slots so that the planner's dispatch model matches the device
 * (a GPC with an odd number of free SMs leaves one SM out). Sets the current device to
 * `device` for the query and restores it.
 */
int mla_device_pair_slots(int device, int* slots);

/* Message of the last failed call on this thread ("" if none). */
const char* mla_last_error(void);

/* Library version, e.g. 100 for 0.1.0. */
int mla_version(void);

#ifdef __cplusplus
}
#endif

#endif /* MLA_DECODE_H_ */

/*
 * pagedattn -- batched ragged attention over a paged KV cache, for one
 * GB300 GPU (sm_103a).  Plain C ABI: plain pointers and sizes, no C++ or
 * framework types cross it.
 *
 * The problem statement follows the FlashInfer issue "How are prefill and
 * decode kernels different?" (the timing script and its
 * BatchDecodeWithPagedKVCacheWrapper / BatchPrefillWithPagedKVCacheWrapper
 * calls): a batch of requests, request b owning
 *
 *   - qo_len_b query rows packed in q[T, Hq, D] between qo_indptr[b] and
 *     qo_indptr[b+1] (prefill chunks have qo_len > 1, decodes qo_len = 1);
 *   - kv_len_b keys/values stored in the pages kv_page_indices[
 *     kv_page_indptr[b] .. kv_page_indptr[b+1]) of the cache
 *     kv_cache[num_pages, 2, page_size, Hkv, D] ("NHD": index 0 of the
 *     second dimension holds K, index 1 holds V); every page is full except
 *     the last, which holds kv_last_page_len[b] slots, 1 <= last <= page_size.
 *     kv_len_b = (pages_b - 1) * page_size + last_b.
 *
 * Query head h reads kv head h / (Hq / Hkv) (grouped-query attention).  Query
 * row i of request b sits at absolute position kv_len_b - qo_len_b + i and,
 * with causal = 1, sees keys [0, kv_len_b - qo_len_b + i] (the mask aligned
 * to the bottom-right, so new tokens appended after a shared prefix -- the
 * vLLM issue "Question about efficient memory sharing (prefix sharing)" --
 * see the whole prefix, and fully masked tails are never visited, as the
 * llama.cpp discussion "Pad for prefill stage?" describes).  With scale =
 * 1/sqrt(D):
 *
 *   out[row, h, :] = sum_t softmax_t(scale * q[row,h,:] . K[t,:]) * V[t,:]
 *   lse[row, h]    = ln sum_t exp(scale * q[row,h,:] . K[t,:])   (natural log)
 *
 * Several page tables may list the same physical page (prefix sharing): the
 * library only reads the cache.
 *
 * Life cycle (the script's begin_forward / forward / end_forward):
 *   pagedattn_plan()          once per batch: host work, one H2D copy
 *   pagedattn_run()           any number of times, asynchronous, no alloc
 *   pagedattn_plan_destroy()  when the batch is done
 *
 * Errors: every call returns a pagedattn_status; the text of the last error
 * on the calling thread is pagedattn_last_error().  No call aborts, prints or
 * throws.
 */
#ifndef PAGEDATTN_H_
#define PAGEDATTN_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define PAGEDATTN_API __attribute__((visibility("default")))
#else
#define PAGEDATTN_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* CUDA stream handle, identical to cudaStream_t (a CUstream_st pointer). */
typedef struct CUstream_st* pagedattn_stream_t;

typedef struct pagedattn_plan_s* pagedattn_plan_t; /* opaque, owned by the library */

typedef enum {
  PA_OK = 0,
  PA_ERR_INVALID_ARG = 1,         /* malformed indptr / page ids / lengths / pointers  */
  PA_ERR_UNSUPPORTED = 2,         /* head_dim, page_size, dtype or group size not built */
  PA_ERR_WORKSPACE_TOO_SMALL = 3, /* workspace_bytes < pagedattn_workspace_size()       */
  PA_ERR_CUDA = 4,                /* a CUDA runtime call failed (message has the code)  */
  PA_ERR_DEVICE_CHECK = 5,        /* an in-kernel check fired (see device_status)       */
  PA_ERR_TIMEOUT = 6              /* an in-kernel wait gave up after its bound          */
} pagedattn_status;

typedef enum { PA_FP16 = 0, PA_BF16 = 1 } pagedattn_dtype;

/* Optional planner settings; pass NULL for the defaults (all zero). */
typedef struct {
  int32_t num_sms;             /* SMs to plan for; 0 = ask the current device        */
  int32_t force_prefill;       /* 1: every request uses the tcgen05 prefill kernel    */
  int32_t decode_chunk_pages;  /* > 0: pages per decode split (default: see plan)    */
  int32_t prefill_chunk_tiles; /* > 0: 128-key tiles per prefill split               */
  int32_t force_cp_async;      /* 1: stage K/V with cp.async instead of TMA           */
  int32_t decode_cuda_cores;   /* 1: single-token requests at group sizes <= 8 run on
                                  the CUDA-core decode kernel, and multi-token
                                  requests all go to the prefill kernel (default:
                                  the warp-MMA small-query kernel, see plan)        */
  int32_t kv_layout;           /* PA_LAYOUT_NHD (default) or PA_LAYOUT_HND: see below */
  int32_t prefill_q_tiles;     /* 128-row query tiles per prefill work item: 1 or 2;
                                  0 = the planner's choice (see plan).  head_dim 256
                                  takes 1 only                                      */
  int32_t wait_limit_cycles;   /* test hook: > 0 bounds every in-kernel pipeline wait
                                  at that many SM clock cycles instead of about 2 s,
                                  and makes one thread of every CTA first wait on a
                                  barrier that nothing completes, so the waits give
                                  up (the run then reports PA_DEV_TIMEOUT through
                                  device_status and leaves out / lse undefined);
                                  0 = the default                                   */
  int32_t reserved[1];         /* must be 0                                          */
} pagedattn_options;

/*
 * Cache layouts (pagedattn_options.kv_layout).  Both hold, per physical page,
 * the page_size K rows and then the page_size V rows of every kv head; the
 * FlashInfer timing script passes "NHD" and the alternative it implies keeps
 * each head's rows together:
 *   PA_LAYOUT_NHD  kv_cache[num_pages][2][page_size][num_kv_heads][head_dim]
 *   PA_LAYOUT_HND  kv_cache[num_pages][2][num_kv_heads][page_size][head_dim]
 * The results are identical (bit for bit) for the same logical cache.
 */
#define PA_LAYOUT_NHD 0
#define PA_LAYOUT_HND 1

/* Stage bits for pagedattn_run_stages. */
#define PA_STAGE_PREFILL 1u
#define PA_STAGE_DECODE 2u
#define PA_STAGE_MERGE 4u
#define PA_STAGE_ALL 7u

/* Status bits the kernels OR into the device status word. */
#define PA_DEV_TIMEOUT 1
#define PA_DEV_BAD_INDEX 2

/*
 * Build the work partition for one batch ("auxiliary data structures" that
 * begin_forward builds, in the timing script).
 *
 * qo_indptr        host, int32[batch_size + 1], [0] == 0, nondecreasing.
 * kv_page_indptr   host, int32[batch_size + 1], [0] == 0, nondecreasing.
 * kv_page_indices  host, int32[kv_page_indptr[batch_size]], each in [0, num_pages).
 * kv_last_page_len host, int32[batch_size], in [1, page_size] for every request
 *                  that has pages.
 * num_qo_heads, num_kv_heads: num_qo_heads a positive multiple of num_kv_heads;
 *                  the group size num_qo_heads / num_kv_heads must divide 128.
 * head_dim         64, 128 or 256 (at 256 decode runs on the CUDA-core kernel
 *                  for single-token requests at group size <= 8, everything
 *                  else on the tensor-core prefill kernel).  page_size: a
 *                  power of two in [1, 128].
 * causal           1: bottom-right causal mask (qo_len <= kv_len required);
 *                  0: every row sees all kv_len keys.
 * workspace        caller-owned device buffer (the wrapper's workspace in the
 *                  script); the plan writes its metadata (work items, page ids,
 *                  merge map) to its start with one cudaMemcpyAsync on `stream`
 *                  and keeps fp32 split-KV partial states after it.  The copy's
 *                  source is pageable host memory, so the call may hold the
 *                  host until `stream` reaches it: a serving loop that plans
 *                  the next step while the current one runs passes a stream
 *                  that is not queued behind the running kernels (its upload
 *                  stream).  It must stay
 *                  allocated and untouched while the plan is used.  NULL builds a
 *                  host-only plan (metadata inspection; run() then fails).
 * workspace_bytes  its size; PA_ERR_WORKSPACE_TOO_SMALL below the size
 *                  pagedattn_workspace_size() reports.
 * opts             NULL or settings (see pagedattn_options).
 * out_plan         receives the handle; destroy it with pagedattn_plan_destroy.
 *
 * Host arrays are read during the call only; the library keeps its own copy.
 * The call is synchronous on the host and asynchronous on the device (the
 * metadata copy is queued on `stream`).
 */
PAGEDATTN_API pagedattn_status pagedattn_plan(const int32_t* qo_indptr, const int32_t* kv_page_indptr,
                                const int32_t* kv_page_indices, const int32_t* kv_last_page_len,
                                int32_t batch_size, int32_t num_qo_heads, int32_t num_kv_heads,
                                int32_t head_dim, int32_t page_size, int32_t num_pages,
                                pagedattn_dtype dtype, int32_t causal, void* workspace,
                                size_t workspace_bytes, const pagedattn_options* opts,
                                pagedattn_stream_t stream, pagedattn_plan_t* out_plan);

/*
 * Bytes of workspace the same arguments need (metadata + partial states).
 * Pure host computation; writes *bytes.
 */
PAGEDATTN_API pagedattn_status pagedattn_workspace_size(const int32_t* qo_indptr, const int32_t* kv_page_indptr,
                                          const int32_t* kv_page_indices,
                                          const int32_t* kv_last_page_len, int32_t batch_size,
                                          int32_t num_qo_heads, int32_t num_kv_heads,
                                          int32_t head_dim, int32_t page_size, int32_t num_pages,
                                          pagedattn_dtype dtype, int32_t causal,
                                          const pagedattn_options* opts, size_t* bytes);

/*
 * Shared-prefix cascade (the vLLM issue "Question about efficient memory
 * sharing (prefix sharing)": requests that start from one system prompt
 * should share its attention work, not only its pages).
 *
 * The requests of group g -- consecutive in the batch: requests
 * [group_indptr[g], group_indptr[g+1]) -- all begin with the same prefix
 * of full pages prefix_page_indices[prefix_page_indptr[g] ..
 * prefix_page_indptr[g+1]), followed by their own pages as described by
 * kv_page_indptr / kv_page_indices / kv_last_page_len (which then count only
 * the keys after the prefix).  Request b of the group attends to
 * prefix_len_g + kv_len_b keys: exactly what pagedattn_plan computes for the
 * flattened page table (prefix pages, then the request's own), with the
 * bottom-right causal mask over the whole sequence.  Its query rows must lie
 * after the prefix (qo_len_b <= kv_len_b, the usual check on the request's
 * own keys), so each of them sees the whole prefix.
 *
 * The plan computes the prefix attention once for all query tokens of the
 * group (they are consecutive in q) as one unmasked prefill, the rest per
 * request, and merges the two with the split-KV merge; results agree with
 * the flattened plan within the usual tolerance (sums in another order).
 * A group with no prefix pages is planned like ordinary requests.
 */
typedef struct {
  const int32_t* group_indptr;        /* host, [num_groups + 1], [0] == 0, nondecreasing,
                                         [num_groups] == batch_size                       */
  const int32_t* prefix_page_indptr;  /* host, [num_groups + 1], [0] == 0, nondecreasing    */
  const int32_t* prefix_page_indices; /* host, the groups' full prefix pages, each in
                                         [0, num_pages)                                    */
  int32_t num_groups;                 /* >= 0; 0 plans like pagedattn_plan                 */
} pagedattn_prefix_groups;

/* pagedattn_plan with shared-prefix groups (NULL groups: pagedattn_plan). */
PAGEDATTN_API pagedattn_status pagedattn_plan_cascade(const pagedattn_prefix_groups* groups,
                                        const int32_t* qo_indptr, const int32_t* kv_page_indptr,
                                        const int32_t* kv_page_indices, const int32_t* kv_last_page_len,
                                        int32_t batch_size, int32_t num_qo_heads, int32_t num_kv_heads,
                                        int32_t head_dim, int32_t page_size, int32_t num_pages,
                                        pagedattn_dtype dtype, int32_t causal, void* workspace,
                                        size_t workspace_bytes, const pagedattn_options* opts,
                                        pagedattn_stream_t stream, pagedattn_plan_t* out_plan);

/* pagedattn_workspace_size for pagedattn_plan_cascade. */
PAGEDATTN_API pagedattn_status pagedattn_workspace_size_cascade(const pagedattn_prefix_groups* groups,
                                          const int32_t* qo_indptr, const int32_t* kv_page_indptr,
                                          const int32_t* kv_page_indices,
                                          const int32_t* kv_last_page_len, int32_t batch_size,
                                          int32_t num_qo_heads, int32_t num_kv_heads,
                                          int32_t head_dim, int32_t page_size, int32_t num_pages,
                                          pagedattn_dtype dtype, int32_t causal,
                                          const pagedattn_options* opts, size_t* bytes);

/*
 * Attention for the planned batch (the script's forward(q, kv_cache)).
 *
 * q        device, dtype[T, Hq, D] contiguous, 16-byte aligned (T = qo_indptr[B]).
 * kv_cache device, dtype[num_pages, 2, page_size, Hkv, D] contiguous, 16-byte aligned.
 * out      device, dtype[T, Hq, D], caller-allocated; every row of a request
 *          with qo_len >= 1 is written.
 * lse      device, float[T, Hq] natural-log sums, or NULL to skip.
 * stream   the stream every kernel is queued on.
 *
 * Launches the prefill kernel (tcgen05 / TMEM), the small-query kernels
 * (decode and requests of qo_len * G <= 32 rows: warp-level MMA, one launch
 * per row class, or the CUDA-core decode kernel) and, when some request was
 * split, the merge kernel, in that order on `stream`.  Allocates nothing and does not synchronise the host.
 * The kernels are launched with programmatic stream serialization: each may
 * begin its set-up while the kernel before it on `stream` finishes, and
 * waits for that kernel's completion before it reads q, kv_cache or partial
 * states or writes anything, so stream order holds for every buffer.  In-kernel
 * waits are bounded; a wait that gives up sets PA_DEV_TIMEOUT in the device
 * status word (read it with pagedattn_device_status).  Calls that overlap on
 * the device must use different workspaces (the partial states live there),
 * so two such calls need two plans.  Host threads may call run on one plan
 * at once: the plan's host-side state (its cache of TMA descriptors) is
 * locked; kernel launch settings are applied per device.
 */
PAGEDATTN_API pagedattn_status pagedattn_run(pagedattn_plan_t plan, const void* q, const void* kv_cache,
                               void* out, float* lse, pagedattn_stream_t stream);

/*
 * Same as pagedattn_run restricted to the stages in `stage_mask`
 * (PA_STAGE_* bits).  Running PREFILL, DECODE and MERGE in that order is
 * exactly pagedattn_run; used to time the kernels one by one.
 */
PAGEDATTN_API pagedattn_status pagedattn_run_stages(pagedattn_plan_t plan, const void* q, const void* kv_cache,
                                      void* out, float* lse, pagedattn_stream_t stream,
                                      uint32_t stage_mask);

/* Release a plan (end_forward in the script).  NULL is a no-op. */
PAGEDATTN_API pagedattn_status pagedattn_plan_destroy(pagedattn_plan_t plan);

/* Thread-local text of the last error ("" when none).  Never NULL. */
PAGEDATTN_API const char* pagedattn_last_error(void);

/*
 * Wait for `stream`, read the device status word of the plan's workspace
 * (PA_DEV_* bits OR-ed by the kernels since the plan or the last read) into
 * *flags and clear it.  Returns PA_ERR_TIMEOUT / PA_ERR_DEVICE_CHECK when a
 * bit is set, PA_OK otherwise.
 */
PAGEDATTN_API pagedattn_status pagedattn_device_status(pagedattn_plan_t plan, pagedattn_stream_t stream,
                                         int32_t* flags);

/*
 * Copy the plan metadata (exactly the bytes copied to the workspace) into
 * host_buf.  With host_buf NULL, only writes the size to *bytes; otherwise
 * *bytes is the buffer size on input and the bytes written on output.
 * Layout: int32 words, documented with the planner rules in the source.
 */
PAGEDATTN_API pagedattn_status pagedattn_debug_plan_dump(pagedattn_plan_t plan, void* host_buf, size_t* bytes);

/*
 * Test hook for the page-table walk: a kernel that resolves every logical
 * token t < kv_len_b of every request b (in request order) with the same
 * device index code the attention kernels use, writing the physical page id
 * and slot to page_out / slot_out (device, int32[sum_b kv_len_b]).
 * Asynchronous on `stream`.
 */
PAGEDATTN_API pagedattn_status pagedattn_debug_gather(pagedattn_plan_t plan, int32_t* page_out,
                                        int32_t* slot_out, pagedattn_stream_t stream);

/*
 * Decode without a device workspace.  The source pages have no counterpart
 * to this call; it exists for callers that cannot allocate device memory --
 * serving processes that reserve all free GPU memory for their KV cache up
 * front, and latency-critical code that must not call cudaFree (which
 * synchronises the device).
 *
 * Runs the decode kernel and the split merge of `plan` (build it with
 * pagedattn_plan and workspace = NULL) with the plan's metadata and split-KV
 * partial states in a fixed 16 MiB device array inside the library instead
 * of a caller workspace.  The array exists once per GPU that loads the
 * library and stays allocated until the process exits.  q, kv_cache, out and
 * lse are as for pagedattn_run.
 *
 * The batch must have no prefill items (every request has qo_len 0 or
 * qo_len * G <= 32 with the group size G = num_qo_heads / num_kv_heads in
 * {1, 2, 4, 8, 16}, and force_prefill is off; with decode_cuda_cores or at
 * head_dim 256, qo_len <= 1 and G <= 8): PA_ERR_UNSUPPORTED otherwise.  A plan whose metadata and partial
 * states exceed 16 MiB returns PA_ERR_WORKSPACE_TOO_SMALL (plan with a larger
 * decode_chunk_pages).  The call allocates no memory.  Its first call on a
 * device looks up the array's device address (cudaGetSymbolAddress) while
 * that device is current; make that first call before any stream capture.
 * Every call overwrites the array, whose contents are whatever the last call
 * left (the plan's metadata copy clears the in-kernel status word): calls
 * that overlap on the GPU -- on different streams or from different host
 * threads -- race and must not be issued.  The in-kernel status word of the
 * last call is read with pagedattn_noalloc_device_status.
 */
PAGEDATTN_API pagedattn_status pagedattn_run_decode_noalloc(pagedattn_plan_t plan, const void* q,
                                                            const void* kv_cache, void* out, float* lse,
                                                            pagedattn_stream_t stream);

/*
 * The device status word (PA_DEV_* bits) that the kernels of the last
 * pagedattn_run_decode_noalloc call on the current device left in the
 * library's no-alloc array: waits for `stream` (pass the stream of that
 * call), copies the word into *flags and returns PA_ERR_TIMEOUT /
 * PA_ERR_DEVICE_CHECK when a bit is set, PA_OK otherwise.  Allocates
 * nothing; the next no-alloc call clears the word.
 */
PAGEDATTN_API pagedattn_status pagedattn_noalloc_device_status(pagedattn_stream_t stream, int32_t* flags);

/* Library version as "major.minor.patch". */
PAGEDATTN_API const char* pagedattn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* PAGEDATTN_H_ */

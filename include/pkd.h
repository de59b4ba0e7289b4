/*
 * pkd.h - paged KV decode attention with split-KV partial states and the
 * log-sum-exp merge, for NVIDIA GB300 (sm_103a).
 *
 * A C ABI: plain pointers and sizes, no C++ or framework types.  Every call
 * returns a pkd_status; pkd_last_error() gives a message for the calling
 * thread's last failure.  No call throws, aborts or allocates device memory:
 * the caller owns every buffer (tensors, page tables, workspaces, pinned
 * staging memory and the pkd_plan_t itself).
 *
 * Sources (page title, section):
 *  [W] "FlashInfer" (aiwiki.ai/wiki/flashinfer)
 *  [D] "Welcome to FlashInfer's documentation!" (docs.flashinfer.ai)
 *
 * Shapes and layouts (B requests, Hq query heads, Hkv key/value heads,
 * g = Hq / Hkv, D = head_dim, P = page_size):
 *  q          [B][Hq][D]                      dtype
 *  k_pages    [num_pages][P][Hkv][D]          dtype  (NHD, [D] tutorial
 *  v_pages    [num_pages][P][Hkv][D]          dtype   "KV-Cache Layout"), or
 *             [num_pages][Hkv][P][D] with problem.kv_layout = PKD_LAYOUT_HND
 *  kv_indptr  [B + 1] int32, kv_indices [kv_indptr[B]] int32,
 *  kv_last_page_len [B] int32: CSR page table ([D] "Page Table Layout";
 *    [W] "Block-sparse cache representation").  Request b owns pages
 *    kv_indices[kv_indptr[b] .. kv_indptr[b+1]) in sequence order; all are
 *    full except the last, which holds kv_last_page_len[b] in [1, P] tokens.
 *    A request with no pages is empty.  Page ids lie in [0, num_pages);
 *    several requests may list the same page (shared prefixes).
 *  out        [B][Hq][D] dtype;  lse [B][Hq] float (natural log).
 *  Query head h attends with key/value head h / g ([W] "Custom attention
 *  templates": grouped-query heads).
 *
 * Semantics: out[b,h] = sum_t softmax_t(s) v_t and lse[b,h] = log sum_t
 * exp(s_t) with s_t = sm_scale * <q[b,h], k_t>, over the request's tokens.
 * The running maximum starts at -infinity and an empty request yields
 * out = 0, lse = -infinity ([W] "Extreme-negative-logit correction").
 *
 * Supported: dtype PKD_F16 or PKD_BF16; head_dim 128; Hkv in {1, 2, 4, 8};
 * 1 <= g <= 16; page_size >= 1; 16-byte aligned device pointers.  Anything
 * else returns PKD_ERR_UNSUPPORTED; there is no fallback path.
 */
#ifndef PKD_H
#define PKD_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define PKD_ABI_VERSION 5

typedef enum {
  PKD_OK = 0,
  PKD_ERR_INVALID_ARG = -1,  /* null pointer, negative size, bad enum */
  PKD_ERR_PAGE_TABLE = -2,   /* page table fails the CSR rules above */
  PKD_ERR_WORKSPACE = -3,    /* a workspace or staging buffer is too small */
  PKD_ERR_UNSUPPORTED = -4,  /* valid but outside the supported set */
  PKD_ERR_CUDA = -5,         /* a CUDA runtime call or launch failed */
  PKD_ERR_DEVICE_CHECK = -6  /* a kernel recorded a failed check */
} pkd_status;

typedef enum { PKD_F16 = 0, PKD_BF16 = 1, PKD_F32 = 2 } pkd_dtype;

/* Page tensor layouts ([D] "KV-Cache Layout in FlashInfer", "Layout: NHD/HND"). */
typedef enum {
  PKD_LAYOUT_NHD = 0,  /* [num_pages][page_size][num_kv_heads][head_dim] */
  PKD_LAYOUT_HND = 1   /* [num_pages][num_kv_heads][page_size][head_dim] */
} pkd_layout;

/* How the decode kernel moves K/V pages into shared memory. */
typedef enum {
  PKD_LOADER_AUTO = 0,       /* the library's choice: TMA tiles for HND pages when
                                page_size % 16 == 0 and for NHD pages of exactly 16
                                tokens, else bulk rows */
  PKD_LOADER_TMA_TILES = 1,  /* TMA tiled loads, one box per (tensor, d-half) covering
                                16 slots of every head (page_size % 16 == 0) */
  PKD_LOADER_BULK_ROWS = 2   /* one bulk copy per token row of all heads (NHD) or per
                                (token, head) row (HND); any page_size */
} pkd_loader;

/* Bits of the device status word (see pkd_check_status). */
#define PKD_DEVICE_BAD_PAGE 1u    /* a page id outside [0, num_pages) */
#define PKD_DEVICE_BAD_LENGTH 2u  /* a plan unit runs past the request */
#define PKD_DEVICE_BAD_PLAN 4u    /* workspace does not hold a plan image for this
                                     launch, or one of its units is malformed (a
                                     request or slot out of range, a start off a
                                     16-token tile boundary) */
#define PKD_DEVICE_TIMEOUT 8u     /* a bounded pipeline wait ran out */
/* Test hook: with the environment variable PKD_TEST_INJECT set to "no-loader"
 * or "no-consumers" when a decode kernel is launched, that role of every CTA
 * is left out and, after about 100 us, the CTA's abort flag is raised, so the
 * other role's waits give up and record PKD_DEVICE_TIMEOUT (a host-side
 * failure injection for tests of the timeout path; the results of such a
 * launch are meaningless).  Unset in normal use. */

/* Problem geometry and planning knobs. */
typedef struct {
  int32_t batch;         /* B >= 0 */
  int32_t num_qo_heads;  /* Hq */
  int32_t num_kv_heads;  /* Hkv, Hq % Hkv == 0 */
  int32_t head_dim;      /* D (128) */
  int32_t page_size;     /* P >= 1 */
  int32_t dtype;         /* pkd_dtype of q, k_pages, v_pages and out */
  int64_t num_pages;     /* pages in the pool; bounds every page id */
  int32_t num_ctas;      /* decode CTAs (one per SM is the intent); 0 = the
                            current device's multiprocessor count */
  int32_t min_chunks_per_request; /* each request of n tiles is cut into at
                            least min(this, n) partial states; 0 or 1 = no
                            minimum */
  int32_t tile_tokens;   /* tokens per pipeline tile; 0 = 16 (the decode
                            kernel's tile); other values are unsupported */
  int32_t max_batch;     /* capacity used to size workspaces; 0 = batch */
  int32_t kv_loader;     /* pkd_loader */
  int32_t kv_layout;     /* pkd_layout of k_pages and v_pages */
} pkd_problem;

/* Result of planning: plain data, owned and stored by the caller. */
typedef struct {
  pkd_problem problem;          /* resolved copy (num_ctas, tile_tokens set) */
  int32_t num_units;            /* work units in the plan */
  int32_t num_partials;         /* partial-state slots used */
  int32_t num_split_requests;   /* requests merged from >1 partial state */
  int32_t total_tiles;          /* sum over requests of ceil(L_b / tile) */
  int64_t total_tokens;         /* sum over requests of L_b */
  int64_t int_ws_bytes_used;    /* bytes of the plan image */
  int64_t float_ws_bytes_needed;/* bytes of partial states run() writes */
  int32_t valid;                /* 1 once planned */
  int32_t reserved;
} pkd_plan_t;

/* ABI version of the loaded library (PKD_ABI_VERSION). */
int32_t pkd_abi_version(void);

/* Message for the calling thread's last failed call ("" if none). */
const char *pkd_last_error(void);

/*
 * Workspace sizes for a problem's capacity (max_batch, num_ctas,
 * min_chunks_per_request), valid for every plan of that capacity:
 *   int_ws_bytes   device buffer holding the plan image (int32 words);
 *   float_ws_bytes device buffer for fp32 partial states: a slot per work
 *                  unit the capacity allows plus one per request (the
 *                  states-only decode of pkd_run_decode_states and the
 *                  cascade keep every request's state in fp32);
 *   staging_bytes  pinned host buffer pkd_plan() builds the image in.
 * num_ctas == 0 queries the current device.  Any output pointer may be NULL.
 */
pkd_status pkd_workspace_size(const pkd_problem *problem,
                              size_t *int_ws_bytes, size_t *float_ws_bytes,
                              size_t *staging_bytes);

/*
 * Plans on the host only (no CUDA call): validates the page table, computes
 * request lengths and the split-KV work list ([W] "Plan and run": planning
 * reads sequence lengths and cache metadata, selects a schedule and prepares
 * workspace data; "Attention states": a long cache is split across work units
 * whose partial states are merged) and writes the plan image (int32 words)
 * to host_image.  problem->num_ctas must be explicit (> 0).
 * kv_indices_h may be NULL; if given, every page id is range-checked.
 * Errors: PKD_ERR_INVALID_ARG, PKD_ERR_PAGE_TABLE, PKD_ERR_UNSUPPORTED,
 * PKD_ERR_WORKSPACE (image larger than host_image_bytes).
 */
pkd_status pkd_plan_host(const pkd_problem *problem, const int32_t *kv_indptr_h,
                         const int32_t *kv_last_page_len_h,
                         const int32_t *kv_indices_h, pkd_plan_t *plan,
                         int32_t *host_image, size_t host_image_bytes);

/*
 * pkd_plan_host into pinned_staging, then one asynchronous host-to-device
 * copy of the image into int_ws_dev on `stream` (a cudaStream_t; NULL = the
 * legacy default stream).  The staging buffer must stay untouched until that
 * copy has run.  Reusing int_ws_dev keeps device addresses stable across
 * plans ([W] "Plan and run": stable workspace buffers, updated schedule data).
 */
pkd_status pkd_plan(const pkd_problem *problem, const int32_t *kv_indptr_h,
                    const int32_t *kv_last_page_len_h,
                    const int32_t *kv_indices_h, pkd_plan_t *plan,
                    int32_t *pinned_staging, size_t staging_bytes,
                    void *int_ws_dev, size_t int_ws_bytes, void *stream);

/*
 * Copies a plan image (of pkd_plan_host or pkd_plan_shared_prefix_host) from
 * pinned host memory into int_ws_dev on `stream`, with one small kernel that
 * reads the host buffer directly (no copy-engine transfer): in a CUDA graph
 * it chains onto the decode kernel without an engine hand-off ([W] "Plan and
 * run": a captured run keeps its device addresses while the scheduling data
 * in them is updated).  The number of words copied is read from the image's
 * header when the kernel runs, so a captured copy follows whatever plan the
 * host last wrote into the same buffer; the host must not rewrite the buffer
 * until the stream has passed the copy.  pinned_image must be page-locked
 * host memory (cudaHostAlloc / cudaHostRegister), both pointers 16-byte
 * aligned, and both sizes at least a 64-byte header (else
 * PKD_ERR_INVALID_ARG / PKD_ERR_UNSUPPORTED / PKD_ERR_WORKSPACE, nothing
 * launched).  An image that is not a plan, or whose header describes more
 * words than pinned_image_bytes or int_ws_bytes hold, is not copied beyond
 * its header, and PKD_DEVICE_BAD_PLAN is set in the device copy's status
 * word (every kernel then rejects it).
 */
pkd_status pkd_copy_plan(const int32_t *pinned_image, size_t pinned_image_bytes,
                         void *int_ws_dev, size_t int_ws_bytes, void *stream);

/*
 * Decode attention for a planned batch, on `stream`: the decode kernel walks
 * the work list, writing out/lse directly for requests handled by one unit
 * and fp32 partial (output, lse) states to float_ws_dev otherwise; then, if
 * any request was split, the merge kernel combines each split request's
 * partial states ([W] "Attention states").  Device pointers: q, k_pages,
 * v_pages, the page table (the same table the plan saw), int_ws_dev (holding
 * the plan image), float_ws_dev (>= plan->float_ws_bytes_needed), out, lse.
 * Kernels range-check page ids and plan units against the device page table
 * and record failures in the device status word instead of reading out of
 * bounds.  Returns PKD_ERR_UNSUPPORTED / PKD_ERR_INVALID_ARG /
 * PKD_ERR_WORKSPACE before launching, PKD_ERR_CUDA if a launch fails.
 */
pkd_status pkd_run(const pkd_plan_t *plan, const void *q, const void *k_pages,
                   const void *v_pages, const int32_t *kv_indptr_d,
                   const int32_t *kv_indices_d,
                   const int32_t *kv_last_page_len_d, void *int_ws_dev,
                   void *float_ws_dev, size_t float_ws_bytes, float sm_scale,
                   void *out, float *lse, void *stream);

/*
 * CUDA graphs ([W] "Plan and run": stable workspace addresses, updated
 * scheduling data for a captured run).  pkd_run, pkd_run_decode and
 * pkd_run_merge may be captured on a stream.  While capturing, the merge
 * kernel is launched even if the plan split nothing, and both launches are
 * sized for the problem's capacity (max_batch, the float workspace's size),
 * because they read the plan image at run time: a replay computes whatever
 * plan pkd_plan last copied into the same int_ws_dev (same problem apart from
 * batch <= max_batch), with q / out / lse and the page-table buffers at the
 * captured addresses sized for max_batch and int_ws_dev of pkd_workspace_size.
 */

/*
 * The two launches of pkd_run, for callers that put other work or events
 * between them: pkd_run_decode launches the decode kernel (same arguments and
 * errors as pkd_run); pkd_run_merge then launches the merge kernel for the
 * plan's split requests, and does nothing when no request was split.  Both
 * must see the same plan, workspaces and out/lse on streams ordered the same
 * way as in pkd_run.
 */
pkd_status pkd_run_decode(const pkd_plan_t *plan, const void *q,
                          const void *k_pages, const void *v_pages,
                          const int32_t *kv_indptr_d, const int32_t *kv_indices_d,
                          const int32_t *kv_last_page_len_d, void *int_ws_dev,
                          void *float_ws_dev, size_t float_ws_bytes,
                          float sm_scale, void *out, float *lse, void *stream);

pkd_status pkd_run_merge(const pkd_plan_t *plan, const void *int_ws_dev,
                         const void *float_ws_dev, size_t float_ws_bytes,
                         void *out, float *lse, void *stream);

/*
 * The decode kernel in its states-only mode ([W] "Attention states"): every
 * request's attention state stays fp32 in float_ws_dev and nothing is written
 * to an out / lse in the input type.  A request the plan split leaves its
 * partial states in its plan slots (as pkd_run_decode); an unsplit request b,
 * an empty one included, leaves its state in slot plan->num_partials + b
 * (o [Hq][head_dim] then lse [Hq], padded to 4 floats; (0, -inf) when empty).
 * float_ws_bytes must hold plan->num_partials + batch slots
 * (pkd_workspace_size's float size always does), else PKD_ERR_WORKSPACE.
 * Other arguments, errors and graph capture as pkd_run_decode; a replay whose
 * plan needs more slots than float_ws_bytes holds is skipped with
 * PKD_DEVICE_BAD_PLAN in the status word.  pkd_run_cascade_merge consumes
 * these states.
 */
pkd_status pkd_run_decode_states(const pkd_plan_t *plan, const void *q,
                                 const void *k_pages, const void *v_pages,
                                 const int32_t *kv_indptr_d, const int32_t *kv_indices_d,
                                 const int32_t *kv_last_page_len_d, void *int_ws_dev,
                                 void *float_ws_dev, size_t float_ws_bytes, float sm_scale,
                                 void *stream);

/*
 * Merge of two attention states over disjoint regions into the state of
 * their union ([W] "Attention states"; [D] flashinfer.cascade "Merge
 * Attention States"): with M = max(s_a, s_b),
 *   s = M + log(exp(s_a - M) + exp(s_b - M)),
 *   v = exp(s_a - s) v_a + exp(s_b - s) v_b;
 * a side with s = -infinity contributes nothing and two empty sides give
 * (0, -infinity).  v_* are [n][num_heads][head_dim] of v_dtype (F16, BF16 or
 * F32), s_* are [n][num_heads] float.  In-place use (v_out == v_a, s_out ==
 * s_a) is allowed.  head_dim must be a multiple of 8 and at most 1024.
 */
pkd_status pkd_merge_states(const void *v_a, const float *s_a, const void *v_b,
                            const float *s_b, void *v_out, float *s_out,
                            int64_t n, int32_t num_heads, int32_t head_dim,
                            int32_t v_dtype, void *stream);

/*
 * Reads the device status word of int_ws_dev (synchronising `stream`) into
 * *device_status (PKD_DEVICE_* bits).  Returns PKD_ERR_DEVICE_CHECK if any
 * bit is set, PKD_OK otherwise.  Planning clears the word.
 */
pkd_status pkd_check_status(const void *int_ws_dev, uint32_t *device_status,
                            void *stream);

/*
 * pkd_run with no device allocation at all.  The pages have no counterpart to
 * this call.  It is for callers that cannot allocate device memory when they
 * decode: code whose device memory belongs to another allocator (a serving
 * engine's pool, a plug-in inside a framework that forbids raw cudaMalloc) or
 * a latency-critical loop that cannot pay for cudaMalloc / cudaFree, which may
 * synchronise the device.  The plan image and the fp32 partial states live
 * in a fixed __device__ array inside this library (256 KiB + 8 MiB, held by
 * every GPU that loads the library until the process exits).
 *
 * plan and host_image come from pkd_plan_host; host_image must hold at
 * least plan->int_ws_bytes_used bytes, all of which are copied into the
 * array on `stream` (from pageable memory the call returns once the copy is
 * staged; pinned memory must stay untouched until the stream passes the
 * copy).  The other arguments are those of pkd_run.  A plan whose image
 * exceeds 262144 bytes or whose partial states exceed 8388608 bytes returns
 * PKD_ERR_WORKSPACE before any CUDA call; plan with a smaller
 * min_chunks_per_request or split the batch.  A call on a stream that is
 * being captured returns PKD_ERR_UNSUPPORTED without launching anything.
 * The first call on a device looks up the array's address (with that device
 * current) and keeps it for the life of the process; make that call before
 * any stream capture, and do not call this entry point on a device again
 * after cudaDeviceReset on it.  All calls share the array: calls that
 * overlap on the GPU race.  Kernel range-check failures land in the array's
 * copy of the status word and are not reported.
 */
pkd_status pkd_run_static(const pkd_plan_t *plan, const int32_t *host_image,
                          const void *q, const void *k_pages,
                          const void *v_pages, const int32_t *kv_indptr_d,
                          const int32_t *kv_indices_d,
                          const int32_t *kv_last_page_len_d, float sm_scale,
                          void *out, float *lse, void *stream);

/*
 * Page append: writes new tokens' key and value rows into the paged cache, the
 * step before decode ([D] flashinfer.page "Append new K/V tensors to Paged
 * KV-Cache").  New token i (of num_new) belongs to request
 * batch_indices_d[i] at position positions_d[i] of that request; the page
 * table (kv_indptr_d, kv_indices_d, kv_last_page_len_d, for problem->batch
 * requests) must already cover the requests' new lengths.  k_new / v_new are
 * [num_new][Hkv][D] of problem->dtype; k_pages / v_pages NHD.  A token outside
 * its request's length or on a page id outside [0, num_pages) is skipped and
 * flagged (PKD_DEVICE_BAD_LENGTH / _BAD_PAGE) in *device_status if that
 * device word is given (may be NULL).  Two new tokens mapping to one slot
 * race.
 */
pkd_status pkd_append_kv(const pkd_problem *problem, const void *k_new,
                         const void *v_new, const int32_t *batch_indices_d,
                         const int32_t *positions_d, int64_t num_new, void *k_pages,
                         void *v_pages, const int32_t *kv_indptr_d,
                         const int32_t *kv_indices_d,
                         const int32_t *kv_last_page_len_d, uint32_t *device_status,
                         void *stream);

/*
 * Shared-prefix (cascade) attention ([W] "Attention states": a shared prefix
 * is evaluated separately from request-specific suffixes and the partial
 * states merged; [D] flashinfer.cascade "Cascade Attention").  The queries of
 * `problem->batch` requests attend to one KV prefix they all share, stored
 * once in the page pool as prefix_num_pages pages (all full but the last,
 * which holds prefix_last_page_len tokens).  out / lse are the states over
 * the prefix tokens only; pkd_merge_states with the requests' suffix states
 * (pkd_run on their own pages) gives attention over prefix + suffix.
 * Per key/value head the prefix work is one dense tile (batch x g query rows
 * against the prefix), computed once on the tensor cores, so the prefix is
 * read once per (head, 256-row tile, chunk) instead of once per request.
 * Needs page_size % 16 == 0 (TMA boxes of 16 tokens) and a nonzero
 * problem->num_ctas-derived chunk count; other fields as for pkd_plan.
 * A run captured in a CUDA graph stays valid while the prefix plan (length,
 * chunks, row tiles) is unchanged; the kernel checks the image against its
 * launch and reports a mismatch as PKD_DEVICE_BAD_PLAN.
 */
typedef struct {
  pkd_problem problem;          /* resolved copy (num_ctas set) */
  int32_t prefix_len;           /* tokens of the shared prefix */
  int32_t prefix_num_pages;
  int32_t chunks;               /* KV chunks of the prefix (partial states per row) */
  int32_t chunk_tiles;          /* 64-token tiles per chunk */
  int32_t row_tiles;            /* 256-row tiles per key/value head */
  int32_t num_blocks;           /* CTAs of the prefix kernel */
  int64_t int_ws_bytes_used;    /* bytes of the prefix plan image */
  int64_t float_ws_bytes_needed;/* bytes of fp32 partial states */
  int32_t valid;
  int32_t reserved;
} pkd_prefix_plan_t;

/* Workspace sizes for shared prefixes of up to max_prefix_pages pages. */
pkd_status pkd_prefix_workspace_size(const pkd_problem *problem,
                                     int32_t max_prefix_pages,
                                     size_t *int_ws_bytes, size_t *float_ws_bytes,
                                     size_t *staging_bytes);

/* Plans a shared prefix on the host only (no CUDA call; [W] "Plan and run"):
 * validates the prefix page list (ids in [0, num_pages), 1 <= last_page_len
 * <= page_size), chooses the chunking and writes the prefix plan image
 * (a 16-word header, then the page ids) to host_image.  Chunking: per
 * key/value head the batch x g query rows form row_tiles = ceil(rows / 256)
 * tiles; the prefix, walked in 64-token steps, is cut into as many equal
 * pieces (chunks of chunk_tiles steps) as fit (Hkv x row_tiles) x chunks <=
 * num_ctas, at least one.  problem->num_ctas must be explicit (> 0).
 * Errors: PKD_ERR_INVALID_ARG, PKD_ERR_PAGE_TABLE, PKD_ERR_UNSUPPORTED,
 * PKD_ERR_WORKSPACE (image larger than host_image_bytes). */
pkd_status pkd_plan_shared_prefix_host(const pkd_problem *problem,
                                       const int32_t *prefix_pages_h,
                                       int32_t prefix_num_pages,
                                       int32_t prefix_last_page_len,
                                       pkd_prefix_plan_t *plan, int32_t *host_image,
                                       size_t host_image_bytes);

/* pkd_plan_shared_prefix_host into pinned_staging, then one asynchronous
 * copy of the image into int_ws_dev on `stream`. */
pkd_status pkd_plan_shared_prefix(const pkd_problem *problem,
                                  const int32_t *prefix_pages_h,
                                  int32_t prefix_num_pages,
                                  int32_t prefix_last_page_len,
                                  pkd_prefix_plan_t *plan, int32_t *pinned_staging,
                                  size_t staging_bytes, void *int_ws_dev,
                                  size_t int_ws_bytes, void *stream);

/* Launches the shared-prefix kernel and the merge of its chunk states.
 * q [batch][Hq][D], k_pages / v_pages in problem->kv_layout (NHD or HND);
 * out [batch][Hq][D], lse [batch][Hq].
 * Range-check failures and wait timeouts land in the image's status word
 * (pkd_check_status on int_ws_dev). */
pkd_status pkd_run_shared_prefix(const pkd_prefix_plan_t *plan, const void *q,
                                 const void *k_pages, const void *v_pages,
                                 void *int_ws_dev, void *float_ws_dev,
                                 size_t float_ws_bytes, float sm_scale, void *out,
                                 float *lse, void *stream);

/* The shared-prefix kernel alone: leaves the state of every (request, query
 * head, prefix chunk) in float_ws_dev (fp32, the layout of pkd_run's partial
 * states, slot b * plan->chunks + c) for pkd_run_cascade_merge.  Arguments
 * and errors as pkd_run_shared_prefix, without out / lse. */
pkd_status pkd_run_shared_prefix_states(const pkd_prefix_plan_t *plan, const void *q,
                                        const void *k_pages, const void *v_pages,
                                        void *int_ws_dev, void *float_ws_dev,
                                        size_t float_ws_bytes, float sm_scale,
                                        void *stream);

/*
 * Cascade attention in one call ([W] "Attention states": the states of a
 * shared prefix and of each request's own suffix merge into the state over
 * both): attention of every request over the shared prefix followed by its
 * suffix.  `plan` is the suffix plan (pkd_plan over each request's own
 * pages; kv_* describe those pages) and `prefix_plan` the shared prefix
 * (pkd_plan_shared_prefix); both must have the same batch, heads, head_dim,
 * dtype, page_size, num_pages and kv_layout (else PKD_ERR_INVALID_ARG, no
 * launch), and one q / k_pages / v_pages serves both.  Launches, on
 * `stream`: the shared-prefix kernel (chunk states into
 * prefix_float_ws_dev), the decode kernel of pkd_run_decode_states (every
 * request's suffix state fp32 in float_ws_dev, which must hold
 * plan->num_partials + batch slots), then pkd_run_cascade_merge, which rounds
 * each final state to the output type once.  The decode kernel reads nothing
 * the prefix kernel writes, so it is launched as a programmatic dependent of
 * it (its CTAs may start while the prefix kernel's last CTAs run) and waits
 * for the prefix grid before exiting; the merge, ordered after the decode
 * grid, therefore sees both kernels' states.  out [batch][Hq][D] and lse
 * [batch][Hq] receive the final states; a request with no tokens at all gets
 * (0, -inf).  No separate prefix out / lse and no pkd_merge_states pass: the
 * prefix states stay fp32 until the final merge.  Workspaces: each plan's
 * own, as for pkd_run and pkd_run_shared_prefix.  Graph capture: as for
 * pkd_run_shared_prefix (the prefix plan, which fixes the batch, must stay
 * unchanged); the suffix plan may change between replays within the same
 * batch.  Device-side mismatches land in the suffix image's status word
 * (PKD_DEVICE_BAD_PLAN) or the prefix image's (pkd_check_status).
 */
pkd_status pkd_run_cascade(const pkd_plan_t *plan, const void *q, const void *k_pages,
                           const void *v_pages, const int32_t *kv_indptr_d,
                           const int32_t *kv_indices_d,
                           const int32_t *kv_last_page_len_d, void *int_ws_dev,
                           void *float_ws_dev, size_t float_ws_bytes,
                           const pkd_prefix_plan_t *prefix_plan, void *prefix_int_ws_dev,
                           void *prefix_float_ws_dev, size_t prefix_float_ws_bytes,
                           float sm_scale, void *out, float *lse, void *stream);

/* The last launch of pkd_run_cascade, for callers that launch the prefix
 * states (pkd_run_shared_prefix_states) and the suffix decode
 * (pkd_run_decode_states) themselves, in that order on `stream`, immediately
 * before this call.  Per (request b, query head h) row it folds the prefix
 * chunk states with the fp32 suffix state (the request's partial states if
 * its suffix plan split it, else slot plan->num_partials + b) and writes the
 * result, rounded once, to out / lse.  float_ws_bytes must hold
 * plan->num_partials + batch slots (PKD_ERR_WORKSPACE).  Launched as a
 * programmatic dependent of the decode kernel. */
pkd_status pkd_run_cascade_merge(const pkd_plan_t *plan, void *int_ws_dev,
                                 const void *float_ws_dev, size_t float_ws_bytes,
                                 const pkd_prefix_plan_t *prefix_plan,
                                 const void *prefix_int_ws_dev,
                                 const void *prefix_float_ws_dev,
                                 size_t prefix_float_ws_bytes, void *out, float *lse,
                                 void *stream);

#ifdef __cplusplus
}
#endif

#endif /* PKD_H */

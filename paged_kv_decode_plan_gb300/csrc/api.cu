// C-ABI entry points declared in include/pkd.h.
#include <cuda_runtime.h>

#include <cmath>
#include <string>

#include "pkd_internal.h"

namespace {

using pkd::fail;

pkd_status cuda_fail(cudaError_t e, const char *what) {
  return fail(PKD_ERR_CUDA, std::string(what) + ": " + cudaGetErrorString(e));
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// True while `stream` is being captured into a CUDA graph.
bool capturing(void *stream) {
  cudaStreamCaptureStatus st = cudaStreamCaptureStatusNone;
  return cudaStreamIsCapturing(static_cast<cudaStream_t>(stream), &st) == cudaSuccess &&
         st == cudaStreamCaptureStatusActive;
}

// Bounds a launch may trust for the plan image and partial states.  Under
// capture they are the capacity of the problem and of the float workspace, so
// that replays stay valid for any later plan of the same problem.
struct Bounds {
  int batch, max_partials, image_words;
};

Bounds launch_bounds(const pkd_plan_t &plan, size_t float_ws_bytes, bool capture) {
  const pkd_problem &p = plan.problem;
  Bounds b;
  const long long slot = pkd::partial_slot_floats(p.num_qo_heads, p.head_dim) * 4;
  const long long slots = static_cast<long long>(float_ws_bytes) / slot;
  b.max_partials = static_cast<int>(slots < INT32_MAX ? slots : INT32_MAX);
  if (capture) {
    size_t int_ws = 0;
    pkd::workspace_bytes(p, &int_ws, nullptr, nullptr);
    b.batch = p.max_batch > 0 ? p.max_batch : p.batch;
    b.image_words = static_cast<int>(int_ws / 4);
  } else {
    b.batch = p.batch;
    b.image_words = static_cast<int>(plan.int_ws_bytes_used / 4);
  }
  return b;
}

// Fills num_ctas from the current device when it is 0.
pkd_status resolve_ctas(pkd_problem *p) {
  if (p->num_ctas > 0) return PKD_OK;
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess)
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return cuda_fail(e, "querying the multiprocessor count");
  p->num_ctas = sms;
  return PKD_OK;
}

// Checks a prefix plan's launch and starts the shared-prefix kernel, which
// leaves each (request, head, chunk) state in the prefix float workspace.
pkd_status start_prefix(const pkd_prefix_plan_t *plan, const void *q, const void *k_pages,
                        const void *v_pages, void *int_ws_dev, void *float_ws_dev,
                        size_t float_ws_bytes, float sm_scale, void *stream) {
  if (!plan || !plan->valid) return fail(PKD_ERR_INVALID_ARG, "prefix plan not valid");
  const pkd_problem &p = plan->problem;
  pkd_status st = pkd::check_problem(p, true);
  if (st != PKD_OK) return st;
  if (p.batch == 0) return PKD_OK;
  if (!q || !k_pages || !v_pages || !int_ws_dev || !float_ws_dev)
    return fail(PKD_ERR_INVALID_ARG, "null device pointer");
  if (!aligned16(q) || !aligned16(k_pages) || !aligned16(v_pages) ||
      !aligned16(int_ws_dev) || !aligned16(float_ws_dev))
    return fail(PKD_ERR_UNSUPPORTED, "device pointers must be 16-byte aligned");
  if (float_ws_bytes < static_cast<size_t>(plan->float_ws_bytes_needed))
    return fail(PKD_ERR_WORKSPACE, "float workspace smaller than the prefix plan needs");
  if (!std::isfinite(sm_scale) || !(sm_scale > 0.f))
    return fail(PKD_ERR_INVALID_ARG, "sm_scale must be finite and positive");
  pkd::PrefixArgs a;
  a.q = q;
  a.k_pages = k_pages;
  a.v_pages = v_pages;
  a.image = static_cast<int32_t *>(int_ws_dev);
  a.partials = static_cast<float *>(float_ws_dev);
  a.sm_scale_log2 = sm_scale * 1.4426950408889634f;
  a.num_pages = p.num_pages;
  a.batch = p.batch;
  a.num_qo_heads = p.num_qo_heads;
  a.num_kv_heads = p.num_kv_heads;
  a.page_size = p.page_size;
  a.dtype = p.dtype;
  a.length = plan->prefix_len;
  a.chunks = plan->chunks;
  a.chunk_tiles = plan->chunk_tiles;
  a.row_tiles = plan->row_tiles;
  a.layout = p.kv_layout;
  cudaError_t e = static_cast<cudaError_t>(pkd::launch_shared_prefix(a, stream));
  if (e == cudaErrorNotSupported)
    return fail(PKD_ERR_UNSUPPORTED, "TMA tensor maps unavailable for these pages");
  if (e != cudaSuccess) return cuda_fail(e, "launching the shared-prefix kernel");
  return PKD_OK;
}

// A suffix plan and a prefix plan that describe one cascade: the same
// requests, heads and dtype over one page pool.
pkd_status check_cascade(const pkd_plan_t *plan, const pkd_prefix_plan_t *prefix_plan) {
  if (!plan || !plan->valid) return fail(PKD_ERR_INVALID_ARG, "plan not valid");
  if (!prefix_plan || !prefix_plan->valid)
    return fail(PKD_ERR_INVALID_ARG, "prefix plan not valid");
  const pkd_problem &a = plan->problem, &b = prefix_plan->problem;
  pkd_status st = pkd::check_problem(a, true);
  if (st != PKD_OK) return st;
  if (a.batch != b.batch || a.num_qo_heads != b.num_qo_heads ||
      a.num_kv_heads != b.num_kv_heads || a.head_dim != b.head_dim || a.dtype != b.dtype ||
      a.page_size != b.page_size || a.num_pages != b.num_pages ||
      a.kv_layout != b.kv_layout)
    return fail(PKD_ERR_INVALID_ARG,
                "suffix and prefix plans differ in batch, heads, dtype or page pool");
  return PKD_OK;
}

// fp32 state slots of a states-only decode: the plan's partial slots, then
// one per request (pkd_run_decode_states).
size_t states_bytes(const pkd_plan_t &plan) {
  const pkd_problem &p = plan.problem;
  return static_cast<size_t>(plan.num_partials + p.batch) *
         static_cast<size_t>(pkd::partial_slot_floats(p.num_qo_heads, p.head_dim)) *
         sizeof(float);
}

// Checks a decode launch and starts the decode kernel (pkd_run_decode, or
// pkd_run_decode_states with states_only; the cascade launches the latter as
// a programmatic dependent of the prefix kernel).
pkd_status launch_decode_checked(const pkd_plan_t *plan, const void *q, const void *k_pages,
                                 const void *v_pages, const int32_t *kv_indptr_d,
                                 const int32_t *kv_indices_d,
                                 const int32_t *kv_last_page_len_d, void *int_ws_dev,
                                 void *float_ws_dev, size_t float_ws_bytes, float sm_scale,
                                 void *out, float *lse, void *stream, int programmatic,
                                 int states_only, bool check_only = false) {
  if (!plan || !plan->valid) return fail(PKD_ERR_INVALID_ARG, "plan not valid");
  const pkd_problem &p = plan->problem;
  pkd_status st = pkd::check_problem(p, true);
  if (st != PKD_OK) return st;
  if (p.batch == 0) return PKD_OK;
  if (!q || (!states_only && (!out || !lse)) || !kv_indptr_d || !kv_last_page_len_d ||
      !int_ws_dev)
    return fail(PKD_ERR_INVALID_ARG, "null device pointer");
  if (plan->total_tokens > 0 && (!k_pages || !v_pages || !kv_indices_d))
    return fail(PKD_ERR_INVALID_ARG, "null page pool or page ids");
  if (!aligned16(q) || !aligned16(k_pages) || !aligned16(v_pages) ||
      !aligned16(out) || !aligned16(int_ws_dev) || !aligned16(float_ws_dev))
    return fail(PKD_ERR_UNSUPPORTED, "device pointers must be 16-byte aligned");
  const size_t need =
      states_only ? states_bytes(*plan) : static_cast<size_t>(plan->float_ws_bytes_needed);
  if ((plan->num_partials > 0 || states_only) && (!float_ws_dev || float_ws_bytes < need))
    return fail(PKD_ERR_WORKSPACE, "float workspace smaller than the plan needs");
  if (!std::isfinite(sm_scale) || !(sm_scale > 0.f))
    return fail(PKD_ERR_INVALID_ARG, "sm_scale must be finite and positive");
  if (check_only) return PKD_OK;

  pkd::DecodeArgs a;
  a.q = q;
  a.k_pages = k_pages;
  a.v_pages = v_pages;
  a.kv_indptr = kv_indptr_d;
  a.kv_indices = kv_indices_d;
  a.kv_last_page_len = kv_last_page_len_d;
  a.image = static_cast<int32_t *>(int_ws_dev);
  a.partials = static_cast<float *>(float_ws_dev);
  a.out = out;
  a.lse = lse;
  a.sm_scale_log2 = sm_scale * 1.4426950408889634f;
  const Bounds bounds = launch_bounds(*plan, float_ws_bytes, capturing(stream));
  a.num_pages = p.num_pages;
  a.batch = bounds.batch;
  a.num_qo_heads = p.num_qo_heads;
  a.num_kv_heads = p.num_kv_heads;
  a.page_size = p.page_size;
  a.num_ctas = p.num_ctas;
  a.dtype = p.dtype;
  a.max_partials = bounds.max_partials;
  a.image_words = bounds.image_words;
  a.loader = p.kv_loader;
  a.layout = p.kv_layout;
  a.programmatic = programmatic;
  a.states_only = states_only;
  cudaError_t e = static_cast<cudaError_t>(pkd::launch_decode(a, stream));
  if (e == cudaErrorNotSupported)
    return fail(PKD_ERR_UNSUPPORTED, "TMA tensor maps unavailable for these pages");
  if (e != cudaSuccess) return cuda_fail(e, "launching the decode kernel");
  return PKD_OK;
}

}  // namespace

extern "C" {

int32_t pkd_abi_version(void) { return PKD_ABI_VERSION; }

const char *pkd_last_error(void) { return pkd::last_error_cstr(); }

pkd_status pkd_workspace_size(const pkd_problem *problem, size_t *int_ws_bytes,
                              size_t *float_ws_bytes, size_t *staging_bytes) {
  pkd::clear_error();
  if (!problem) return fail(PKD_ERR_INVALID_ARG, "null problem");
  pkd_problem p = *problem;
  pkd_status st = resolve_ctas(&p);
  if (st != PKD_OK) return st;
  st = pkd::check_problem(p, true);
  if (st != PKD_OK) return st;
  pkd::workspace_bytes(p, int_ws_bytes, float_ws_bytes, staging_bytes);
  return PKD_OK;
}

pkd_status pkd_plan_host(const pkd_problem *problem, const int32_t *kv_indptr_h,
                         const int32_t *kv_last_page_len_h,
                         const int32_t *kv_indices_h, pkd_plan_t *plan,
                         int32_t *host_image, size_t host_image_bytes) {
  pkd::clear_error();
  if (!problem) return fail(PKD_ERR_INVALID_ARG, "null problem");
  return pkd::plan_host_impl(*problem, kv_indptr_h, kv_last_page_len_h,
                             kv_indices_h, plan, host_image, host_image_bytes);
}

pkd_status pkd_plan(const pkd_problem *problem, const int32_t *kv_indptr_h,
                    const int32_t *kv_last_page_len_h,
                    const int32_t *kv_indices_h, pkd_plan_t *plan,
                    int32_t *pinned_staging, size_t staging_bytes,
                    void *int_ws_dev, size_t int_ws_bytes, void *stream) {
  pkd::clear_error();
  if (!problem || !int_ws_dev) return fail(PKD_ERR_INVALID_ARG, "null pointer");
  pkd_problem p = *problem;
  pkd_status st = resolve_ctas(&p);
  if (st != PKD_OK) return st;
  st = pkd::plan_host_impl(p, kv_indptr_h, kv_last_page_len_h, kv_indices_h,
                           plan, pinned_staging, staging_bytes);
  if (st != PKD_OK) return st;
  if (static_cast<size_t>(plan->int_ws_bytes_used) > int_ws_bytes) {
    plan->valid = 0;
    return fail(PKD_ERR_WORKSPACE, "int workspace smaller than the plan image");
  }
  cudaError_t e = cudaMemcpyAsync(int_ws_dev, pinned_staging,
                                  static_cast<size_t>(plan->int_ws_bytes_used),
                                  cudaMemcpyHostToDevice,
                                  static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) {
    plan->valid = 0;
    return cuda_fail(e, "copying the plan image");
  }
  return PKD_OK;
}

pkd_status pkd_run_decode(const pkd_plan_t *plan, const void *q,
                          const void *k_pages, const void *v_pages,
                          const int32_t *kv_indptr_d, const int32_t *kv_indices_d,
                          const int32_t *kv_last_page_len_d, void *int_ws_dev,
                          void *float_ws_dev, size_t float_ws_bytes,
                          float sm_scale, void *out, float *lse, void *stream) {
  pkd::clear_error();
  return launch_decode_checked(plan, q, k_pages, v_pages, kv_indptr_d, kv_indices_d,
                               kv_last_page_len_d, int_ws_dev, float_ws_dev, float_ws_bytes,
                               sm_scale, out, lse, stream, 0, 0);
}

pkd_status pkd_run_decode_states(const pkd_plan_t *plan, const void *q,
                                 const void *k_pages, const void *v_pages,
                                 const int32_t *kv_indptr_d, const int32_t *kv_indices_d,
                                 const int32_t *kv_last_page_len_d, void *int_ws_dev,
                                 void *float_ws_dev, size_t float_ws_bytes, float sm_scale,
                                 void *stream) {
  pkd::clear_error();
  return launch_decode_checked(plan, q, k_pages, v_pages, kv_indptr_d, kv_indices_d,
                               kv_last_page_len_d, int_ws_dev, float_ws_dev, float_ws_bytes,
                               sm_scale, nullptr, nullptr, stream, 0, 1);
}

pkd_status pkd_run_merge(const pkd_plan_t *plan, const void *int_ws_dev,
                         const void *float_ws_dev, size_t float_ws_bytes,
                         void *out, float *lse, void *stream) {
  pkd::clear_error();
  if (!plan || !plan->valid) return fail(PKD_ERR_INVALID_ARG, "plan not valid");
  const pkd_problem &p = plan->problem;
  pkd_status st = pkd::check_problem(p, true);
  if (st != PKD_OK) return st;
  // a captured merge runs whatever later plan the image holds, so it is
  // launched even when this plan split nothing
  const bool capture = capturing(stream);
  if (plan->num_split_requests == 0 && !capture) return PKD_OK;
  if (!int_ws_dev || !float_ws_dev || !out || !lse)
    return fail(PKD_ERR_INVALID_ARG, "null device pointer");
  if (!aligned16(out) || !aligned16(int_ws_dev) || !aligned16(float_ws_dev))
    return fail(PKD_ERR_UNSUPPORTED, "device pointers must be 16-byte aligned");
  if (float_ws_bytes < static_cast<size_t>(plan->float_ws_bytes_needed))
    return fail(PKD_ERR_WORKSPACE, "float workspace smaller than the plan needs");
  pkd::MergePartialsArgs m;
  m.image = static_cast<const int32_t *>(int_ws_dev);
  m.partials = static_cast<const float *>(float_ws_dev);
  m.out = out;
  m.lse = lse;
  m.num_qo_heads = p.num_qo_heads;
  m.dtype = p.dtype;
  const Bounds bounds = launch_bounds(*plan, float_ws_bytes, capture);
  m.batch = bounds.batch;
  m.max_partials = bounds.max_partials;
  m.image_words = bounds.image_words;
  m.num_partials = plan->num_partials;
  m.num_split = plan->num_split_requests;
  m.rows_bound = capture ? bounds.batch : plan->num_split_requests;
  m.grid = 4 * p.num_ctas;  // upper bound on CTAs; rows loop inside
  cudaError_t e = static_cast<cudaError_t>(pkd::launch_merge_partials(m, stream));
  if (e != cudaSuccess) return cuda_fail(e, "launching the merge kernel");
  return PKD_OK;
}

pkd_status pkd_run(const pkd_plan_t *plan, const void *q, const void *k_pages,
                   const void *v_pages, const int32_t *kv_indptr_d,
                   const int32_t *kv_indices_d,
                   const int32_t *kv_last_page_len_d, void *int_ws_dev,
                   void *float_ws_dev, size_t float_ws_bytes, float sm_scale,
                   void *out, float *lse, void *stream) {
  pkd_status st = pkd_run_decode(plan, q, k_pages, v_pages, kv_indptr_d,
                                 kv_indices_d, kv_last_page_len_d, int_ws_dev,
                                 float_ws_dev, float_ws_bytes, sm_scale, out, lse,
                                 stream);
  if (st != PKD_OK) return st;
  return pkd_run_merge(plan, int_ws_dev, float_ws_dev, float_ws_bytes, out, lse,
                       stream);
}

pkd_status pkd_merge_states(const void *v_a, const float *s_a, const void *v_b,
                            const float *s_b, void *v_out, float *s_out,
                            int64_t n, int32_t num_heads, int32_t head_dim,
                            int32_t v_dtype, void *stream) {
  pkd::clear_error();
  if (n < 0 || num_heads <= 0 || head_dim <= 0)
    return fail(PKD_ERR_INVALID_ARG, "negative or zero size");
  if (v_dtype != PKD_F16 && v_dtype != PKD_BF16 && v_dtype != PKD_F32)
    return fail(PKD_ERR_UNSUPPORTED, "v_dtype must be F16, BF16 or F32");
  if (head_dim % 8 != 0 || head_dim > 1024)
    return fail(PKD_ERR_UNSUPPORTED, "head_dim must be a multiple of 8, <= 1024");
  if (n == 0) return PKD_OK;
  if (!v_a || !s_a || !v_b || !s_b || !v_out || !s_out)
    return fail(PKD_ERR_INVALID_ARG, "null pointer");
  if (!aligned16(v_a) || !aligned16(v_b) || !aligned16(v_out))
    return fail(PKD_ERR_UNSUPPORTED, "state pointers must be 16-byte aligned");
  cudaError_t e = static_cast<cudaError_t>(pkd::launch_merge_states(
      v_a, s_a, v_b, s_b, v_out, s_out, n, num_heads, head_dim, v_dtype, stream));
  if (e != cudaSuccess) return cuda_fail(e, "launching merge_states");
  return PKD_OK;
}

pkd_status pkd_append_kv(const pkd_problem *problem, const void *k_new,
                         const void *v_new, const int32_t *batch_indices_d,
                         const int32_t *positions_d, int64_t num_new, void *k_pages,
                         void *v_pages, const int32_t *kv_indptr_d,
                         const int32_t *kv_indices_d,
                         const int32_t *kv_last_page_len_d, uint32_t *device_status,
                         void *stream) {
  pkd::clear_error();
  if (!problem) return fail(PKD_ERR_INVALID_ARG, "null problem");
  pkd_problem p = *problem;
  if (p.num_ctas == 0) p.num_ctas = 1;  // not used here
  pkd_status st = pkd::check_problem(p, false);
  if (st != PKD_OK) return st;
  if (num_new < 0) return fail(PKD_ERR_INVALID_ARG, "negative token count");
  if (num_new == 0) return PKD_OK;
  if (!k_new || !v_new || !batch_indices_d || !positions_d || !k_pages || !v_pages ||
      !kv_indptr_d || !kv_indices_d || !kv_last_page_len_d)
    return fail(PKD_ERR_INVALID_ARG, "null device pointer");
  if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(k_pages) || !aligned16(v_pages))
    return fail(PKD_ERR_UNSUPPORTED, "K/V pointers must be 16-byte aligned");
  pkd::AppendArgs a;
  a.k_new = k_new;
  a.v_new = v_new;
  a.batch_indices = batch_indices_d;
  a.positions = positions_d;
  a.k_pages = k_pages;
  a.v_pages = v_pages;
  a.kv_indptr = kv_indptr_d;
  a.kv_indices = kv_indices_d;
  a.kv_last_page_len = kv_last_page_len_d;
  a.status = device_status;
  a.num_new = num_new;
  a.num_pages = p.num_pages;
  a.batch = p.batch;
  a.num_kv_heads = p.num_kv_heads;
  a.page_size = p.page_size;
  a.layout = p.kv_layout;
  cudaError_t e = static_cast<cudaError_t>(pkd::launch_append(a, stream));
  if (e != cudaSuccess) return cuda_fail(e, "launching the append kernel");
  return PKD_OK;
}

pkd_status pkd_prefix_workspace_size(const pkd_problem *problem,
                                     int32_t max_prefix_pages, size_t *int_ws_bytes,
                                     size_t *float_ws_bytes, size_t *staging_bytes) {
  pkd::clear_error();
  if (!problem) return fail(PKD_ERR_INVALID_ARG, "null problem");
  if (max_prefix_pages < 0) return fail(PKD_ERR_INVALID_ARG, "negative page count");
  pkd_problem p = *problem;
  pkd_status st = resolve_ctas(&p);
  if (st != PKD_OK) return st;
  st = pkd::check_problem(p, true);
  if (st != PKD_OK) return st;
  pkd::prefix_workspace_bytes(p, max_prefix_pages, int_ws_bytes, float_ws_bytes,
                              staging_bytes);
  return PKD_OK;
}

pkd_status pkd_plan_shared_prefix_host(const pkd_problem *problem,
                                       const int32_t *prefix_pages_h,
                                       int32_t prefix_num_pages,
                                       int32_t prefix_last_page_len,
                                       pkd_prefix_plan_t *plan, int32_t *host_image,
                                       size_t host_image_bytes) {
  pkd::clear_error();
  if (!problem) return fail(PKD_ERR_INVALID_ARG, "null problem");
  return pkd::plan_prefix_impl(*problem, prefix_pages_h, prefix_num_pages,
                               prefix_last_page_len, plan, host_image, host_image_bytes);
}

pkd_status pkd_plan_shared_prefix(const pkd_problem *problem,
                                  const int32_t *prefix_pages_h,
                                  int32_t prefix_num_pages,
                                  int32_t prefix_last_page_len,
                                  pkd_prefix_plan_t *plan, int32_t *pinned_staging,
                                  size_t staging_bytes, void *int_ws_dev,
                                  size_t int_ws_bytes, void *stream) {
  pkd::clear_error();
  if (!problem || !int_ws_dev) return fail(PKD_ERR_INVALID_ARG, "null pointer");
  pkd_problem p = *problem;
  pkd_status st = resolve_ctas(&p);
  if (st != PKD_OK) return st;
  st = pkd::plan_prefix_impl(p, prefix_pages_h, prefix_num_pages, prefix_last_page_len,
                             plan, pinned_staging, staging_bytes);
  if (st != PKD_OK) return st;
  if (static_cast<size_t>(plan->int_ws_bytes_used) > int_ws_bytes) {
    plan->valid = 0;
    return fail(PKD_ERR_WORKSPACE, "int workspace smaller than the prefix plan image");
  }
  cudaError_t e = cudaMemcpyAsync(int_ws_dev, pinned_staging,
                                  static_cast<size_t>(plan->int_ws_bytes_used),
                                  cudaMemcpyHostToDevice,
                                  static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) {
    plan->valid = 0;
    return cuda_fail(e, "copying the prefix plan image");
  }
  return PKD_OK;
}

pkd_status pkd_run_shared_prefix_states(const pkd_prefix_plan_t *plan, const void *q,
                                        const void *k_pages, const void *v_pages,
                                        void *int_ws_dev, void *float_ws_dev,
                                        size_t float_ws_bytes, float sm_scale,
                                        void *stream) {
  pkd::clear_error();
  return start_prefix(plan, q, k_pages, v_pages, int_ws_dev, float_ws_dev, float_ws_bytes,
                      sm_scale, stream);
}

pkd_status pkd_run_shared_prefix(const pkd_prefix_plan_t *plan, const void *q,
                                 const void *k_pages, const void *v_pages,
                                 void *int_ws_dev, void *float_ws_dev,
                                 size_t float_ws_bytes, float sm_scale, void *out,
                                 float *lse, void *stream) {
  pkd::clear_error();
  if (plan && plan->valid && plan->problem.batch > 0) {
    if (!out || !lse) return fail(PKD_ERR_INVALID_ARG, "null device pointer");
    if (!aligned16(out)) return fail(PKD_ERR_UNSUPPORTED, "device pointers must be 16-byte aligned");
  }
  pkd_status st = start_prefix(plan, q, k_pages, v_pages, int_ws_dev, float_ws_dev,
                               float_ws_bytes, sm_scale, stream);
  if (st != PKD_OK || plan->problem.batch == 0) return st;
  const pkd_problem &p = plan->problem;
  cudaError_t e = static_cast<cudaError_t>(pkd::launch_merge_uniform(
      static_cast<const float *>(float_ws_dev), out, lse, p.batch, p.num_qo_heads,
      plan->chunks, p.dtype, 4 * p.num_ctas, stream));
  if (e != cudaSuccess) return cuda_fail(e, "launching the prefix merge");
  return PKD_OK;
}

pkd_status pkd_run_cascade_merge(const pkd_plan_t *plan, void *int_ws_dev,
                                 const void *float_ws_dev, size_t float_ws_bytes,
                                 const pkd_prefix_plan_t *prefix_plan,
                                 const void *prefix_int_ws_dev,
                                 const void *prefix_float_ws_dev,
                                 size_t prefix_float_ws_bytes, void *out, float *lse,
                                 void *stream) {
  pkd::clear_error();
  pkd_status st = check_cascade(plan, prefix_plan);
  if (st != PKD_OK) return st;
  const pkd_problem &p = plan->problem;
  if (p.batch == 0) return PKD_OK;
  if (!int_ws_dev || !prefix_int_ws_dev || !prefix_float_ws_dev || !out || !lse)
    return fail(PKD_ERR_INVALID_ARG, "null device pointer");
  if (!aligned16(out) || !aligned16(int_ws_dev) || !aligned16(float_ws_dev) ||
      !aligned16(prefix_int_ws_dev) || !aligned16(prefix_float_ws_dev))
    return fail(PKD_ERR_UNSUPPORTED, "device pointers must be 16-byte aligned");
  if (prefix_float_ws_bytes < static_cast<size_t>(prefix_plan->float_ws_bytes_needed))
    return fail(PKD_ERR_WORKSPACE, "prefix float workspace smaller than its plan needs");
  const bool capture = capturing(stream);
  if (!float_ws_dev || float_ws_bytes < states_bytes(*plan))
    return fail(PKD_ERR_WORKSPACE, "float workspace smaller than the suffix states need");
  const Bounds bounds = launch_bounds(*plan, float_ws_bytes, capture);
  pkd::CascadeMergeArgs m;
  m.image = static_cast<const int32_t *>(int_ws_dev);
  m.partials = static_cast<const float *>(float_ws_dev);
  m.prefix_image = static_cast<const int32_t *>(prefix_int_ws_dev);
  m.prefix_partials = static_cast<const float *>(prefix_float_ws_dev);
  m.out = out;
  m.lse = lse;
  m.num_qo_heads = p.num_qo_heads;
  m.dtype = p.dtype;
  m.batch = p.batch;
  m.chunks = prefix_plan->chunks;
  m.max_partials = bounds.max_partials;
  m.image_words = bounds.image_words;
  cudaError_t e = static_cast<cudaError_t>(pkd::launch_cascade_merge(m, stream));
  if (e != cudaSuccess) return cuda_fail(e, "launching the cascade merge");
  return PKD_OK;
}

pkd_status pkd_run_cascade(const pkd_plan_t *plan, const void *q, const void *k_pages,
                           const void *v_pages, const int32_t *kv_indptr_d,
                           const int32_t *kv_indices_d,
                           const int32_t *kv_last_page_len_d, void *int_ws_dev,
                           void *float_ws_dev, size_t float_ws_bytes,
                           const pkd_prefix_plan_t *prefix_plan, void *prefix_int_ws_dev,
                           void *prefix_float_ws_dev, size_t prefix_float_ws_bytes,
                           float sm_scale, void *out, float *lse, void *stream) {
  pkd::clear_error();
  // every host-side check before the first launch
  pkd_status st = check_cascade(plan, prefix_plan);
  if (st != PKD_OK) return st;
  if (plan->problem.batch == 0) return PKD_OK;
  if (!out || !lse || !prefix_float_ws_dev)
    return fail(PKD_ERR_INVALID_ARG, "null device pointer");
  if (!aligned16(out))
    return fail(PKD_ERR_UNSUPPORTED, "device pointers must be 16-byte aligned");
  if (prefix_float_ws_bytes < static_cast<size_t>(prefix_plan->float_ws_bytes_needed))
    return fail(PKD_ERR_WORKSPACE, "prefix float workspace smaller than its plan needs");
  st = launch_decode_checked(plan, q, k_pages, v_pages, kv_indptr_d, kv_indices_d,
                             kv_last_page_len_d, int_ws_dev, float_ws_dev, float_ws_bytes,
                             sm_scale, nullptr, nullptr, stream, 1, 1, true);
  if (st != PKD_OK) return st;
  st = start_prefix(prefix_plan, q, k_pages, v_pages, prefix_int_ws_dev,
                    prefix_float_ws_dev, prefix_float_ws_bytes, sm_scale, stream);
  if (st != PKD_OK) return st;
  // the suffix decode reads nothing the prefix kernel writes: it may start as
  // the prefix kernel's CTAs retire (and waits for that grid before exiting).
  // It leaves every request's suffix state in fp32, so the final state is
  // rounded to the output type once.
  st = launch_decode_checked(plan, q, k_pages, v_pages, kv_indptr_d, kv_indices_d,
                             kv_last_page_len_d, int_ws_dev, float_ws_dev, float_ws_bytes,
                             sm_scale, nullptr, nullptr, stream, 1, 1);
  if (st != PKD_OK) return st;
  return pkd_run_cascade_merge(plan, int_ws_dev, float_ws_dev, float_ws_bytes, prefix_plan,
                               prefix_int_ws_dev, prefix_float_ws_dev,
                               prefix_float_ws_bytes, out, lse, stream);
}

pkd_status pkd_check_status(const void *int_ws_dev, uint32_t *device_status,
                            void *stream) {
  pkd::clear_error();
  if (!int_ws_dev || !device_status) return fail(PKD_ERR_INVALID_ARG, "null pointer");
  uint32_t word = 0;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemcpyAsync(
      &word, static_cast<const int32_t *>(int_ws_dev) + pkd::kHStatus,
      sizeof(word), cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_fail(e, "reading the device status word");
  *device_status = word;
  if (word != 0)
    return fail(PKD_ERR_DEVICE_CHECK,
                "device status word " + std::to_string(word));
  return PKD_OK;
}

}  // extern "C"

// Internal declarations shared by the library's translation units.
#pragma once

#include <cstddef>
#include <cstdint>
#include <string>

#include "pkd.h"

#ifdef __CUDACC__
#define PKD_HD __host__ __device__
#else
#define PKD_HD
#endif

namespace pkd {

// Plan image layout (int32 words).  Header words:
constexpr int kMagic = 0x31444B50;  // "PKD1"
constexpr int kLayoutVersion = 1;
constexpr int kHeaderWords = 16;
enum HeaderWord {
  kHMagic = 0,
  kHVersion = 1,
  kHBatch = 2,
  kHNumCtas = 3,
  kHNumUnits = 4,
  kHNumPartials = 5,
  kHNumSplit = 6,
  kHTileTokens = 7,
  kHPageSize = 8,
  kHTotalTiles = 9,
  kHQuota = 10,
  kHMinChunks = 11,
  kHStatus = 12,
  kHNumQoHeads = 13,
};
constexpr int kUnitWords = 4;  // req, tok_begin, tok_end, partial slot (-1)

// Word offsets of the arrays that follow the header.
struct ImageOffsets {
  int64_t cta_ptr, units, merge_indptr, merge_req, end;
};
PKD_HD inline ImageOffsets image_offsets(int64_t num_ctas, int64_t num_units,
                                         int64_t num_split) {
  ImageOffsets o;
  o.cta_ptr = kHeaderWords;
  o.units = o.cta_ptr + num_ctas + 1;
  o.merge_indptr = o.units + kUnitWords * num_units;
  o.merge_req = o.merge_indptr + num_split + 1;
  o.end = o.merge_req + num_split;
  return o;
}

// Partial states: per slot, o [Hq][D] floats then lse [Hq] floats padded to a
// multiple of 4, so every o row starts 16-byte aligned.
PKD_HD inline int64_t partial_slot_floats(int64_t hq, int64_t d) {
  return hq * d + ((hq + 3) / 4) * 4;
}

constexpr int kHeadDim = 128;
constexpr int kMaxGroup = 16;
constexpr int kTileTokens = 16;  // tokens per decode tile, every Hkv

// Thread-local error message; returns `status` for convenience.
pkd_status fail(pkd_status status, const std::string &message);
void clear_error();
const char *last_error_cstr();

// Validates the parts of a problem every entry point needs.
pkd_status check_problem(const pkd_problem &p, bool need_ctas);
int64_t max_units(const pkd_problem &p);

// Workspace sizes for a problem with explicit num_ctas.
void workspace_bytes(const pkd_problem &p, size_t *int_ws, size_t *float_ws,
                     size_t *staging);

// Planning on the host (plan.cpp).
pkd_status plan_host_impl(const pkd_problem &in, const int32_t *kv_indptr,
                          const int32_t *kv_last_page_len,
                          const int32_t *kv_indices, pkd_plan_t *plan,
                          int32_t *image, size_t image_bytes);

// Launchers (decode.cu, merge.cu).  Return cudaError_t as int.
struct DecodeArgs {
  const void *q, *k_pages, *v_pages;
  const int32_t *kv_indptr, *kv_indices, *kv_last_page_len;
  int32_t *image;
  float *partials;
  void *out;
  float *lse;
  float sm_scale_log2;
  int64_t num_pages;
  int batch, num_qo_heads, num_kv_heads, page_size, num_ctas, dtype;
  int max_partials, image_words;
  int loader;  // pkd_loader of the problem
  int layout;  // pkd_layout of the page tensors
  int programmatic;  // launch as a programmatic dependent of the previous kernel
  int states_only;   // fp32 states for every request (slot num_partials + b when unsplit)
};
int launch_decode(const DecodeArgs &a, void *stream);

struct MergePartialsArgs {
  const int32_t *image;
  const float *partials;
  void *out;
  float *lse;
  int num_qo_heads, dtype, grid, batch, max_partials, image_words;
  int num_partials, num_split;  // from the plan, to choose warps per row
  int rows_bound;               // split requests the grid is sized for
};
int launch_merge_partials(const MergePartialsArgs &a, void *stream);

// Page append (append.cu).
struct AppendArgs {
  const void *k_new, *v_new;
  const int32_t *batch_indices, *positions;
  void *k_pages, *v_pages;
  const int32_t *kv_indptr, *kv_indices, *kv_last_page_len;
  uint32_t *status;
  int64_t num_new, num_pages;
  int batch, num_kv_heads, page_size, layout;
};
int launch_append(const AppendArgs &a, void *stream);

// Shared-prefix attention (prefix.cu) and its chunk merge (merge.cu).
constexpr int kPrefixMagic = 0x50444B50;  // "PKDP"
enum PrefixHeaderWord {
  kPBatch = 2, kPNumQoHeads = 3, kPNumKvHeads = 4, kPPageSize = 5, kPLength = 6,
  kPNumPages = 7, kPChunks = 8, kPChunkTiles = 9, kPRowTiles = 10,
};
struct PrefixArgs {
  const void *q, *k_pages, *v_pages;
  int32_t *image;
  float *partials;
  float sm_scale_log2;
  int64_t num_pages;
  int batch, num_qo_heads, num_kv_heads, page_size, dtype;
  int length, chunks, chunk_tiles, row_tiles;
  int layout;
};
int launch_shared_prefix(const PrefixArgs &a, void *stream);
int launch_merge_uniform(const float *partials, void *out, float *lse, int batch, int hq,
                         int chunks, int dtype, int grid, void *stream);
// Cascade merge (merge.cu): prefix chunk states + suffix states -> out, lse.
struct CascadeMergeArgs {
  const int32_t *image;          // suffix plan image
  const float *partials;         // suffix partial states
  const int32_t *prefix_image;   // prefix plan image
  const float *prefix_partials;  // prefix chunk states
  void *out;
  float *lse;
  int num_qo_heads, dtype;
  int batch, chunks;             // of the prefix plan (the suffix image must agree)
  int max_partials, image_words; // bounds for the suffix image
};
int launch_cascade_merge(const CascadeMergeArgs &a, void *stream);
pkd_status plan_prefix_impl(const pkd_problem &in, const int32_t *pages,
                            int32_t num_prefix_pages, int32_t last_page_len,
                            pkd_prefix_plan_t *plan, int32_t *image, size_t image_bytes);
void prefix_workspace_bytes(const pkd_problem &p, int32_t max_prefix_pages,
                            size_t *int_ws, size_t *float_ws, size_t *staging);

// Tensor maps for K and V page pools: NHD viewed as [token row][head][d]
// (3-D), HND as [page][head][slot][d] (4-D); boxes of 16 token rows x 1 head x
// 64 elements, 128-byte swizzle; cached per pool.  (CUtensorMap comes from
// <cuda.h>; callers include it first.)
#ifdef CUDA_VERSION
bool page_tensor_maps(CUtensorMap *mk, CUtensorMap *mv, const void *k, const void *v,
                      long long num_pages, int page_size, int hkv, int layout);
// Queries [batch][hq][d] as a 3-D map with boxes of 64 elements x `group`
// heads x 128 / group requests (128 query rows of one key/value head, in
// request-major order), 128-byte swizzle.  False when 128 % group != 0.
bool query_tensor_map(CUtensorMap *map, const void *q, int batch, int hq, int group);
#endif

int launch_merge_states(const void *v_a, const float *s_a, const void *v_b,
                        const float *s_b, void *v_out, float *s_out, int64_t n,
                        int num_heads, int head_dim, int dtype, void *stream);

}  // namespace pkd

// Host-side planning: page-table validation, request lengths, the split-KV
// work list and the plan image.  No CUDA here.
//
// The pages fix only that planning reads sequence lengths and page-table
// metadata, chooses a schedule and prepares workspace data that a later run
// applies ("FlashInfer" (aiwiki.ai/wiki/flashinfer), "Plan and run"), and
// that a long cache may be split across work units whose partial states are
// merged afterwards (same page, "Attention states").  The rule below is this
// library's own ("balanced contiguous split"):
//   * request b has n_b = ceil(L_b / T) tiles of T tokens;
//   * with m = min_chunks_per_request > 1, request b is first cut at tile
//     multiples of c_b = max(1, floor(n_b / m));
//   * the requests' tiles, in order, are dealt to CTAs 0..C-1, each taking a
//     quota Q = max(1, ceil(W / C)) of the W tiles (the last CTA takes what
//     remains), a piece ending at a cap-chunk boundary, a quota boundary or
//     the request's end; every piece is one unit (req, tok_begin, tok_end);
//   * an empty request is one unit (b, 0, 0) in the current CTA;
//   * a request with one unit writes its output directly; the units of a
//     split request get consecutive partial-state slots and the request is
//     listed for the merge step.
#include <algorithm>
#include <cstring>
#include <string>
#include <vector>

#include "pkd_internal.h"

namespace pkd {

namespace {
thread_local std::string g_last_error;
}

pkd_status fail(pkd_status status, const std::string &message) {
  g_last_error = message;
  return status;
}

void clear_error() { g_last_error.clear(); }

const char *last_error_cstr() { return g_last_error.c_str(); }

pkd_status check_problem(const pkd_problem &p, bool need_ctas) {
  if (p.batch < 0 || p.num_qo_heads <= 0 || p.num_kv_heads <= 0 ||
      p.head_dim <= 0 || p.page_size <= 0 || p.num_pages < 0 ||
      p.num_ctas < 0 || p.min_chunks_per_request < 0 || p.tile_tokens < 0 ||
      p.max_batch < 0)
    return fail(PKD_ERR_INVALID_ARG, "negative or zero problem field");
  if (p.max_batch != 0 && p.max_batch < p.batch)
    return fail(PKD_ERR_INVALID_ARG, "batch exceeds max_batch");
  if (p.num_qo_heads % p.num_kv_heads != 0)
    return fail(PKD_ERR_INVALID_ARG, "num_qo_heads % num_kv_heads != 0");
  if (p.dtype != PKD_F16 && p.dtype != PKD_BF16)
    return fail(PKD_ERR_UNSUPPORTED, "dtype must be PKD_F16 or PKD_BF16");
  if (p.head_dim != kHeadDim)
    return fail(PKD_ERR_UNSUPPORTED, "head_dim must be 128");
  if (p.num_kv_heads != 1 && p.num_kv_heads != 2 && p.num_kv_heads != 4 &&
      p.num_kv_heads != 8)
    return fail(PKD_ERR_UNSUPPORTED, "num_kv_heads must be 1, 2, 4 or 8");
  if (p.num_qo_heads / p.num_kv_heads > kMaxGroup)
    return fail(PKD_ERR_UNSUPPORTED, "query group larger than 16");
  if (p.tile_tokens != 0 && p.tile_tokens != kTileTokens)
    return fail(PKD_ERR_UNSUPPORTED, "tile_tokens must be 0 or 16");
  if (p.kv_layout != PKD_LAYOUT_NHD && p.kv_layout != PKD_LAYOUT_HND)
    return fail(PKD_ERR_INVALID_ARG, "kv_layout must be a pkd_layout value");
  if (p.kv_loader < PKD_LOADER_AUTO || p.kv_loader > PKD_LOADER_BULK_ROWS)
    return fail(PKD_ERR_INVALID_ARG, "kv_loader must be a pkd_loader value");
  if (p.kv_loader == PKD_LOADER_TMA_TILES && p.page_size % kTileTokens != 0)
    return fail(PKD_ERR_UNSUPPORTED, "TMA tiles need page_size % 16 == 0");
  if (need_ctas && p.num_ctas <= 0)
    return fail(PKD_ERR_INVALID_ARG, "num_ctas must be explicit here");
  return PKD_OK;
}

int64_t max_units(const pkd_problem &p) {
  const int64_t cap_batch = p.max_batch > 0 ? p.max_batch : p.batch;
  const int64_t m = std::max(1, p.min_chunks_per_request);
  // a request yields at most 2m - 1 cap-chunks; each quota boundary adds at
  // most one cut
  return cap_batch * (2 * m - 1) + p.num_ctas;
}

void workspace_bytes(const pkd_problem &p, size_t *int_ws, size_t *float_ws,
                     size_t *staging) {
  const int64_t cap_batch = p.max_batch > 0 ? p.max_batch : p.batch;
  const int64_t units = max_units(p);
  const ImageOffsets o = image_offsets(p.num_ctas, units, cap_batch);
  const size_t int_bytes = static_cast<size_t>(o.end) * sizeof(int32_t);
  if (int_ws) *int_ws = int_bytes;
  if (staging) *staging = int_bytes;
  // partial slots for every unit, plus one per request: a states-only decode
  // (the cascade's suffix) puts unsplit request b's state in slot
  // num_partials + b
  if (float_ws)
    *float_ws = static_cast<size_t>(units + cap_batch) *
                partial_slot_floats(p.num_qo_heads, p.head_dim) * sizeof(float);
}

pkd_status plan_host_impl(const pkd_problem &in, const int32_t *kv_indptr,
                          const int32_t *kv_last_page_len,
                          const int32_t *kv_indices, pkd_plan_t *plan,
                          int32_t *image, size_t image_bytes) {
  if (!plan || !image || (in.batch > 0 && (!kv_indptr || !kv_last_page_len)) ||
      (in.batch == 0 && !kv_indptr))
    return fail(PKD_ERR_INVALID_ARG, "null pointer");
  pkd_problem p = in;
  if (p.tile_tokens == 0) p.tile_tokens = kTileTokens;
  pkd_status st = check_problem(p, true);
  if (st != PKD_OK) return st;
  // tile_tokens is 0 or kTileTokens (check_problem): a compile-time divisor
  constexpr int T = kTileTokens;
  const int B = p.batch, P = p.page_size, C = p.num_ctas;
  const int m = std::max(1, p.min_chunks_per_request);

  // 1. validate the CSR table, compute lengths and tiles
  if (kv_indptr[0] < 0) return fail(PKD_ERR_PAGE_TABLE, "kv_indptr[0] < 0");
  std::vector<int64_t> length(B), tiles(B);
  int64_t total_tiles = 0, total_tokens = 0;
  for (int b = 0; b < B; ++b) {
    const int64_t npages = static_cast<int64_t>(kv_indptr[b + 1]) - kv_indptr[b];
    if (npages < 0)
      return fail(PKD_ERR_PAGE_TABLE,
                  "kv_indptr decreases at request " + std::to_string(b));
    if (npages == 0) {
      length[b] = 0;
    } else {
      const int32_t last = kv_last_page_len[b];
      if (last < 1 || last > P)
        return fail(PKD_ERR_PAGE_TABLE, "kv_last_page_len out of [1, page_size] "
                                        "at request " + std::to_string(b));
      length[b] = (npages - 1) * P + last;
    }
    if (length[b] > INT32_MAX - T)
      return fail(PKD_ERR_UNSUPPORTED, "request longer than 2^31 tokens");
    tiles[b] = (length[b] + T - 1) / T;
    total_tiles += tiles[b];
    total_tokens += length[b];
  }
  if (kv_indices) {
    // branch-free min / max pass (vectorised); the failing index is looked up
    // only when a page id is out of range
    const int64_t i0 = kv_indptr[0], i1 = kv_indptr[B];
    const int32_t *__restrict ids = kv_indices + i0;
    const int64_t n = i1 - i0;
    int32_t lo = n > 0 ? ids[0] : 0, hi = lo;
    for (int64_t i = 0; i < n; ++i) {
      const int32_t v = ids[i];
      lo = v < lo ? v : lo;
      hi = v > hi ? v : hi;
    }
    if (n > 0 && (lo < 0 || hi >= p.num_pages))
      for (int64_t i = i0; i < i1; ++i)
        if (kv_indices[i] < 0 || kv_indices[i] >= p.num_pages)
          return fail(PKD_ERR_PAGE_TABLE,
                      "page id out of range at kv_indices[" + std::to_string(i) + "]");
  } else if (total_tokens > 0 && p.num_pages <= 0) {
    return fail(PKD_ERR_PAGE_TABLE, "non-empty table over an empty pool");
  }
  if (total_tiles > INT32_MAX)
    return fail(PKD_ERR_UNSUPPORTED, "more than 2^31 tiles");

  // 2-4. deal tiles to CTAs
  const int64_t quota = std::max<int64_t>(1, (total_tiles + C - 1) / C);
  struct Unit { int32_t req, t0, t1, slot; };
  std::vector<Unit> units;
  units.reserve(static_cast<size_t>(std::min<int64_t>(max_units(p), total_tiles + B + C)));
  std::vector<int32_t> cta_ptr;
  cta_ptr.reserve(C + 1);
  cta_ptr.push_back(0);
  int cta = 0;
  int64_t used = 0;
  for (int b = 0; b < B; ++b) {
    const int64_t n = tiles[b];
    if (n == 0) {
      units.push_back({b, 0, 0, -1});
      continue;
    }
    const int64_t cap = m <= 1 ? n : std::max<int64_t>(1, n / m);
    int64_t pos = 0;
    while (pos < n) {
      if (used >= quota && cta < C - 1) {
        cta_ptr.push_back(static_cast<int32_t>(units.size()));
        ++cta;
        used = 0;
      }
      const int64_t room = cta < C - 1 ? quota - used : n - pos;
      const int64_t to_cap = m <= 1 ? n - pos : cap - pos % cap;
      const int64_t take = std::min(std::min(n - pos, to_cap), room);
      units.push_back({b, static_cast<int32_t>(pos * T),
                       static_cast<int32_t>(std::min((pos + take) * T, length[b])),
                       -1});
      pos += take;
      used += take;
    }
  }
  while (static_cast<int>(cta_ptr.size()) < C + 1)
    cta_ptr.push_back(static_cast<int32_t>(units.size()));

  // 5. partial slots and merge lists
  std::vector<int32_t> pieces(B, 0);
  for (const Unit &u : units) ++pieces[u.req];
  int32_t slot = 0;
  for (Unit &u : units)
    if (pieces[u.req] > 1) u.slot = slot++;
  std::vector<int32_t> merge_indptr{0}, merge_req;
  for (int b = 0; b < B; ++b)
    if (pieces[b] > 1) {
      merge_req.push_back(b);
      merge_indptr.push_back(merge_indptr.back() + pieces[b]);
    }

  const int64_t nunits = static_cast<int64_t>(units.size());
  const int64_t nsplit = static_cast<int64_t>(merge_req.size());
  if (nunits > max_units(p))
    return fail(PKD_ERR_WORKSPACE, "work list exceeds the capacity bound");
  const ImageOffsets o = image_offsets(C, nunits, nsplit);
  const size_t need = static_cast<size_t>(o.end) * sizeof(int32_t);
  if (need > image_bytes)
    return fail(PKD_ERR_WORKSPACE, "plan image needs " + std::to_string(need) +
                                       " bytes, buffer has " +
                                       std::to_string(image_bytes));

  int32_t *w = image;
  std::memset(w, 0, kHeaderWords * sizeof(int32_t));
  w[kHMagic] = kMagic;
  w[kHVersion] = kLayoutVersion;
  w[kHBatch] = B;
  w[kHNumCtas] = C;
  w[kHNumUnits] = static_cast<int32_t>(nunits);
  w[kHNumPartials] = slot;
  w[kHNumSplit] = static_cast<int32_t>(nsplit);
  w[kHTileTokens] = T;
  w[kHPageSize] = P;
  w[kHTotalTiles] = static_cast<int32_t>(total_tiles);
  w[kHQuota] = static_cast<int32_t>(quota);
  w[kHMinChunks] = m;
  w[kHStatus] = 0;
  w[kHNumQoHeads] = p.num_qo_heads;
  std::memcpy(w + o.cta_ptr, cta_ptr.data(), cta_ptr.size() * sizeof(int32_t));
  for (int64_t i = 0; i < nunits; ++i) {
    int32_t *u = w + o.units + kUnitWords * i;
    u[0] = units[i].req;
    u[1] = units[i].t0;
    u[2] = units[i].t1;
    u[3] = units[i].slot;
  }
  std::memcpy(w + o.merge_indptr, merge_indptr.data(),
              merge_indptr.size() * sizeof(int32_t));
  if (nsplit)
    std::memcpy(w + o.merge_req, merge_req.data(), nsplit * sizeof(int32_t));

  std::memset(plan, 0, sizeof(*plan));
  plan->problem = p;
  plan->num_units = static_cast<int32_t>(nunits);
  plan->num_partials = slot;
  plan->num_split_requests = static_cast<int32_t>(nsplit);
  plan->total_tiles = static_cast<int32_t>(total_tiles);
  plan->total_tokens = total_tokens;
  plan->int_ws_bytes_used = static_cast<int64_t>(need);
  plan->float_ws_bytes_needed =
      static_cast<int64_t>(slot) * partial_slot_floats(p.num_qo_heads, p.head_dim) *
      static_cast<int64_t>(sizeof(float));
  plan->valid = 1;
  return PKD_OK;
}

// Shared-prefix planning: validate the page list, split the prefix into KV
// chunks so that (heads x row tiles x chunks) fills the CTA budget, write the
// image (header + page ids).
namespace {
constexpr int kPrefixTile = 64;   // tokens per prefix stage (prefix.cu)
constexpr int kPrefixRows = 256;  // query rows per prefix CTA: two 128-row MMA tiles (prefix.cu)
}  // namespace

void prefix_workspace_bytes(const pkd_problem &p, int32_t max_prefix_pages,
                            size_t *int_ws, size_t *float_ws, size_t *staging) {
  const int64_t cap_batch = p.max_batch > 0 ? p.max_batch : p.batch;
  const int64_t max_chunks = std::max(1, p.num_ctas / std::max(1, p.num_kv_heads));
  const size_t ib = static_cast<size_t>(kHeaderWords + std::max(0, max_prefix_pages)) * 4;
  if (int_ws) *int_ws = ib;
  if (staging) *staging = ib;
  if (float_ws)
    *float_ws = static_cast<size_t>(cap_batch * max_chunks) *
                partial_slot_floats(p.num_qo_heads, p.head_dim) * sizeof(float);
}

pkd_status plan_prefix_impl(const pkd_problem &in, const int32_t *pages,
                            int32_t num_prefix_pages, int32_t last_page_len,
                            pkd_prefix_plan_t *plan, int32_t *image, size_t image_bytes) {
  if (!plan || !image || (num_prefix_pages > 0 && !pages))
    return fail(PKD_ERR_INVALID_ARG, "null pointer");
  pkd_problem p = in;
  if (p.tile_tokens == 0) p.tile_tokens = kTileTokens;
  pkd_status st = check_problem(p, true);
  if (st != PKD_OK) return st;
  if (p.page_size % kTileTokens != 0)
    return fail(PKD_ERR_UNSUPPORTED, "shared prefix needs page_size % 16 == 0");
  if (num_prefix_pages < 0) return fail(PKD_ERR_INVALID_ARG, "negative page count");
  if (num_prefix_pages > 0 && (last_page_len < 1 || last_page_len > p.page_size))
    return fail(PKD_ERR_PAGE_TABLE, "prefix last_page_len out of [1, page_size]");
  for (int32_t i = 0; i < num_prefix_pages; ++i)
    if (pages[i] < 0 || pages[i] >= p.num_pages)
      return fail(PKD_ERR_PAGE_TABLE,
                  "prefix page id out of range at index " + std::to_string(i));
  const int64_t length =
      num_prefix_pages > 0
          ? static_cast<int64_t>(num_prefix_pages - 1) * p.page_size + last_page_len
          : 0;
  if (length > INT32_MAX - kPrefixTile ||
      static_cast<int64_t>(p.num_pages) * p.page_size >= (1ll << 31))
    return fail(PKD_ERR_UNSUPPORTED, "prefix or pool too long for 32-bit token rows");
  const int64_t need = static_cast<int64_t>(kHeaderWords + num_prefix_pages) * 4;
  if (static_cast<size_t>(need) > image_bytes)
    return fail(PKD_ERR_WORKSPACE, "prefix plan image needs " + std::to_string(need) +
                                       " bytes, buffer has " + std::to_string(image_bytes));
  const int group = p.num_qo_heads / p.num_kv_heads;
  const int64_t rows = static_cast<int64_t>(p.batch) * group;
  const int row_tiles = static_cast<int>(std::max<int64_t>(1, (rows + kPrefixRows - 1) / kPrefixRows));
  const int total_tiles = static_cast<int>((length + kPrefixTile - 1) / kPrefixTile);
  const int base = p.num_kv_heads * row_tiles;
  int chunks = std::max(1, std::min(total_tiles, p.num_ctas / base));
  int chunk_tiles = total_tiles > 0 ? (total_tiles + chunks - 1) / chunks : 0;
  if (chunk_tiles > 0) chunks = (total_tiles + chunk_tiles - 1) / chunk_tiles;

  std::memset(image, 0, kHeaderWords * sizeof(int32_t));
  image[kHMagic] = kPrefixMagic;
  image[kHVersion] = 1;
  image[kPBatch] = p.batch;
  image[kPNumQoHeads] = p.num_qo_heads;
  image[kPNumKvHeads] = p.num_kv_heads;
  image[kPPageSize] = p.page_size;
  image[kPLength] = static_cast<int32_t>(length);
  image[kPNumPages] = num_prefix_pages;
  image[kPChunks] = chunks;
  image[kPChunkTiles] = chunk_tiles;
  image[kPRowTiles] = row_tiles;
  image[kHStatus] = 0;
  if (num_prefix_pages > 0)
    std::memcpy(image + kHeaderWords, pages, num_prefix_pages * sizeof(int32_t));

  std::memset(plan, 0, sizeof(*plan));
  plan->problem = p;
  plan->prefix_len = static_cast<int32_t>(length);
  plan->prefix_num_pages = num_prefix_pages;
  plan->chunks = chunks;
  plan->chunk_tiles = chunk_tiles;
  plan->row_tiles = row_tiles;
  plan->num_blocks = p.num_kv_heads * row_tiles * chunks;
  plan->int_ws_bytes_used = need;
  plan->float_ws_bytes_needed = static_cast<int64_t>(p.batch) * chunks *
                                partial_slot_floats(p.num_qo_heads, p.head_dim) * 4;
  plan->valid = 1;
  return PKD_OK;
}

}  // namespace pkd

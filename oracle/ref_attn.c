/*
 * Oracle for paged decode attention and attention-state merging.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the plain, slow, fp64 CPU statement
 * of what the GPU path computes.  Only the test-suite, the smoke check and the
 * benchmark's CPU-baseline leg may load it.  It shares no code, header, table
 * or helper with the CUDA library, and the library never calls it.
 *
 * Sources (page title, section):
 *  - "FlashInfer" (aiwiki.ai/wiki/flashinfer), "Block-sparse cache
 *    representation": the cache is a set of non-contiguous blocks (pages)
 *    reached through a page table.
 *  - same page, "Custom attention templates": grouped-query heads, several
 *    query heads share one key/value head.
 *  - same page, "Attention states": attention over part of a cache is an
 *    (output, log-sum-exp) pair; states of disjoint regions merge into the
 *    state of their union, using the log-sum-exp values to put both parts
 *    under one normaliser (partial outputs may not simply be averaged).
 *  - same page, "Extreme-negative-logit correction": the running maximum
 *    starts at IEEE -infinity, never a finite sentinel; a row with nothing to
 *    attend to yields a zero output with -infinity log-sum-exp.
 *  - "Welcome to FlashInfer's documentation!" (docs.flashinfer.ai), tutorial
 *    "KV-Cache Layout in FlashInfer": NHD layout and the page-table layout.
 *
 * Readings where the pages are silent (each also listed in the design notes):
 *  - The page table is CSR: request b owns pages
 *    kv_indices[kv_indptr[b] .. kv_indptr[b+1]) in sequence order; every page
 *    is full except the last, which holds kv_last_page_len[b] tokens, 1..P.
 *    A request with no pages has length 0 and its last_page_len is ignored.
 *  - NHD: a page tensor is [num_pages][page_size][num_kv_heads][head_dim];
 *    HND: [num_pages][num_kv_heads][page_size][head_dim]; both row-major, K
 *    and V separate tensors of the same layout.
 *  - Query head h reads key/value head h / g with g = Hq / Hkv.
 *  - Logits include the scale: s_t = sm_scale * <q, k_t>; the log-sum-exp is
 *    the natural logarithm of sum_t exp(s_t).
 *
 * Method: the plain definition of softmax attention, two passes per row
 * (maximum, then normaliser and weighted sum), everything in double.  The
 * inputs are half / bfloat16 / float / double values, widened exactly.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { ORC_F16 = 0, ORC_BF16 = 1, ORC_F32 = 2, ORC_F64 = 3 };
enum { ORC_NHD = 0, ORC_HND = 1 };

enum {
  ORC_OK = 0,
  ORC_ERR_ARG = -1,
  ORC_ERR_PAGE_TABLE = -2,
  ORC_ERR_NOMEM = -3
};

/* IEEE 754 binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction
 * bits.  Exponent 0 is subnormal (fraction * 2^-24); exponent 31 is inf/NaN. */
static double widen_f16(uint16_t bits) {
  int sign = (bits >> 15) & 1;
  int expo = (bits >> 10) & 0x1f;
  int frac = bits & 0x3ff;
  double mag;
  if (expo == 0) {
    mag = ldexp((double)frac, -24);
  } else if (expo == 31) {
    mag = frac ? NAN : INFINITY;
  } else {
    mag = ldexp((double)(frac | 0x400), expo - 25);
  }
  return sign ? -mag : mag;
}

/* bfloat16 is the upper half of an IEEE binary32 word. */
static double widen_bf16(uint16_t bits) {
  uint32_t word = (uint32_t)bits << 16;
  float f;
  memcpy(&f, &word, sizeof f);
  return (double)f;
}

static double element(const void *base, int dtype, int64_t i) {
  switch (dtype) {
    case ORC_F16: return widen_f16(((const uint16_t *)base)[i]);
    case ORC_BF16: return widen_bf16(((const uint16_t *)base)[i]);
    case ORC_F32: return (double)((const float *)base)[i];
    default: return ((const double *)base)[i];
  }
}

int orc_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* Element offset of (page, slot, kv head, d = 0) in a page tensor. */
static int64_t row_base(int layout, int64_t page, int64_t slot, int kvh,
                        int page_size, int num_kv_heads, int head_dim) {
  if (layout == ORC_HND)
    return ((page * num_kv_heads + kvh) * page_size + slot) * head_dim;
  return ((page * page_size + slot) * num_kv_heads + kvh) * head_dim;
}

/* Number of tokens of request b under the CSR reading above. */
static int64_t request_length(const int32_t *kv_indptr,
                              const int32_t *kv_last_page_len, int page_size,
                              int b) {
  int64_t npages = (int64_t)kv_indptr[b + 1] - kv_indptr[b];
  if (npages == 0) return 0;
  return (npages - 1) * page_size + kv_last_page_len[b];
}

/* Checks the page table; returns ORC_OK or ORC_ERR_PAGE_TABLE. */
static int check_table(int batch, int page_size, int64_t num_pages,
                       const int32_t *kv_indptr, const int32_t *kv_indices,
                       const int32_t *kv_last_page_len) {
  if (kv_indptr[0] < 0) return ORC_ERR_PAGE_TABLE;
  for (int b = 0; b < batch; ++b) {
    if (kv_indptr[b + 1] < kv_indptr[b]) return ORC_ERR_PAGE_TABLE;
    if (kv_indptr[b + 1] > kv_indptr[b] &&
        (kv_last_page_len[b] < 1 || kv_last_page_len[b] > page_size))
      return ORC_ERR_PAGE_TABLE;
    for (int32_t p = kv_indptr[b]; p < kv_indptr[b + 1]; ++p)
      if (kv_indices[p] < 0 || kv_indices[p] >= num_pages)
        return ORC_ERR_PAGE_TABLE;
  }
  return ORC_OK;
}

/*
 * Decode attention for the listed rows (row r = b * Hq + h), or for all
 * B * Hq rows when `rows` is NULL.  out is [n_rows][head_dim], lse [n_rows].
 * q is [B][Hq][D]; k_pages and v_pages are page tensors in `layout`.
 */
int orc_decode(int batch, int num_qo_heads, int num_kv_heads, int head_dim,
               int page_size, int dtype, int layout, const void *q, const void *k_pages,
               const void *v_pages, int64_t num_pages, const int32_t *kv_indptr,
               const int32_t *kv_indices, const int32_t *kv_last_page_len,
               double sm_scale, const int64_t *rows, int64_t n_rows,
               double *out, double *lse) {
  if (batch < 0 || num_qo_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0 ||
      page_size <= 0 || num_qo_heads % num_kv_heads != 0 || dtype < ORC_F16 ||
      dtype > ORC_F64 || (layout != ORC_NHD && layout != ORC_HND))
    return ORC_ERR_ARG;
  int rc = check_table(batch, page_size, num_pages, kv_indptr, kv_indices,
                       kv_last_page_len);
  if (rc != ORC_OK) return rc;
  if (rows == NULL) n_rows = (int64_t)batch * num_qo_heads;
  for (int64_t i = 0; i < n_rows; ++i) {
    int64_t r = rows ? rows[i] : i;
    if (r < 0 || r >= (int64_t)batch * num_qo_heads) return ORC_ERR_ARG;
  }

  const int group = num_qo_heads / num_kv_heads;
  int failed = 0;

#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t i = 0; i < n_rows; ++i) {
    int64_t r = rows ? rows[i] : i;
    int b = (int)(r / num_qo_heads);
    int h = (int)(r % num_qo_heads);
    int kvh = h / group;
    int64_t n = request_length(kv_indptr, kv_last_page_len, page_size, b);
    double *o = out + i * head_dim;
    for (int d = 0; d < head_dim; ++d) o[d] = 0.0;
    if (n == 0) {
      lse[i] = -INFINITY;
      continue;
    }
    double *s = (double *)malloc((size_t)n * sizeof(double));
    if (!s) {
#pragma omp atomic write
      failed = 1;
      continue;
    }
    const int64_t q_base = r * head_dim;
    /* token t lives in page kv_indices[kv_indptr[b] + t / P], slot t % P */
    for (int64_t t = 0; t < n; ++t) {
      int64_t page = kv_indices[kv_indptr[b] + t / page_size];
      int64_t slot = t % page_size;
      int64_t k_base =
          row_base(layout, page, slot, kvh, page_size, num_kv_heads, head_dim);
      double dot = 0.0;
      for (int d = 0; d < head_dim; ++d)
        dot += element(q, dtype, q_base + d) * element(k_pages, dtype, k_base + d);
      s[t] = sm_scale * dot;
    }
    double m = -INFINITY;
    for (int64_t t = 0; t < n; ++t)
      if (s[t] > m) m = s[t];
    double z = 0.0;
    for (int64_t t = 0; t < n; ++t) {
      double w = exp(s[t] - m);
      z += w;
      int64_t page = kv_indices[kv_indptr[b] + t / page_size];
      int64_t slot = t % page_size;
      int64_t v_base =
          row_base(layout, page, slot, kvh, page_size, num_kv_heads, head_dim);
      for (int d = 0; d < head_dim; ++d)
        o[d] += w * element(v_pages, dtype, v_base + d);
    }
    for (int d = 0; d < head_dim; ++d) o[d] /= z;
    lse[i] = m + log(z);
    free(s);
  }
  return failed ? ORC_ERR_NOMEM : ORC_OK;
}

/*
 * Merge of two attention states (v_a, s_a) and (v_b, s_b) over disjoint
 * regions into the state of their union ("Attention states"):
 *   s = log(exp(s_a) + exp(s_b)),   v = exp(s_a - s) v_a + exp(s_b - s) v_b,
 * evaluated against the common maximum M = max(s_a, s_b).  A side whose
 * log-sum-exp is -infinity covers nothing and contributes nothing; when both
 * sides are empty the union is empty: (0, -infinity).
 * v arrays are [n_rows][head_dim]; s arrays are [n_rows].
 */
int orc_merge(int64_t n_rows, int head_dim, const double *v_a, const double *s_a,
              const double *v_b, const double *s_b, double *v_out,
              double *s_out) {
  if (n_rows < 0 || head_dim <= 0) return ORC_ERR_ARG;
  for (int64_t i = 0; i < n_rows; ++i) {
    double *v = v_out + i * head_dim;
    if (s_a[i] == -INFINITY && s_b[i] == -INFINITY) {
      for (int d = 0; d < head_dim; ++d) v[d] = 0.0;
      s_out[i] = -INFINITY;
      continue;
    }
    double m = s_a[i] > s_b[i] ? s_a[i] : s_b[i];
    double wa = exp(s_a[i] - m);
    double wb = exp(s_b[i] - m);
    double z = wa + wb;
    for (int d = 0; d < head_dim; ++d)
      v[d] = (wa * v_a[i * head_dim + d] + wb * v_b[i * head_dim + d]) / z;
    s_out[i] = m + log(z);
  }
  return ORC_OK;
}

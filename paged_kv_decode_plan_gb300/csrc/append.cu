// Page append: writes new tokens' key and value rows into their slots of the
// paged cache ("Welcome to FlashInfer's documentation!", flashinfer.page
// "Append new K/V tensors to Paged KV-Cache").
//
// New token i belongs to request batch_indices[i] at position positions[i];
// the page table already covers the request's new length, so the token's
// slot is page kv_indices[kv_indptr[b] + t / P], slot t % P.  One warp per
// (token, tensor) copies the token's rows of all heads (Hkv * 256 contiguous
// bytes in NHD) with 16-byte loads and stores.  Tokens outside their
// request's length or on a page id outside the pool are skipped and reported
// in the optional status word.
#include <cuda_runtime.h>

#include "pkd_internal.h"

namespace pkd {
namespace {

struct AppendParams {
  const uint16_t *k_new, *v_new;
  const int32_t *batch_indices, *positions;
  uint16_t *k_pages, *v_pages;
  const int32_t *indptr, *indices, *last;
  uint32_t *status;
  long long num_new, num_pages;
  int batch, hkv, page_size, hnd;
};

__global__ void __launch_bounds__(256) append_kernel(const AppendParams p) {
  const int lane = threadIdx.x & 31;
  const long long warps = static_cast<long long>(gridDim.x) * (blockDim.x >> 5);
  const int chunks = p.hkv * (kHeadDim * 2 / 16);  // 16-byte chunks per row
  for (long long w = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
       w < 2 * p.num_new; w += warps) {
    const long long i = w >> 1;
    const int tensor = static_cast<int>(w & 1);
    const int b = __ldg(p.batch_indices + i);
    const int t = __ldg(p.positions + i);
    unsigned bad = 0;
    long long row = 0;
    if (b < 0 || b >= p.batch || t < 0) {
      bad = PKD_DEVICE_BAD_LENGTH;
    } else {
      const int pb = __ldg(p.indptr + b), pe = __ldg(p.indptr + b + 1);
      const int last = min(max(__ldg(p.last + b), 1), p.page_size);
      const long long len =
          pe > pb ? static_cast<long long>(pe - pb - 1) * p.page_size + last : 0;
      if (t >= len) {
        bad = PKD_DEVICE_BAD_LENGTH;
      } else {
        const int pi = t / p.page_size;
        const int page = __ldg(p.indices + pb + pi);
        if (page < 0 || page >= p.num_pages)
          bad = PKD_DEVICE_BAD_PAGE;
        else
          row = static_cast<long long>(page) * p.page_size + (t - pi * p.page_size);
      }
    }
    if (bad) {
      if (lane == 0 && p.status) atomicOr(p.status, bad);
      continue;
    }
    const uint4 *src = reinterpret_cast<const uint4 *>(
        (tensor ? p.v_new : p.k_new) + i * p.hkv * kHeadDim);
    uint16_t *pages = tensor ? p.v_pages : p.k_pages;
    if (p.hnd) {
      // HND: head h's row of this token is at ((page * Hkv + h) * P + slot)
      const long long page = row / p.page_size, slot = row - page * p.page_size;
      for (int c = lane; c < chunks; c += 32) {
        const int h = c >> 4, w = c & 15;
        reinterpret_cast<uint4 *>(
            pages + ((page * p.hkv + h) * p.page_size + slot) * kHeadDim)[w] =
            __ldg(src + c);
      }
    } else {
      uint4 *dst = reinterpret_cast<uint4 *>(pages + row * p.hkv * kHeadDim);
      for (int c = lane; c < chunks; c += 32) dst[c] = __ldg(src + c);
    }
  }
}

}  // namespace

int launch_append(const AppendArgs &a, void *stream) {
  if (a.num_new == 0) return cudaSuccess;
  AppendParams p;
  p.k_new = static_cast<const uint16_t *>(a.k_new);
  p.v_new = static_cast<const uint16_t *>(a.v_new);
  p.batch_indices = a.batch_indices;
  p.positions = a.positions;
  p.k_pages = static_cast<uint16_t *>(a.k_pages);
  p.v_pages = static_cast<uint16_t *>(a.v_pages);
  p.indptr = a.kv_indptr;
  p.indices = a.kv_indices;
  p.last = a.kv_last_page_len;
  p.status = a.status;
  p.num_new = a.num_new;
  p.num_pages = a.num_pages;
  p.batch = a.batch;
  p.hkv = a.num_kv_heads;
  p.page_size = a.page_size;
  p.hnd = a.layout == PKD_LAYOUT_HND;
  const long long warps = 2 * a.num_new;
  const long long want = (warps + 7) / 8;
  const int grid = static_cast<int>(want < 65535LL * 8 ? want : 65535LL * 8);
  append_kernel<<<grid, 256, 0, static_cast<cudaStream_t>(stream)>>>(p);
  return cudaGetLastError();
}

}  // namespace pkd

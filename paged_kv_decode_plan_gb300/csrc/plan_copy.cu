// pkd_copy_plan: the plan image from pinned host memory into the device
// workspace, copied by one small kernel instead of the copy engine.
//
// "FlashInfer" (aiwiki.ai/wiki/flashinfer), "Plan and run": planning prepares
// workspace data on the host and a captured run keeps its device addresses
// while the scheduling data in them is updated.  On GB300 the GPU reads
// pinned host memory directly over the coherent CPU-GPU link, and inside a
// CUDA graph a kernel that loads the image chains onto the decode kernel
// after it without the copy-engine hand-off a cudaMemcpy node costs.  The
// number of words copied is read from the image's own header at run time,
// so a captured copy follows whatever plan the host last wrote into the same
// pinned buffer, and copies only that plan's words.
#include <cuda_runtime.h>

#include <string>

#include "pkd_internal.h"

namespace pkd {
namespace {

constexpr int kCopyThreads = 256;

// Loads that fetch host memory again instead of trusting a cached line.
__device__ __forceinline__ uint4 ld_cv4(const int32_t *p) {
  uint4 v;
  asm volatile("ld.global.cv.v4.u32 {%0, %1, %2, %3}, [%4];\n"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ int32_t ld_cv(const int32_t *p) {
  int32_t v;
  asm volatile("ld.global.cv.u32 %0, [%1];\n" : "=r"(v) : "l"(p));
  return v;
}

// Words of the image the header describes (decode or shared-prefix plan),
// or -1 if the header is neither.
__device__ long long image_words(const int32_t *host) {
  const int magic = ld_cv(host + kHMagic);
  if (magic == kMagic) {
    const int ctas = ld_cv(host + kHNumCtas);
    const int units = ld_cv(host + kHNumUnits);
    const int split = ld_cv(host + kHNumSplit);
    if (ctas < 0 || units < 0 || split < 0) return -1;
    return image_offsets(ctas, units, split).end;
  }
  if (magic == kPrefixMagic) {
    const int pages = ld_cv(host + kPNumPages);
    return pages < 0 ? -1 : kHeaderWords + static_cast<long long>(pages);
  }
  return -1;
}

// cap_words: the fewer of the host buffer's and the workspace's words.
__global__ void __launch_bounds__(kCopyThreads)
    plan_copy_kernel(const int32_t *host, int32_t *dev, long long cap_words) {
  __shared__ long long words_s;
  if (threadIdx.x == 0) words_s = image_words(host);
  __syncthreads();
  const long long want = words_s;
  // an image that is not a plan, or larger than its host buffer or the
  // workspace: copy the header only and flag the device copy, which no
  // kernel then accepts (the entry point checked cap_words >= the header)
  const bool bad = want < kHeaderWords || want > cap_words;
  const long long words = bad ? kHeaderWords : want;
  const long long vecs = words / 4;
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < vecs;
       i += stride)
    reinterpret_cast<uint4 *>(dev)[i] = ld_cv4(host + 4 * i);
  for (long long w = 4 * vecs + static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
       w < words; w += stride)
    dev[w] = ld_cv(host + w);
  if (bad && blockIdx.x == 0) {
    __syncthreads();  // this block copied the status word; flag after it
    if (threadIdx.x == 0)
      atomicOr(reinterpret_cast<unsigned int *>(dev + kHStatus), PKD_DEVICE_BAD_PLAN);
  }
}

}  // namespace
}  // namespace pkd

extern "C" pkd_status pkd_copy_plan(const int32_t *pinned_image, size_t pinned_image_bytes,
                                    void *int_ws_dev, size_t int_ws_bytes, void *stream) {
  pkd::clear_error();
  if (!pinned_image || !int_ws_dev)
    return pkd::fail(PKD_ERR_INVALID_ARG, "null pointer");
  if ((reinterpret_cast<uintptr_t>(pinned_image) & 15u) ||
      (reinterpret_cast<uintptr_t>(int_ws_dev) & 15u))
    return pkd::fail(PKD_ERR_UNSUPPORTED, "image and workspace must be 16-byte aligned");
  if (int_ws_bytes < static_cast<size_t>(pkd::kHeaderWords) * 4 ||
      pinned_image_bytes < static_cast<size_t>(pkd::kHeaderWords) * 4)
    return pkd::fail(PKD_ERR_WORKSPACE, "image or workspace smaller than a plan header");
  cudaPointerAttributes attr;
  cudaError_t e = cudaPointerGetAttributes(&attr, pinned_image);
  if (e != cudaSuccess || attr.type != cudaMemoryTypeHost || !attr.devicePointer) {
    cudaGetLastError();  // a failed query leaves no sticky error
    return pkd::fail(PKD_ERR_INVALID_ARG,
                     "the image must be in pinned (page-locked) host memory");
  }
  const size_t cap_bytes = int_ws_bytes < pinned_image_bytes ? int_ws_bytes : pinned_image_bytes;
  const long long cap_words = static_cast<long long>(cap_bytes / 4);
  const long long vecs = (cap_words + 3) / 4;
  long long blocks = (vecs + pkd::kCopyThreads - 1) / pkd::kCopyThreads;
  if (blocks > 64) blocks = 64;
  if (blocks < 1) blocks = 1;
  pkd::plan_copy_kernel<<<static_cast<unsigned>(blocks), pkd::kCopyThreads, 0,
                          static_cast<cudaStream_t>(stream)>>>(
      static_cast<const int32_t *>(attr.devicePointer), static_cast<int32_t *>(int_ws_dev),
      cap_words);
  e = cudaGetLastError();
  if (e != cudaSuccess)
    return pkd::fail(PKD_ERR_CUDA, std::string("launching the plan copy: ") +
                                       cudaGetErrorString(e));
  return PKD_OK;
}

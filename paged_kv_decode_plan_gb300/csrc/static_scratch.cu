// pkd_run_static: decode attention without any device allocation.
//
// Some callers cannot allocate device memory when they run decode: code whose
// device memory is owned by another allocator (a serving engine's own pool,
// a plug-in inside a framework that forbids raw cudaMalloc), or a latency-
// critical loop that cannot afford cudaMalloc / cudaFree, which may
// synchronise the whole device.  For them this entry point keeps the two
// scratch buffers the decode path needs (the plan image and the fp32 partial
// states) in one file-scope __device__ array of fixed size, which every GPU
// that loads this library holds until the process exits.  It calls no
// cudaMalloc, cudaFree or allocating library routine.
//
// The array's device address is looked up once per device (cudaGetSymbolAddress
// with that device current) on the first call made on that device; make that
// first call before any stream capture.  The address is kept for the life of
// the process: after cudaDeviceReset on a device, do not call this entry
// point on that device again.  A call on a stream that is being captured is
// refused (PKD_ERR_UNSUPPORTED): the plan image is copied from host memory by
// each call and the kernels are bounded by that call's plan, which a captured
// copy and launch would freeze.  Every call shares the array: calls whose
// work overlaps on the GPU (other streams, other threads) race on it.  Each
// call overwrites the plan image completely (its status word starts at 0)
// and every partial slot a plan uses is written before it is read, so
// nothing is left to clear between calls.
#include <cuda_runtime.h>

#include <mutex>
#include <string>

#include "pkd_internal.h"

namespace {

constexpr size_t kStaticImageWords = 64 * 1024;            // 256 KiB
constexpr size_t kStaticPartialFloats = 2 * 1024 * 1024;   // 8 MiB
constexpr int kMaxDevices = 64;

static __device__ __align__(256) int32_t
    g_scratch[kStaticImageWords + kStaticPartialFloats];

std::mutex g_mutex;
void *g_address[kMaxDevices] = {};

pkd_status scratch_address(void **out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess)
    return pkd::fail(PKD_ERR_CUDA, std::string("cudaGetDevice: ") +
                                       cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices)
    return pkd::fail(PKD_ERR_UNSUPPORTED, "device ordinal above 63");
  std::lock_guard<std::mutex> lock(g_mutex);
  if (!g_address[dev]) {
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, g_scratch);
    if (e != cudaSuccess || !p)
      return pkd::fail(PKD_ERR_CUDA, std::string("cudaGetSymbolAddress: ") +
                                         cudaGetErrorString(e));
    g_address[dev] = p;
  }
  *out = g_address[dev];
  return PKD_OK;
}

}  // namespace

extern "C" pkd_status pkd_run_static(const pkd_plan_t *plan,
                                     const int32_t *host_image, const void *q,
                                     const void *k_pages, const void *v_pages,
                                     const int32_t *kv_indptr_d,
                                     const int32_t *kv_indices_d,
                                     const int32_t *kv_last_page_len_d,
                                     float sm_scale, void *out, float *lse,
                                     void *stream) {
  pkd::clear_error();
  if (!plan || !plan->valid || !host_image)
    return pkd::fail(PKD_ERR_INVALID_ARG, "plan not valid or no plan image");
  if (plan->int_ws_bytes_used < 0 ||
      static_cast<size_t>(plan->int_ws_bytes_used) > kStaticImageWords * 4)
    return pkd::fail(PKD_ERR_WORKSPACE,
                     "plan image of " + std::to_string(plan->int_ws_bytes_used) +
                         " bytes exceeds the static limit of 262144 bytes");
  if (plan->float_ws_bytes_needed < 0 ||
      static_cast<size_t>(plan->float_ws_bytes_needed) > kStaticPartialFloats * 4)
    return pkd::fail(PKD_ERR_WORKSPACE,
                     "partial states of " +
                         std::to_string(plan->float_ws_bytes_needed) +
                         " bytes exceed the static limit of 8388608 bytes");
  if (plan->problem.batch == 0) return PKD_OK;
  cudaStreamCaptureStatus capture = cudaStreamCaptureStatusNone;
  cudaError_t e = cudaStreamIsCapturing(static_cast<cudaStream_t>(stream), &capture);
  if (e != cudaSuccess)
    return pkd::fail(PKD_ERR_CUDA, std::string("cudaStreamIsCapturing: ") +
                                       cudaGetErrorString(e));
  if (capture != cudaStreamCaptureStatusNone)
    return pkd::fail(PKD_ERR_UNSUPPORTED,
                     "pkd_run_static is not supported on a capturing stream");
  void *base = nullptr;
  pkd_status st = scratch_address(&base);
  if (st != PKD_OK) return st;
  int32_t *image_d = static_cast<int32_t *>(base);
  float *partials_d = reinterpret_cast<float *>(image_d + kStaticImageWords);
  e = cudaMemcpyAsync(image_d, host_image, static_cast<size_t>(plan->int_ws_bytes_used),
                      cudaMemcpyHostToDevice, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess)
    return pkd::fail(PKD_ERR_CUDA, std::string("copying the plan image: ") +
                                       cudaGetErrorString(e));
  return pkd_run(plan, q, k_pages, v_pages, kv_indptr_d, kv_indices_d,
                 kv_last_page_len_d, image_d, partials_d,
                 kStaticPartialFloats * sizeof(float), sm_scale, out, lse, stream);
}

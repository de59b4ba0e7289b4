// Attention-state merge kernels.
//
// "FlashInfer" (aiwiki.ai/wiki/flashinfer), "Attention states": states of
// disjoint cache regions merge into the state of their union; the partial
// outputs cannot be averaged, their log-sum-exp values give the rescaling to a
// common normaliser.  With M the largest partial lse and w_i = exp(s_i - M):
//   s = M + log(sum_i w_i),   v = sum_i w_i v_i / sum_i w_i.
// A state with s = -infinity covers nothing and gets weight 0; if every state
// is empty the result is (0, -infinity) ("Extreme-negative-logit
// correction": no -inf - (-inf) reaches exp).
#include <cuda_runtime.h>

#include <climits>
#include <cmath>

#include "pkd_internal.h"
#include "ptx.cuh"

namespace pkd {
namespace {

constexpr int kMergeWarps = 8;
constexpr int kMergeThreads = 32 * kMergeWarps;

// Folds one state (lse s, normalised output v) into a running (m, ws, acc)
// by the online rule: a new maximum rescales what was folded so far; a state
// with s = -inf has weight 0.
__device__ __forceinline__ void fold_one(float s, float4 v, float &m, float &ws, float4 &acc) {
  if (s > m) {
    const float f = m == -INFINITY ? 0.f : expf(m - s);
    acc.x *= f;
    acc.y *= f;
    acc.z *= f;
    acc.w *= f;
    ws *= f;
    m = s;
  }
  const float w = s == -INFINITY ? 0.f : expf(s - m);
  acc.x += w * v.x;
  acc.y += w * v.y;
  acc.z += w * v.z;
  acc.w += w * v.w;
  ws += w;
}

// Folds partial states s0, s0 + stride, ... (< s1) of query head h into a
// running (m, ws, acc); kUnroll states' loads are in flight per step.
template <int kUnroll = 4>
__device__ __forceinline__ void fold_states(const float *partials, long long slot_floats,
                                            int hq, int h, int s0, int s1, int stride,
                                            int lane, float &m, float &ws, float4 &acc) {
  for (int j = s0; j < s1; j += kUnroll * stride) {
    float sv[kUnroll];
    float4 ov[kUnroll];
#pragma unroll
    for (int k = 0; k < kUnroll; ++k) {
      const int jj = j + k * stride;
      sv[k] = -INFINITY;
      ov[k] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (jj < s1) {
        const float *base = partials + jj * slot_floats;
        sv[k] = base[hq * kHeadDim + h];
        ov[k] = reinterpret_cast<const float4 *>(base + h * kHeadDim)[lane];
      }
    }
#pragma unroll
    for (int k = 0; k < kUnroll; ++k) fold_one(sv[k], ov[k], m, ws, acc);
  }
}

template <typename T>
__device__ __forceinline__ void write_state(uint16_t *out, float *lse, int b, int hq,
                                            int h, int lane, float m, float ws,
                                            float4 acc) {
  const float inv = ws > 0.f ? 1.f / ws : 0.f;
  uint16_t *dst = out + (static_cast<long long>(b) * hq + h) * kHeadDim + 4 * lane;
  uint2 packed;
  packed.x = ptx::pack2<T>(acc.x * inv, acc.y * inv);
  packed.y = ptx::pack2<T>(acc.z * inv, acc.w * inv);
  *reinterpret_cast<uint2 *>(dst) = packed;
  if (lane == 0)
    lse[static_cast<long long>(b) * hq + h] = ws > 0.f ? m + logf(ws) : -INFINITY;
}

// Chunk merge of the shared-prefix kernel: every request has `chunks` partial
// states in slots b * chunks .. b * chunks + chunks - 1; one warp per
// (request, head) row.
template <typename T>
__global__ void __launch_bounds__(kMergeThreads)
    merge_uniform_kernel(const float *partials, uint16_t *out, float *lse, int batch,
                         int hq, int chunks) {
  const int lane = threadIdx.x & 31;
  const long long slot_floats = partial_slot_floats(hq, kHeadDim);
  const long long rows = static_cast<long long>(batch) * hq;
  ptx::wait_primary_grid();
  for (long long row = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
       row < rows; row += (static_cast<long long>(gridDim.x) * blockDim.x) >> 5) {
    const int b = static_cast<int>(row / hq), h = static_cast<int>(row % hq);
    float m = -INFINITY, ws = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    // a request's chunks are read in one round (the partials sit in L2)
    fold_states<8>(partials, slot_floats, hq, h, b * chunks, (b + 1) * chunks, 1, lane, m,
                   ws, acc);
    write_state<T>(out, lse, b, hq, h, lane, m, ws, acc);
  }
}

// Cascade merge ("FlashInfer" (aiwiki.ai/wiki/flashinfer), "Attention
// states": the states of the shared prefix and of a request's own suffix
// merge into the state over both).  One warp per (request b, query head h)
// row folds the prefix's chunk states (slots b * chunks .. b * chunks +
// chunks - 1 of the prefix workspace) and the suffix state, fp32 throughout
// (the decode kernel ran in its states-only mode): the request's partial
// slots if the suffix plan split it, else slot num_partials + b.  The final
// state is rounded to the output type once.  The suffix plan lists its split
// requests in increasing order; a warp finds b among them 128 at a time (all
// loads in flight) with ballots, before it waits for the decode grid.
//
// At most 64 registers a thread (four CTAs per SM instead of three at the 79
// the compiler would take): once the decode grid ends, the cascade
// workload's 512 CTAs are resident in one wave rather than two (cascade step
// 62.4 -> 59.4 us, A/B on one GPU; 128-thread CTAs, eight per SM, 59.6 us).
template <typename T>
__global__ void __launch_bounds__(kMergeThreads, 4)
    cascade_merge_kernel(const int32_t *image, const float *partials,
                         const int32_t *prefix_image, const float *prefix_partials,
                         uint16_t *out, float *lse, int hq, int batch, int chunks,
                         int max_partials, int image_words) {
  const int lane = threadIdx.x & 31;
  const int num_ctas = image[kHNumCtas];
  const int num_units = image[kHNumUnits];
  const int num_split = image[kHNumSplit];
  const int num_partials = image[kHNumPartials];
  const ImageOffsets o = image_offsets(num_ctas, num_units, num_split);
  // both images must be the plans the host made for this launch
  if (image[kHMagic] != kMagic || image[kHBatch] != batch || image[kHNumQoHeads] != hq ||
      num_ctas < 0 || num_units < 0 || num_split < 0 || num_partials < 0 ||
      num_partials > max_partials || num_partials + batch > max_partials ||
      o.end > image_words ||
      prefix_image[kHMagic] != kPrefixMagic || prefix_image[kPBatch] != batch ||
      prefix_image[kPNumQoHeads] != hq || prefix_image[kPChunks] != chunks) {
    if (blockIdx.x == 0 && threadIdx.x == 0)
      atomicOr(reinterpret_cast<unsigned int *>(const_cast<int32_t *>(image) + kHStatus),
               PKD_DEVICE_BAD_PLAN);
    return;
  }
  const int32_t *merge_indptr = image + o.merge_indptr;
  const int32_t *merge_req = image + o.merge_req;
  const long long slot_floats = partial_slot_floats(hq, kHeadDim);
  const long long rows = static_cast<long long>(batch) * hq;
  // (suffix slot range) of request b: its partial slots if the suffix plan
  // split it, else slot num_partials + b.  The split requests are listed in
  // increasing order; 128 entries are read per round, all in flight at once.
  auto describe = [&](int b, int &s0, int &s1) {
    int split = -1;
    for (int base = 0; base < num_split && split < 0; base += 128) {
      int r[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int idx = base + 32 * k + lane;
        r[k] = idx < num_split ? merge_req[idx] : INT_MAX;
      }
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const unsigned hit = __ballot_sync(0xffffffffu, r[k] == b);
        if (hit && split < 0) split = base + 32 * k + __ffs(hit) - 1;
      }
      if (__shfl_sync(0xffffffffu, r[3], 31) > b) break;  // past b: not split
    }
    if (split >= 0) {
      s0 = max(0, merge_indptr[split]);
      s1 = min(num_partials, merge_indptr[split + 1]);
    } else {
      s0 = num_partials + b;
      s1 = s0 + 1;
    }
  };
  // The plan images were in place before the kernels of this step started,
  // so the first row is described before the wait; the states are read only
  // after it.  This kernel is a programmatic dependent of the decode kernel,
  // whose threads wait for the prefix kernel before exiting: once the decode
  // kernel is complete, both kernels' states are in place.
  long long row = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  int s0 = 0, s1 = 0;
  if (row < rows) describe(static_cast<int>(row / hq), s0, s1);
  ptx::wait_primary_grid();
  for (bool first = true; row < rows;
       row += (static_cast<long long>(gridDim.x) * blockDim.x) >> 5, first = false) {
    const int b = static_cast<int>(row / hq), h = static_cast<int>(row % hq);
    if (!first) describe(b, s0, s1);
    float m = -INFINITY, ws = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    // four chunk states in flight per round (eight need more than 64
    // registers); the split prefix plan has three chunks
    fold_states<4>(prefix_partials, slot_floats, hq, h, b * chunks, (b + 1) * chunks, 1,
                   lane, m, ws, acc);
    fold_states(partials, slot_floats, hq, h, s0, s1, 1, lane, m, ws, acc);
    write_state<T>(out, lse, b, hq, h, lane, m, ws, acc);
  }
}

// Split-KV merge.  A (split request, query head) row is handled by WPR warps
// (1, 2, 4 or 8, chosen from the average number of partial states per split
// request); each warp folds its share of the row's partial states in one
// online pass (running maximum, rescale when it grows; eight states' loads in
// flight per step: long-context step 625.4 -> 624.5 us, batch-64 86.0 -> 85.3
// us against four), lane l owning d = 4l .. 4l + 3, and the row's warps are
// combined through shared memory by the same rule.
template <typename T, int WPR>
__global__ void __launch_bounds__(kMergeThreads)
    merge_partials_kernel(const int32_t *image, const float *partials,
                          uint16_t *out, float *lse, int hq, int batch,
                          int max_partials, int image_words) {
  constexpr int kRowsPerCta = kMergeWarps / WPR;
  __shared__ float4 red_acc[kMergeWarps][32];
  __shared__ float red_w[kMergeWarps];
  __shared__ float red_m[kMergeWarps];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int slot_in_cta = warp / WPR, sub = warp % WPR;
  const int num_ctas = image[kHNumCtas];
  const int num_units = image[kHNumUnits];
  const int num_split = image[kHNumSplit];
  const int num_partials = image[kHNumPartials];
  const ImageOffsets o = image_offsets(num_ctas, num_units, num_split);
  // only an image the host planned for this launch is trusted (the decode
  // kernel records a mismatch in the status word)
  if (image[kHMagic] != kMagic || image[kHBatch] < 0 || image[kHBatch] > batch ||
      image[kHNumQoHeads] != hq || num_ctas < 0 || num_units < 0 ||
      num_split < 0 || num_partials < 0 || num_partials > max_partials ||
      o.end > image_words)
    return;
  const int32_t *merge_indptr = image + o.merge_indptr;
  const int32_t *merge_req = image + o.merge_req;
  const long long slot_floats = partial_slot_floats(hq, kHeadDim);
  const long long rows = static_cast<long long>(num_split) * hq;
  // (request, head, slot range) of a row, from the plan image alone
  auto describe = [&](long long row, int &b, int &h, int &s0, int &s1) {
    b = -1;
    h = s0 = s1 = 0;
    if (row < rows) {
      const int i = static_cast<int>(row / hq);
      h = static_cast<int>(row % hq);
      b = merge_req[i];
      s0 = max(0, merge_indptr[i]);
      s1 = min(num_partials, merge_indptr[i + 1]);
      if (b < 0 || b >= image[kHBatch]) b = -1;
    }
  };
  // launched as a programmatic dependent of the decode kernel: the plan image
  // was in place before that kernel started, so the first row's description
  // is read before the wait; the partial states are only complete once the
  // decode kernel has finished
  long long first = static_cast<long long>(blockIdx.x) * kRowsPerCta;
  int b, h, s0, s1;
  describe(first + slot_in_cta, b, h, s0, s1);
  ptx::wait_primary_grid();

  for (; first < rows; first += static_cast<long long>(gridDim.x) * kRowsPerCta) {
    if (first != static_cast<long long>(blockIdx.x) * kRowsPerCta)
      describe(first + slot_in_cta, b, h, s0, s1);
    float m = -INFINITY, ws = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    if (b >= 0)
      fold_states<8>(partials, slot_floats, hq, h, s0 + sub, s1, WPR, lane, m, ws, acc);
    if (WPR > 1) {
      red_acc[warp][lane] = acc;
      if (lane == 0) {
        red_m[warp] = m;
        red_w[warp] = ws;
      }
      __syncthreads();
      if (sub == 0 && b >= 0) {
        float mm = m;
#pragma unroll
        for (int w = 1; w < WPR; ++w) mm = fmaxf(mm, red_m[warp + w]);
        const float f0 = m == -INFINITY ? 0.f : expf(m - mm);
        acc.x *= f0;
        acc.y *= f0;
        acc.z *= f0;
        acc.w *= f0;
        ws *= f0;
#pragma unroll
        for (int w = 1; w < WPR; ++w) {
          const float mw = red_m[warp + w];
          const float f = mw == -INFINITY ? 0.f : expf(mw - mm);
          const float4 r = red_acc[warp + w][lane];
          acc.x += f * r.x;
          acc.y += f * r.y;
          acc.z += f * r.z;
          acc.w += f * r.w;
          ws += f * red_w[warp + w];
        }
        m = mm;
      }
    }
    if (sub == 0 && b >= 0) write_state<T>(out, lse, b, hq, h, lane, m, ws, acc);
    if (WPR > 1) __syncthreads();
  }
}

// Pairwise merge of two states, one warp per (n, head) row; lane l handles
// the 8-element chunks l, l + 32, ... of the row.
template <typename V>
struct Vec8;

template <>
struct Vec8<float> {
  static __device__ __forceinline__ void load(const void *p, long long i, float (&x)[8]) {
    const float4 *q = reinterpret_cast<const float4 *>(static_cast<const float *>(p) + i);
    const float4 a = q[0], b = q[1];
    x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
    x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
  }
  static __device__ __forceinline__ void store(void *p, long long i, const float (&x)[8]) {
    float4 *q = reinterpret_cast<float4 *>(static_cast<float *>(p) + i);
    q[0] = make_float4(x[0], x[1], x[2], x[3]);
    q[1] = make_float4(x[4], x[5], x[6], x[7]);
  }
};

template <typename T>
struct Vec8Half {
  static __device__ __forceinline__ void load(const void *p, long long i, float (&x)[8]) {
    const uint4 r = *reinterpret_cast<const uint4 *>(static_cast<const uint16_t *>(p) + i);
    const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float2 f = ptx::unpack2<T>(w[k]);
      x[2 * k] = f.x;
      x[2 * k + 1] = f.y;
    }
  }
  static __device__ __forceinline__ void store(void *p, long long i, const float (&x)[8]) {
    uint4 r;
    r.x = ptx::pack2<T>(x[0], x[1]);
    r.y = ptx::pack2<T>(x[2], x[3]);
    r.z = ptx::pack2<T>(x[4], x[5]);
    r.w = ptx::pack2<T>(x[6], x[7]);
    *reinterpret_cast<uint4 *>(static_cast<uint16_t *>(p) + i) = r;
  }
};

template <>
struct Vec8<__half> : Vec8Half<__half> {};
template <>
struct Vec8<__nv_bfloat16> : Vec8Half<__nv_bfloat16> {};

template <typename V>
__global__ void __launch_bounds__(256)
    merge_states_kernel(const void *v_a, const float *s_a, const void *v_b,
                        const float *s_b, void *v_out, float *s_out,
                        long long rows, int head_dim) {
  const int lane = threadIdx.x & 31;
  const long long warps = static_cast<long long>(gridDim.x) * (blockDim.x >> 5);
  for (long long row = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
       row < rows; row += warps) {
    const float sa = s_a[row], sb = s_b[row];
    __syncwarp();  // every lane has read s before lane 0 may overwrite it
    float wa = 0.f, wb = 0.f, inv = 0.f, s = -INFINITY;
    if (!(sa == -INFINITY && sb == -INFINITY)) {
      const float mx = fmaxf(sa, sb);
      wa = expf(sa - mx);
      wb = expf(sb - mx);
      const float z = wa + wb;
      inv = 1.f / z;
      s = mx + logf(z);
    }
    for (int c = lane; c < head_dim / 8; c += 32) {
      const long long i = row * head_dim + 8 * c;
      float a[8], b[8], r[8];
      Vec8<V>::load(v_a, i, a);
      Vec8<V>::load(v_b, i, b);
#pragma unroll
      for (int k = 0; k < 8; ++k) r[k] = (wa * a[k] + wb * b[k]) * inv;
      Vec8<V>::store(v_out, i, r);
    }
    if (lane == 0) s_out[row] = s;
  }
}

template <typename T, int WPR>
cudaError_t launch_merge_wpr(const MergePartialsArgs &a, cudaLaunchConfig_t *cfg) {
  constexpr int kRowsPerCta = kMergeWarps / WPR;
  const long long rows = static_cast<long long>(a.rows_bound) * a.num_qo_heads;
  const long long want = (rows + kRowsPerCta - 1) / kRowsPerCta;
  cfg->gridDim = dim3(static_cast<unsigned>(want < a.grid ? want : a.grid));
  return cudaLaunchKernelEx(cfg, merge_partials_kernel<T, WPR>, a.image, a.partials,
                            static_cast<uint16_t *>(a.out), a.lse, a.num_qo_heads,
                            a.batch, a.max_partials, a.image_words);
}

template <typename T>
cudaError_t launch_merge_typed(const MergePartialsArgs &a, cudaLaunchConfig_t *cfg) {
  // warps per row from the average number of partial states per split request
  const int avg = a.num_split > 0 ? (a.num_partials + a.num_split - 1) / a.num_split : 1;
  if (avg <= 8) return launch_merge_wpr<T, 1>(a, cfg);
  if (avg <= 16) return launch_merge_wpr<T, 2>(a, cfg);
  if (avg <= 32) return launch_merge_wpr<T, 4>(a, cfg);
  return launch_merge_wpr<T, 8>(a, cfg);
}

}  // namespace

int launch_merge_partials(const MergePartialsArgs &a, void *stream) {
  // programmatic dependent launch: the grid may be scheduled while the decode
  // kernel before it on the stream is still running
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(kMergeThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = static_cast<cudaStream_t>(stream);
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = a.dtype == PKD_BF16 ? launch_merge_typed<__nv_bfloat16>(a, &cfg)
                                      : launch_merge_typed<__half>(a, &cfg);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

int launch_merge_uniform(const float *partials, void *out, float *lse, int batch, int hq,
                         int chunks, int dtype, int grid, void *stream) {
  const long long rows = static_cast<long long>(batch) * hq;
  if (rows == 0) return cudaSuccess;
  const long long want = (rows + kMergeWarps - 1) / kMergeWarps;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(want < grid ? want : grid));
  cfg.blockDim = dim3(kMergeThreads);
  cfg.stream = static_cast<cudaStream_t>(stream);
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  uint16_t *o = static_cast<uint16_t *>(out);
  cudaError_t e = dtype == PKD_BF16
                      ? cudaLaunchKernelEx(&cfg, merge_uniform_kernel<__nv_bfloat16>,
                                           partials, o, lse, batch, hq, chunks)
                      : cudaLaunchKernelEx(&cfg, merge_uniform_kernel<__half>, partials,
                                           o, lse, batch, hq, chunks);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

int launch_cascade_merge(const CascadeMergeArgs &a, void *stream) {
  const long long rows = static_cast<long long>(a.batch) * a.num_qo_heads;
  if (rows == 0) return cudaSuccess;
  // one warp per row: every row is described before the wait on the decode
  // grid, and only its state loads come after it
  const long long want = (rows + kMergeWarps - 1) / kMergeWarps;
  const long long grid = want < 65535 ? want : 65535;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(kMergeThreads);
  cfg.stream = static_cast<cudaStream_t>(stream);
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  uint16_t *o = static_cast<uint16_t *>(a.out);
  cudaError_t e =
      a.dtype == PKD_BF16
          ? cudaLaunchKernelEx(&cfg, cascade_merge_kernel<__nv_bfloat16>, a.image, a.partials,
                               a.prefix_image, a.prefix_partials, o, a.lse, a.num_qo_heads,
                               a.batch, a.chunks, a.max_partials, a.image_words)
          : cudaLaunchKernelEx(&cfg, cascade_merge_kernel<__half>, a.image, a.partials,
                               a.prefix_image, a.prefix_partials, o, a.lse, a.num_qo_heads,
                               a.batch, a.chunks, a.max_partials, a.image_words);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

int launch_merge_states(const void *v_a, const float *s_a, const void *v_b,
                        const float *s_b, void *v_out, float *s_out, int64_t n,
                        int num_heads, int head_dim, int dtype, void *stream) {
  const long long rows = static_cast<long long>(n) * num_heads;
  if (rows == 0) return cudaSuccess;
  const long long want = (rows + 7) / 8;
  const int grid = static_cast<int>(want < 65535 * 16 ? want : 65535 * 16);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  switch (dtype) {
    case PKD_F32:
      merge_states_kernel<float><<<grid, 256, 0, st>>>(v_a, s_a, v_b, s_b, v_out,
                                                        s_out, rows, head_dim);
      break;
    case PKD_BF16:
      merge_states_kernel<__nv_bfloat16><<<grid, 256, 0, st>>>(
          v_a, s_a, v_b, s_b, v_out, s_out, rows, head_dim);
      break;
    default:
      merge_states_kernel<__half><<<grid, 256, 0, st>>>(v_a, s_a, v_b, s_b, v_out,
                                                         s_out, rows, head_dim);
  }
  return cudaGetLastError();
}

}  // namespace pkd

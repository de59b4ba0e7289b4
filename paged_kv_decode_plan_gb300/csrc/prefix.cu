// Shared-prefix attention: the queries of B requests against one KV prefix
// they all share, stored once.
//
// "FlashInfer" (aiwiki.ai/wiki/flashinfer), "Attention states": a serving
// system can evaluate a shared prefix separately from the requests' own
// suffixes and merge the partial states; "Welcome to FlashInfer's
// documentation!", flashinfer.cascade "Cascade Attention".
//
// Per key/value head h the prefix attention is one dense problem: the
// B * g query rows (request b, group head j) against the prefix tokens.  The
// grid is (head, 128-row tile, KV chunk); a CTA has one loader warp (TMA
// tiled loads: 64-token stages of head h's K and V, four 16-token boxes per
// tensor and d-half, 128-byte swizzle) and eight consumer warps of 16 query
// rows each:
//     S = Q K^T      (mma.sync m16n8k16, query rows as M, fp32 accumulate)
//     online softmax over tokens (raw maxima, scale inside one fma, -inf
//     clamp, reference moved only when the maximum grows by > 2^8)
//     O += P V       (P from the S accumulators; bf16 P as hi + lo)
// Each CTA writes fp32 partial states (o / l, lse) of its rows for its chunk
// into slot b * chunks + c of the float workspace; a merge kernel folds the
// chunks of every (request, head) row.  The prefix is read from HBM once per
// (head, row tile, chunk); the row tiles of a head re-read it from L2.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstring>
#include <type_traits>

#include "kernel_common.cuh"
#include "pkd_internal.h"
#include "ptx.cuh"

namespace pkd {
namespace {

constexpr int kPWarps = 8;                   // consumer warps, 16 rows each
constexpr int kPRows = 16 * kPWarps;         // query rows per CTA
constexpr int kPTile = 64;                   // tokens per stage
constexpr int kPSub = kPTile / kTile;        // 16-token boxes per stage
constexpr int kPTensorBytes = kPSub * 2 * kHalfBytes;  // K (or V) of one stage
constexpr int kPStageBytes = 2 * kPTensorBytes;
constexpr int kPStages = 4;
constexpr int kPSmem = 1024 + kPStages * kPStageBytes + 16 * kPStages + 16;

struct PrefixParams {
  const uint16_t *q;
  const int32_t *image;   // prefix plan image: header + page ids
  int32_t *status;        // the image's status word
  float *partials;
  float scale_log2;
  long long num_pages;
  int batch, hq, hkv, group, page_size;
  int length, chunks, chunk_tiles, row_tiles;
  int hnd;                // page tensors are HND
};

__device__ __forceinline__ void give_up(const PrefixParams &p, volatile int *abort) {
  *abort = 1;
  atomicOr(reinterpret_cast<unsigned int *>(p.status), PKD_DEVICE_TIMEOUT);
}

__device__ void load_prefix(const PrefixParams &p, const CUtensorMap *map_k,
                            const CUtensorMap *map_v, int h, int t_begin, int t_end,
                            uint8_t *stages, uint32_t full0, uint32_t empty0,
                            volatile int *abort) {
  const int lane = threadIdx.x & 31;
  const int32_t *pages = p.image + kHeaderWords;
  const uint32_t stage0 = ptx::smem_u32(stages);
  int it = 0;
  for (int t = t_begin; t < t_end; ++t, ++it) {
    const int s = it % kPStages;
    if (!wait_phase(empty0 + 8 * s, ((it / kPStages) & 1) ^ 1, abort)) {
      if (lane == 0) give_up(p, abort);
      break;
    }
    const int tok0 = t * kPTile;
    const int nsub = min(kPSub, (p.length - tok0 + kTile - 1) / kTile);
    if (lane == 0) ptx::mbar_arrive_expect_tx(full0 + 8 * s, nsub * 4 * kHalfBytes);
    __syncwarp();
    if (lane < 4 * nsub) {
      const int sub = lane >> 2, tensor = (lane >> 1) & 1, half = lane & 1;
      const int tok = tok0 + sub * kTile;
      const int pi = tok / p.page_size;
      int page = __ldg(pages + pi);
      if (static_cast<unsigned long long>(page) >=
          static_cast<unsigned long long>(p.num_pages)) {
        atomicOr(reinterpret_cast<unsigned int *>(p.status), PKD_DEVICE_BAD_PAGE);
        page = 0;
      }
      const uint32_t dst = stage0 + s * kPStageBytes + tensor * kPTensorBytes +
                           sub * 2 * kHalfBytes + half * kHalfBytes;
      const int slot = tok - pi * p.page_size;
      if (p.hnd)
        ptx::tma_load_4d(dst, tensor ? map_v : map_k, half * 64, slot, h, page,
                         full0 + 8 * s);
      else
        ptx::tma_load_3d(dst, tensor ? map_v : map_k, half * 64, h,
                         page * p.page_size + slot, full0 + 8 * s);
    }
  }
  for (int j = max(0, it - kPStages); j < it; ++j)
    wait_phase(full0 + 8 * (j % kPStages), (j / kPStages) & 1, abort, true);
}

template <typename T>
__device__ void consume_prefix(const PrefixParams &p, int h, int rt, int c, int t_begin,
                               int t_end, const uint8_t *stages, uint32_t full0,
                               uint32_t empty0, volatile int *abort) {
  constexpr bool kSplitP = std::is_same<T, __nv_bfloat16>::value;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gid = lane >> 2, tq = lane & 3;
  const int rows = p.batch * p.group;
  const float cs = p.scale_log2;
  const uint32_t stage0 = ptx::smem_u32(stages);
  // ldmatrix addressing within a 16-token box (K non-transposed as the B
  // operand of Q K^T, V transposed as the B operand of P V)
  const int k_row = (lane & 7) + ((lane >> 4) << 3);
  const int k_hi = (lane >> 3) & 1;
  const int v_row = (lane & 7) + (((lane >> 3) & 1) << 3);
  const int v_hi = lane >> 4;

  // query rows gid and gid + 8 of this warp: row R -> (request R / g, head j)
  int row_id[2];
  uint32_t qa[8][4];
  {
    const uint16_t *qr[2];
    bool ok[2];
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      row_id[r] = rt * kPRows + warp * 16 + gid + 8 * r;
      ok[r] = row_id[r] < rows;
      const int rr = ok[r] ? row_id[r] : 0;
      const int b = rr / p.group, j = rr % p.group;
      qr[r] = p.q + (static_cast<long long>(b) * p.hq + h * p.group + j) * kHeadDim;
    }
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
      const int d = 16 * kk + 2 * tq;
      qa[kk][0] = ok[0] ? __ldg(reinterpret_cast<const uint32_t *>(qr[0] + d)) : 0u;
      qa[kk][1] = ok[1] ? __ldg(reinterpret_cast<const uint32_t *>(qr[1] + d)) : 0u;
      qa[kk][2] = ok[0] ? __ldg(reinterpret_cast<const uint32_t *>(qr[0] + d + 8)) : 0u;
      qa[kk][3] = ok[1] ? __ldg(reinterpret_cast<const uint32_t *>(qr[1] + d + 8)) : 0u;
    }
  }

  float ref[2] = {-INFINITY, -INFINITY};  // scaled reference per row
  float l[2] = {0.f, 0.f};
  float acc[16][4];
#pragma unroll
  for (int j = 0; j < 16; ++j) acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.f;

  int it = 0;
  for (int t = t_begin; t < t_end; ++t, ++it) {
    const int s = it % kPStages;
    if (!wait_phase(full0 + 8 * s, (it / kPStages) & 1, abort)) {
      if (lane == 0) give_up(p, abort);
      return;
    }
    const uint32_t kb = stage0 + s * kPStageBytes;
    const uint32_t vb = kb + kPTensorBytes;
    const int valid = min(kPTile, p.length - t * kPTile);

    // S = Q K^T over 64 tokens: n-tiles of 8 tokens, box = n-tile pair
    float sc[8][4];
#pragma unroll
    for (int n = 0; n < 8; ++n) sc[n][0] = sc[n][1] = sc[n][2] = sc[n][3] = 0.f;
#pragma unroll
    for (int box = 0; box < kPSub; ++box) {
      const uint32_t kbox = kb + box * 2 * kHalfBytes;
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        uint32_t b0, b1, b2, b3;
        ptx::ldmatrix_x4(kbox + tile_offset(k_row, 2 * kk + k_hi), b0, b1, b2, b3);
        ptx::mma_16816<T>(sc[2 * box], qa[kk], b0, b1);
        ptx::mma_16816<T>(sc[2 * box + 1], qa[kk], b2, b3);
      }
    }

    // online softmax per row (rows gid and gid + 8; columns are tokens)
    float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
    for (int n = 0; n < 8; ++n)
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int tok = n * 8 + 2 * tq + (i & 1);
        if (tok >= valid) sc[n][i] = -INFINITY;
        mx[i >> 1] = fmaxf(mx[i >> 1], sc[n][i]);
      }
    bool need = false;
    float cand[2];
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 1));
      mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 2));
      cand[r] = mx[r] * cs;
      need |= cand[r] > ref[r] + kLazy;
    }
    if (__any_sync(0xffffffffu, need)) {
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        float alpha = 1.f;
        if (cand[r] > ref[r] + kLazy) {
          alpha = exp2f(ref[r] - cand[r]);  // ref = -inf gives 0
          ref[r] = cand[r];
        }
        l[r] *= alpha;
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          acc[j][2 * r] *= alpha;
          acc[j][2 * r + 1] *= alpha;
        }
      }
    }
    const float r0 = ref[0] == -INFINITY ? 0.f : ref[0];  // clamp
    const float r1 = ref[1] == -INFINITY ? 0.f : ref[1];

    // per 16-token box: P as the A operand (from two n-tiles of S), then
    // O += P V; V rows past the prefix end may hold anything: zero them in
    // the B fragments (tokens 2tq, 2tq+1 and 2tq+8, 2tq+9 of the box)
#pragma unroll
    for (int box = 0; box < kPSub; ++box) {
      uint32_t pa[4], pl[4];
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        const float *sv = sc[2 * box + half];
        const float e0 = exp2f(fmaf(sv[0], cs, -r0));
        const float e1 = exp2f(fmaf(sv[1], cs, -r0));
        const float e2 = exp2f(fmaf(sv[2], cs, -r1));
        const float e3 = exp2f(fmaf(sv[3], cs, -r1));
        const uint32_t h01 = ptx::pack2<T>(e0, e1), h23 = ptx::pack2<T>(e2, e3);
        const float2 b01 = ptx::unpack2<T>(h01), b23 = ptx::unpack2<T>(h23);
        pa[2 * half] = h01;
        pa[2 * half + 1] = h23;
        if (kSplitP) {
          const uint32_t l01 = ptx::pack2<T>(e0 - b01.x, e1 - b01.y);
          const uint32_t l23 = ptx::pack2<T>(e2 - b23.x, e3 - b23.y);
          const float2 c01 = ptx::unpack2<T>(l01), c23 = ptx::unpack2<T>(l23);
          pl[2 * half] = l01;
          pl[2 * half + 1] = l23;
          l[0] += (b01.x + c01.x) + (b01.y + c01.y);
          l[1] += (b23.x + c23.x) + (b23.y + c23.y);
        } else {
          pl[2 * half] = pl[2 * half + 1] = 0u;
          l[0] += b01.x + b01.y;
          l[1] += b23.x + b23.y;
        }
      }
      const int tv = valid - box * kTile;
      uint32_t m01 = 0xffffffffu, m89 = 0xffffffffu;
      if (tv < kTile) {
        m01 = (2 * tq < tv ? 0x0000ffffu : 0u) | (2 * tq + 1 < tv ? 0xffff0000u : 0u);
        m89 = (2 * tq + 8 < tv ? 0x0000ffffu : 0u) | (2 * tq + 9 < tv ? 0xffff0000u : 0u);
      }
      const uint32_t vbox = vb + box * 2 * kHalfBytes;
#pragma unroll
      for (int jj = 0; jj < 16; jj += 2) {
        uint32_t b0, b1, b2, b3;
        ptx::ldmatrix_x4_trans(vbox + tile_offset(v_row, jj + v_hi), b0, b1, b2, b3);
        b0 &= m01;
        b1 &= m89;
        b2 &= m01;
        b3 &= m89;
        ptx::mma_16816<T>(acc[jj], pa, b0, b1);
        ptx::mma_16816<T>(acc[jj + 1], pa, b2, b3);
        if (kSplitP) {
          ptx::mma_16816<T>(acc[jj], pl, b0, b1);
          ptx::mma_16816<T>(acc[jj + 1], pl, b2, b3);
        }
      }
    }
    __syncwarp();
    if (lane == 0) ptx::mbar_arrive(empty0 + 8 * s);
  }

  // row totals and the chunk's partial state
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    l[r] += __shfl_xor_sync(0xffffffffu, l[r], 1);
    l[r] += __shfl_xor_sync(0xffffffffu, l[r], 2);
  }
  const long long slot_floats = partial_slot_floats(p.hq, kHeadDim);
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    if (row_id[r] >= rows) continue;
    const int b = row_id[r] / p.group, head = h * p.group + row_id[r] % p.group;
    float *base = p.partials + (static_cast<long long>(b) * p.chunks + c) * slot_floats;
    const float inv = l[r] > 0.f ? 1.f / l[r] : 0.f;
    float *o = base + head * kHeadDim;
#pragma unroll
    for (int j = 0; j < 16; ++j)
      *reinterpret_cast<float2 *>(o + 8 * j + 2 * tq) =
          make_float2(acc[j][2 * r] * inv, acc[j][2 * r + 1] * inv);
    if (tq == 0)
      base[p.hq * kHeadDim + head] =
          l[r] > 0.f ? (ref[r] + log2f(l[r])) * kLn2 : -INFINITY;
  }
}

template <typename T>
__global__ void __launch_bounds__(32 * (kPWarps + 1), 1)
    shared_prefix_kernel(const __grid_constant__ PrefixParams p,
                         const __grid_constant__ CUtensorMap map_k,
                         const __grid_constant__ CUtensorMap map_v) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *stages = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t *bars = reinterpret_cast<uint64_t *>(stages + kPStages * kPStageBytes);
  volatile int *abort = reinterpret_cast<volatile int *>(bars + 2 * kPStages);
  const uint32_t full0 = ptx::smem_u32(bars);
  const uint32_t empty0 = full0 + 8 * kPStages;

  // the image must be the prefix plan the host made for this launch
  const int32_t *img = p.image;
  if (img[kHMagic] != kPrefixMagic || img[kPBatch] != p.batch ||
      img[kPNumQoHeads] != p.hq || img[kPNumKvHeads] != p.hkv ||
      img[kPPageSize] != p.page_size || img[kPLength] != p.length ||
      img[kPChunks] != p.chunks || img[kPChunkTiles] != p.chunk_tiles ||
      img[kPRowTiles] != p.row_tiles ||
      img[kPNumPages] * static_cast<long long>(p.page_size) < p.length) {
    if (threadIdx.x == 0 && blockIdx.x == 0)
      atomicOr(reinterpret_cast<unsigned int *>(p.status), PKD_DEVICE_BAD_PLAN);
    return;
  }
  const int c = blockIdx.x % p.chunks;
  const int rt = (blockIdx.x / p.chunks) % p.row_tiles;
  const int h = blockIdx.x / (p.chunks * p.row_tiles);
  const int total_tiles = (p.length + kPTile - 1) / kPTile;
  const int t_begin = min(total_tiles, c * p.chunk_tiles);
  const int t_end = min(total_tiles, t_begin + p.chunk_tiles);
  ptx::launch_dependents();

  if (threadIdx.x == 0) {
    for (int s = 0; s < kPStages; ++s) {
      ptx::mbar_init(full0 + 8 * s, 1);
      ptx::mbar_init(empty0 + 8 * s, kPWarps);
    }
    *abort = 0;
    ptx::fence_mbar_init();
    ptx::fence_proxy_async();
  }
  __syncthreads();
  if (threadIdx.x >= 32 * kPWarps)
    load_prefix(p, &map_k, &map_v, h, t_begin, t_end, stages, full0, empty0, abort);
  else
    consume_prefix<T>(p, h, rt, c, t_begin, t_end, stages, full0, empty0, abort);
}

}  // namespace

int prefix_tile_tokens() { return kPTile; }
int prefix_tile_rows() { return kPRows; }

int launch_shared_prefix(const PrefixArgs &a, void *stream) {
  alignas(64) CUtensorMap mk;
  alignas(64) CUtensorMap mv;
  if (!page_tensor_maps(&mk, &mv, a.k_pages, a.v_pages, a.num_pages, a.page_size,
                        a.num_kv_heads, a.layout))
    return cudaErrorNotSupported;
  PrefixParams p;
  p.q = static_cast<const uint16_t *>(a.q);
  p.image = a.image;
  p.status = a.image + kHStatus;
  p.partials = a.partials;
  p.scale_log2 = a.sm_scale_log2;
  p.num_pages = a.num_pages;
  p.batch = a.batch;
  p.hq = a.num_qo_heads;
  p.hkv = a.num_kv_heads;
  p.group = a.num_qo_heads / a.num_kv_heads;
  p.page_size = a.page_size;
  p.length = a.length;
  p.chunks = a.chunks;
  p.chunk_tiles = a.chunk_tiles;
  p.row_tiles = a.row_tiles;
  p.hnd = a.layout == PKD_LAYOUT_HND;
  const int grid = a.num_kv_heads * a.row_tiles * a.chunks;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  if (a.dtype == PKD_BF16) {
    e = cudaFuncSetAttribute(shared_prefix_kernel<__nv_bfloat16>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, kPSmem);
    if (e != cudaSuccess) return e;
    shared_prefix_kernel<__nv_bfloat16><<<grid, 32 * (kPWarps + 1), kPSmem, st>>>(p, mk, mv);
  } else {
    e = cudaFuncSetAttribute(shared_prefix_kernel<__half>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, kPSmem);
    if (e != cudaSuccess) return e;
    shared_prefix_kernel<__half><<<grid, 32 * (kPWarps + 1), kPSmem, st>>>(p, mk, mv);
  }
  return cudaGetLastError();
}

}  // namespace pkd

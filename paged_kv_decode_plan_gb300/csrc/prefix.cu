// Shared-prefix attention: the queries of B requests against one KV prefix
// they all share, stored once.
//
// "FlashInfer" (aiwiki.ai/wiki/flashinfer), "Attention states": a serving
// system can evaluate a shared prefix separately from the requests' own
// suffixes and merge the partial states; "Welcome to FlashInfer's
// documentation!", flashinfer.cascade "Cascade Attention".
//
// Per key/value head h the prefix attention is one dense problem: the
// B * g query rows (request b, group head j) against the prefix tokens, so it
// runs on the 5th-generation tensor cores (tcgen05, accumulators in tensor
// memory).  The grid is (head, 256-row tile, KV chunk).  A CTA holds two
// 128-row query tiles that share every K/V stage (loaded once for 256 rows):
//   warps 0-3  softmax of query tile 0, thread r owns row r = tensor lane r
//   warps 4-7  softmax of query tile 1
//   warp 8     tensor-memory allocation; one thread issues tile 0's MMAs
//   warp 9     one thread issues tile 1's MMAs (a thread can issue a
//              tcgen05.mma only every ~120 cycles, so two issuers keep the
//              tensor pipe fed with M 128 x N 128 MMAs)
//   warps 10, 11  loaders of K and of V: TMA tiled loads of head h, 128-token
//              stages, 16-token boxes, 128-byte swizzle; the prefix's ragged
//              last box is copied with plain loads, zeros past the end.  K and
//              V have their own full / empty barriers: K of a stage is free
//              once both S MMAs have read it, well before P V frees V.
// Per query tile q and 128-token tile i:
//   S    = Q_q K_i^T             M 128, N 128, K 128 (A, B from shared memory)
//   P    = exp2(S * c - ref)     softmax threads; P (f16 / bf16 pairs) is
//                                stored over the S columns it came from
//   O   += P V_i                 M 128, N 128, K 128 (A = P from tensor memory)
// bf16 P is split as hi + lo (two MMAs into the same accumulators).  The row
// sum l is kept in fp32 registers.  The running reference moves only when a
// row maximum grows by > 2^8; then O and l are rescaled.  S_q of tile i + 1
// reuses P_q's columns, so the MMA thread issues it once P_q V_i has
// completed; the two query tiles ping-pong, so while one warpgroup computes
// exponentials the tensor core runs the other's MMAs.  N = 128 per MMA keeps
// the tensor pipe's shared-memory reads per flop at the level it sustains.
// Each CTA writes fp32 partial states (o / l, lse) of its rows for its chunk
// into slot b * chunks + c of the float workspace; a merge kernel folds the
// chunks.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstring>
#include <type_traits>

#include "kernel_common.cuh"
#include "pkd_internal.h"
#include "ptx.cuh"
#include "tcgen05.cuh"

namespace pkd {
namespace {

constexpr int kPQRows = 128;                       // rows per query tile (MMA M)
constexpr int kPRows = 2 * kPQRows;                // query rows per CTA
constexpr int kPTile = 128;                        // tokens per stage (MMA N of S)
constexpr int kPHalfRegion = kPTile * 128;         // one 64-column block: 128 rows x 128 B
constexpr int kPTensorBytes = 2 * kPHalfRegion;    // K (or V) of one stage
constexpr int kPOffV = kPTensorBytes;              // V after K in a stage
constexpr int kPStageBytes = 2 * kPTensorBytes;
constexpr int kPStages = 2;
constexpr int kPQBytes = kPQRows * 256;            // [d-half][row][128 B]
constexpr int kSoftmaxThreads = 128;
constexpr int kMmaWarp = 8, kLoadWarp = 10;  // warps 8, 9 issue MMAs; 10, 11 load
constexpr int kPThreads = 32 * 12;
constexpr uint32_t kTmemCols = 512;

// Tensor-memory columns of query tile q: S (128), then O (128).  P of token
// half t (tokens 64 t .. 64 t + 63) is stored over S columns [64 t, 64 t + 64):
// hi pairs in the first 32, bf16 lo pairs in the next 32.
__host__ __device__ constexpr uint32_t col_s(int q) { return 256u * q; }
__host__ __device__ constexpr uint32_t col_o(int q) { return 256u * q + kPTile; }
static_assert(col_o(1) + kHeadDim <= kTmemCols, "tensor-memory budget");

constexpr int kOffQ = kPStages * kPStageBytes;
constexpr int kOffBars = kOffQ + 2 * kPQBytes;
// full[tensor][S], empty[tensor][S], then per query tile s_full, p_full,
// p_free, q_full, drain, and the ping-pong acknowledgement
constexpr int kNumBars = 4 * kPStages + 11;
constexpr int kOffMisc = kOffBars + 8 * kNumBars;
constexpr int kPSmem = 1024 + kOffMisc + 16;
static_assert(kPSmem <= 227 * 1024, "shared memory budget");

struct PrefixParams {
  const uint16_t *q, *k, *v;
  const int32_t *image;   // prefix plan image: header + page ids
  int32_t *status;        // the image's status word
  float *partials;
  float scale_log2;
  long long num_pages;
  int batch, hq, hkv, group, page_size;
  int length, chunks, chunk_tiles, row_tiles;
  int hnd;                // page tensors are HND
  int q_tma;              // queries arrive by TMA (128 % group == 0)
};

struct Bars {
  uint32_t base;
  // tensor 0 = K, 1 = V
  __device__ uint32_t full(int t, int s) const { return base + 8 * (t * kPStages + s); }
  __device__ uint32_t empty(int t, int s) const { return base + 8 * ((2 + t) * kPStages + s); }
  __device__ uint32_t s_full(int q) const { return base + 8 * (4 * kPStages + q); }
  __device__ uint32_t p_full(int q) const { return base + 8 * (4 * kPStages + 2 + q); }
  __device__ uint32_t p_free(int q) const { return base + 8 * (4 * kPStages + 4 + q); }
  __device__ uint32_t q_full(int q) const { return base + 8 * (4 * kPStages + 6 + q); }
  __device__ uint32_t drain(int q) const { return base + 8 * (4 * kPStages + 8 + q); }
  __device__ uint32_t ack() const { return base + 8 * (4 * kPStages + 10); }
};

__device__ __forceinline__ void give_up(const PrefixParams &p, volatile int *abort) {
  *abort = 1;
  atomicOr(reinterpret_cast<unsigned int *>(p.status), PKD_DEVICE_TIMEOUT);
}

// Bounded mbarrier wait whose outcome is the same on every lane of the warp,
// so warp-collective tensor-memory instructions after it are never divergent.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int *abort) {
  for (long long i = 0; i < kWaitPolls; ++i) {
    const bool ok = ptx::mbar_try_wait(bar, parity);
    if (__all_sync(0xffffffffu, ok)) return true;
    if ((i & 63) == 63 && __any_sync(0xffffffffu, *abort != 0)) return false;
  }
  return false;
}

__device__ __forceinline__ long long row_elem(const PrefixParams &p, long long page, int slot,
                                              int h) {
  return p.hnd ? ((page * p.hkv + h) * p.page_size + slot) * kHeadDim
               : ((page * p.page_size + slot) * p.hkv + h) * kHeadDim;
}

__device__ __forceinline__ long long checked_page(const PrefixParams &p, const int32_t *pages,
                                                  int pi) {
  long long page = __ldg(pages + pi);
  if (static_cast<unsigned long long>(page) >= static_cast<unsigned long long>(p.num_pages)) {
    atomicOr(reinterpret_cast<unsigned int *>(p.status), PKD_DEVICE_BAD_PAGE);
    page = 0;
  }
  return page;
}

// Warp kLoadWarp + tensor: fills K (tensor 0) or V (tensor 1) of stage
// it % S with tokens [128 t, 128 t + 128) of head h.
__device__ void load_prefix(const PrefixParams &p, const CUtensorMap *map, int tensor, int h,
                            int t_begin, int n, uint8_t *stages, const Bars &bars,
                            volatile int *abort) {
  const int lane = threadIdx.x & 31;
  const int32_t *pages = p.image + kHeaderWords;
  const uint16_t *src_pages = tensor ? p.v : p.k;
  const uint32_t stage0 = ptx::smem_u32(stages) + tensor * kPOffV;
  if (lane == 0) asm volatile("prefetch.tensormap [%0];\n" ::"l"(map) : "memory");
  int it = 0;
  for (; it < n; ++it) {
    const int s = it % kPStages;
    if (!warp_wait(bars.empty(tensor, s), ((it / kPStages) & 1) ^ 1, abort)) {
      if (lane == 0) give_up(p, abort);
      break;
    }
    const int tok0 = (t_begin + it) * kPTile;
    const int valid = min(kPTile, p.length - tok0);
    const int nfull = valid / kTile;
    uint8_t *dst_tile = stages + s * kPStageBytes + tensor * kPOffV;
    if (valid < kPTile) {
      // rows [16 nfull, 128): plain copies up to the prefix end, zeros after
      const int first = nfull * kTile;
      const int items = (kPTile - first) * 16;  // rows x 16-byte chunks
      for (int idx = lane; idx < items; idx += 32) {
        const int row = first + (idx >> 4), c16 = idx & 15;
        uint4 val = make_uint4(0u, 0u, 0u, 0u);
        if (row < valid) {
          const int tok = tok0 + row;
          const int pi = tok / p.page_size;
          const long long page = checked_page(p, pages, pi);
          const uint16_t *src =
              src_pages + row_elem(p, page, tok - pi * p.page_size, h) + 8 * c16;
          val = __ldg(reinterpret_cast<const uint4 *>(src));
        }
        *reinterpret_cast<uint4 *>(dst_tile + (c16 >> 3) * kPHalfRegion + row * 128 +
                                   (((c16 & 7) ^ (row & 7)) << 4)) = val;
      }
      ptx::fence_proxy_async();
    }
    __syncwarp();
    if (lane == 0) ptx::mbar_arrive_expect_tx(bars.full(tensor, s), nfull * 2 * kHalfBytes);
    __syncwarp();
    if (lane < 2 * nfull) {
      const int sub = lane >> 1, half = lane & 1;
      const int tok = tok0 + sub * kTile;
      const int pi = tok / p.page_size;
      const int page = static_cast<int>(checked_page(p, pages, pi));
      const uint32_t dst = stage0 + s * kPStageBytes + half * kPHalfRegion + sub * kHalfBytes;
      const int slot = tok - pi * p.page_size;
      if (p.hnd)
        ptx::tma_load_4d(dst, map, half * 64, slot, h, page, bars.full(tensor, s));
      else
        ptx::tma_load_3d(dst, map, half * 64, h, page * p.page_size + slot,
                         bars.full(tensor, s));
    }
  }
  // no copy may still be in flight when the CTA exits
  for (int j = max(0, it - kPStages); j < it; ++j)
    wait_phase(bars.full(tensor, j % kPStages), (j / kPStages) & 1, abort, true);
  __syncwarp();
}

// Ping-pong: tile 1's S of KV tile i is issued only after tile 0's softmax of
// tile i has finished (so the two softmaxes alternate with the other tile's
// MMAs); its issuer acknowledges each such wait, and tile 0's S of tile i + 1
// waits for that acknowledgement, so neither side can pass a barrier phase
// the other has not observed yet.
template <typename T>
__device__ void issue_mmas(const PrefixParams &p, int n, int q, int nq, uint8_t *smem,
                           uint32_t tmem, const Bars &bars, volatile int *abort) {
  constexpr bool kSplit = std::is_same<T, __nv_bfloat16>::value;
  constexpr uint32_t kIdescQK = tc::idesc_f16(kSplit, kPQRows, kPTile, false);
  constexpr uint32_t kIdescPV = tc::idesc_f16(kSplit, kPQRows, kHeadDim, true);
  const uint32_t base = ptx::smem_u32(smem);
  // Descriptors are built once; a k-step adds its byte offset / 16 to the
  // start-address field (no carry: shared addresses stay below 256 KB).
  const uint64_t q_desc = tc::smem_desc_sw128(base + kOffQ + q * kPQBytes, 16, 1024);
  const uint64_t k_desc = tc::smem_desc_sw128(base, 16, 1024);
  const uint64_t v_desc = tc::smem_desc_sw128(base + kPOffV, kPHalfRegion, 1024);
  const uint32_t t_s = tmem + col_s(q), t_o = tmem + col_o(q);

  // S_q = Q_q K_i^T: eight K = 16 steps over the head dim
  auto issue_qk = [&](int i) -> bool {
    if (q == 1) {
      if (!wait_phase(bars.p_full(0), i & 1, abort)) return false;
      ptx::mbar_arrive(bars.ack());
    } else if (nq == 2 && i > 0) {
      if (!wait_phase(bars.ack(), (i - 1) & 1, abort)) return false;
    }
    if (!wait_phase(bars.full(0, i % kPStages), (i / kPStages) & 1, abort)) return false;
    tc::fence_after_sync();
    const uint64_t kd = k_desc + (((i % kPStages) * kPStageBytes) >> 4);
#pragma unroll
    for (int kk = 0; kk < kHeadDim / 16; ++kk) {
      const uint32_t off = ((kk >> 2) * kPQRows * 128 + (kk & 3) * 32) >> 4;
      const uint32_t koff = ((kk >> 2) * kPHalfRegion + (kk & 3) * 32) >> 4;
      tc::mma_f16(t_s, q_desc + off, kd + koff, kIdescQK, kk > 0);
    }
    tc::commit(bars.s_full(q));
    tc::commit(bars.empty(0, i % kPStages));  // one arrival per query tile
    return true;
  };

  bool ok = wait_phase(bars.q_full(q), 0, abort);
  bool issued = false;
  if (ok) {
    issued = true;
    ok = issue_qk(0);
  }
  for (int i = 0; ok && i < n; ++i) {
    // the softmax has read S_q and written P_q of tile i
    if (!(ok = wait_phase(bars.p_full(q), i & 1, abort))) break;
    if (!(ok = wait_phase(bars.full(1, i % kPStages), (i / kPStages) & 1, abort))) break;
    tc::fence_after_sync();
    // O += P V: k-steps of 16 tokens; V rows 16 j .. 16 j + 15 are two 8-row
    // groups (SBO 1024), V's d-halves 16 KB apart (LBO); P of those tokens
    // sits in S columns 64 (j / 4) + 8 (j % 4) (+ 32 for the lo copy)
    const uint64_t vd = v_desc + (((i % kPStages) * kPStageBytes) >> 4);
#pragma unroll
    for (int j = 0; j < kPTile / 16; ++j) {
      const uint32_t a = t_s + 64 * (j >> 2) + 8 * (j & 3);
      tc::mma_f16_tmem_a(t_o, a, vd + ((j * 2048) >> 4), kIdescPV, i > 0 || j > 0);
      if (kSplit) tc::mma_f16_tmem_a(t_o, a + 32, vd + ((j * 2048) >> 4), kIdescPV, true);
    }
    tc::commit(bars.p_free(q));
    tc::commit(bars.empty(1, i % kPStages));  // one arrival per query tile
    if (i + 1 < n) {
      // S_q of tile i + 1 overwrites P_q: only once P_q V_i has completed
      if (!(ok = wait_phase(bars.p_free(q), i & 1, abort))) break;
      if (!(ok = issue_qk(i + 1))) break;
    }
  }
  if (!ok) give_up(p, abort);
  if (issued) {
    // every MMA of this thread completes before tensor memory is released
    tc::commit(bars.drain(q));
    wait_phase(bars.drain(q), 0, abort, true);
  }
}

// One 128-token tile of one query row (warp-collective): row maximum, lazy
// reference move (rescaling O and l when it moves and O holds earlier tiles),
// P stored over S, row sum.  kFull: every token of the tile is in the prefix.
template <typename T, bool kFull>
__device__ __forceinline__ void softmax_tile(uint32_t t_s, uint32_t t_o, int valid, float cs,
                                             bool rescale_o, float &ref, float &l) {
  constexpr bool kSplit = std::is_same<T, __nv_bfloat16>::value;
  float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    float s[64];
    tc::ld64(t_s + 64 * half, s);
#pragma unroll
    for (int j = 0; j < 64; ++j)
      if (kFull || 64 * half + j < valid) m4[j & 3] = fmaxf(m4[j & 3], s[j]);
  }
  const float cand = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3])) * cs;
  const bool need = cand > ref + kLazy;
  if (__any_sync(0xffffffffu, need)) {
    float alpha = 1.f;
    if (need) {
      alpha = ptx::ex2(ref - cand);  // ref = -inf gives 0
      ref = cand;
    }
    l *= alpha;
    if (rescale_o) {
#pragma unroll 1
      for (int cc = 0; cc < kHeadDim / 16; ++cc) {
        float v[16];
        tc::ld16(t_o + 16 * cc, v);
#pragma unroll
        for (int e = 0; e < 16; ++e) v[e] *= alpha;
        tc::st16(t_o + 16 * cc, v);
      }
    }
  }
  const float rc = ref == -INFINITY ? 0.f : ref;  // clamp
  float lsum[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 1
  for (int half = 0; half < 2; ++half) {
    // P of this token half replaces the S values it was computed from
    // (the whole half is in registers before any of its columns is written)
    float s[64];
    tc::ld64(t_s + 64 * half, s);
#pragma unroll
    for (int chunk = 0; chunk < 2; ++chunk) {
      float hi[16], lo[16];  // packed pairs, carried as float bit patterns
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const int k = 32 * chunk + 2 * j;
        const int t = 64 * half + k;
        const float e0 = kFull || t < valid ? ptx::ex2(fmaf(s[k], cs, -rc)) : 0.f;
        const float e1 = kFull || t + 1 < valid ? ptx::ex2(fmaf(s[k + 1], cs, -rc)) : 0.f;
        const uint32_t h2 = ptx::pack2<T>(e0, e1);
        hi[j] = __uint_as_float(h2);
        if (kSplit) {
          const float2 f = ptx::unpack2<T>(h2);
          lo[j] = __uint_as_float(ptx::pack2<T>(e0 - f.x, e1 - f.y));
        }
        lsum[j & 3] += e0 + e1;
      }
      tc::st16(t_s + 64 * half + 16 * chunk, hi);
      if (kSplit) tc::st16(t_s + 64 * half + 32 + 16 * chunk, lo);
    }
  }
  l += (lsum[0] + lsum[1]) + (lsum[2] + lsum[3]);
}

// Warps 4q .. 4q + 3: row r of query tile q (zeros past the last row) into
// shared memory as [d-half][row][128 B], 128-byte swizzled.
__device__ void load_q(const PrefixParams &p, int q, int h, int rt, uint8_t *smem,
                       const Bars &bars) {
  const int r = threadIdx.x & (kSoftmaxThreads - 1);
  const int row_id = rt * kPRows + q * kPQRows + r;
  const bool live = row_id < p.batch * p.group;
  const int b = live ? row_id / p.group : 0;
  const int head = h * p.group + (live ? row_id % p.group : 0);
  const uint4 *qr =
      reinterpret_cast<const uint4 *>(p.q + (static_cast<long long>(b) * p.hq + head) * kHeadDim);
  uint8_t *qs = smem + kOffQ + q * kPQBytes;
#pragma unroll
  for (int cc = 0; cc < 16; ++cc) {
    const uint4 v = live ? __ldg(qr + cc) : make_uint4(0u, 0u, 0u, 0u);
    *reinterpret_cast<uint4 *>(qs + (cc >> 3) * (kPQRows * 128) + r * 128 +
                               (((cc & 7) ^ (r & 7)) << 4)) = v;
  }
  ptx::fence_proxy_async();
  ptx::mbar_arrive(bars.q_full(q));
}

// Warps 4q .. 4q + 3: query tile q, softmax, and the chunk's partial states.
template <typename T>
__device__ void softmax_rows(const PrefixParams &p, int q, int h, int rt, int c, int t_begin,
                             int n, uint8_t *smem, uint32_t tmem, const Bars &bars,
                             volatile int *abort) {
  const int r = threadIdx.x & (kSoftmaxThreads - 1);
  const int lane = r & 31;
  const uint32_t lane_base = static_cast<uint32_t>(r & ~31) << 16;
  const uint32_t t_s = tmem + lane_base + col_s(q);
  const uint32_t t_o = tmem + lane_base + col_o(q);
  const int rows = p.batch * p.group;
  const int row_id = rt * kPRows + q * kPQRows + r;
  const bool live = row_id < rows;
  const int b = live ? row_id / p.group : 0;
  const int head = h * p.group + (live ? row_id % p.group : 0);
  const float cs = p.scale_log2;

  float ref = -INFINITY;  // scaled reference of this row
  float l = 0.f;          // row sum of P
  bool failed = false;
  for (int i = 0; i < n; ++i) {
    if (!warp_wait(bars.s_full(q), i & 1, abort)) {
      failed = true;
      break;
    }
    tc::fence_after_sync();
    // S_q of tile i was issued after P_q V_{i-1} completed, so O holds tiles
    // < i from here on
    const int valid = min(kPTile, p.length - (t_begin + i) * kPTile);
    if (valid == kPTile)
      softmax_tile<T, true>(t_s, t_o, valid, cs, i > 0, ref, l);
    else
      softmax_tile<T, false>(t_s, t_o, valid, cs, i > 0, ref, l);
    tc::wait_st();
    tc::fence_before_sync();
    ptx::mbar_arrive(bars.p_full(q));
  }
  if (failed) {
    if (lane == 0) give_up(p, abort);
    return;
  }

  const long long slot_floats = partial_slot_floats(p.hq, kHeadDim);
  float *base = p.partials + (static_cast<long long>(b) * p.chunks + c) * slot_floats;
  float *o = base + head * kHeadDim;
  if (n == 0) {
    if (live) {
      for (int d = 0; d < kHeadDim; d += 4)
        *reinterpret_cast<float4 *>(o + d) = make_float4(0.f, 0.f, 0.f, 0.f);
      base[p.hq * kHeadDim + head] = -INFINITY;
    }
    return;
  }
  if (!warp_wait(bars.p_free(q), (n - 1) & 1, abort)) {
    if (lane == 0) give_up(p, abort);
    return;
  }
  tc::fence_after_sync();
  const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll 1
  for (int cc = 0; cc < kHeadDim / 16; ++cc) {
    float v[16];
    tc::ld16(t_o + 16 * cc, v);
    if (live) {
#pragma unroll
      for (int e = 0; e < 16; e += 4)
        *reinterpret_cast<float4 *>(o + 16 * cc + e) =
            make_float4(v[e] * inv, v[e + 1] * inv, v[e + 2] * inv, v[e + 3] * inv);
    }
  }
  if (live) base[p.hq * kHeadDim + head] = l > 0.f ? (ref + log2f(l)) * kLn2 : -INFINITY;
}

template <typename T>
__global__ void __launch_bounds__(kPThreads, 1)
    shared_prefix_kernel(const __grid_constant__ PrefixParams p,
                         const __grid_constant__ CUtensorMap map_k,
                         const __grid_constant__ CUtensorMap map_v,
                         const __grid_constant__ CUtensorMap map_q) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const Bars bars{ptx::smem_u32(smem + kOffBars)};
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + kOffMisc);
  volatile int *abort = reinterpret_cast<volatile int *>(smem + kOffMisc + 4);
  const int warp = threadIdx.x >> 5;

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
  const int n = min(total_tiles, t_begin + p.chunk_tiles) - t_begin;
  const int nq = p.batch * p.group - rt * kPRows > kPQRows ? 2 : 1;  // live query tiles
  ptx::launch_dependents();

  if (threadIdx.x == 0) {
    for (int t = 0; t < 2; ++t)
      for (int s = 0; s < kPStages; ++s) {
        ptx::mbar_init(bars.full(t, s), 1);
        ptx::mbar_init(bars.empty(t, s), nq);  // released by each live query tile
      }
    for (int q = 0; q < 2; ++q) {
      ptx::mbar_init(bars.s_full(q), 1);
      ptx::mbar_init(bars.p_full(q), kSoftmaxThreads);
      ptx::mbar_init(bars.p_free(q), 1);
      ptx::mbar_init(bars.q_full(q), p.q_tma ? 1 : kSoftmaxThreads);
      ptx::mbar_init(bars.drain(q), 1);
    }
    ptx::mbar_init(bars.ack(), 1);
    *abort = 0;
    ptx::fence_mbar_init();
    ptx::fence_proxy_async();
  }
  __syncthreads();  // barriers initialised

  if (warp >= kLoadWarp) {
    // the loaders start at once; they touch no tensor memory.  The K loader
    // first fetches the query tiles: two boxes (d-halves) of 128 rows each
    const int tensor = warp - kLoadWarp;
    if (tensor == 0 && p.q_tma && (threadIdx.x & 31) == 0) {
      const uint32_t q_s = ptx::smem_u32(smem + kOffQ);
      for (int q = 0; q < nq; ++q) {
        const int b0 = (rt * kPRows + q * kPQRows) / p.group;
        ptx::mbar_arrive_expect_tx(bars.q_full(q), kPQBytes);
        for (int half = 0; half < 2; ++half)
          ptx::tma_load_3d(q_s + q * kPQBytes + half * kPQRows * 128, &map_q, half * 64,
                           h * p.group, b0, bars.q_full(q));
      }
    }
    __syncwarp();
    load_prefix(p, tensor ? &map_v : &map_k, tensor, h, t_begin, n, smem, bars, abort);
  } else {
    const int q = warp < kMmaWarp ? warp >> 2 : warp - kMmaWarp;
    if (warp < kMmaWarp && q < nq && !p.q_tma) load_q(p, q, h, rt, smem, bars);
    if (warp == kMmaWarp) {
      tc::alloc(ptx::smem_u32(tmem_slot), kTmemCols);
      tc::relinquish();
    }
    // tensor-memory address handoff among warps 0 .. kLoadWarp - 1
    tc::fence_before_sync();
    asm volatile("bar.sync 1, %0;\n" ::"n"(32 * kLoadWarp) : "memory");
    tc::fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    if (warp < kMmaWarp) {
      if (q < nq) softmax_rows<T>(p, q, h, rt, c, t_begin, n, smem, tmem, bars, abort);
    } else {
      if ((threadIdx.x & 31) == 0 && n > 0 && q < nq)
        issue_mmas<T>(p, n, q, nq, smem, tmem, bars, abort);
      __syncwarp();
    }
  }

  tc::fence_before_sync();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc::fence_after_sync();
    tc::dealloc(*tmem_slot, kTmemCols);
  }
}

template <typename T>
cudaError_t launch_typed(const PrefixParams &p, const CUtensorMap &mk, const CUtensorMap &mv,
                         const CUtensorMap &mq, int grid, cudaStream_t st) {
  cudaError_t e = cudaFuncSetAttribute(shared_prefix_kernel<T>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, kPSmem);
  if (e != cudaSuccess) return e;
  shared_prefix_kernel<T><<<grid, kPThreads, kPSmem, st>>>(p, mk, mv, mq);
  return cudaGetLastError();
}

}  // namespace

int launch_shared_prefix(const PrefixArgs &a, void *stream) {
  alignas(64) CUtensorMap mk;
  alignas(64) CUtensorMap mv;
  if (!page_tensor_maps(&mk, &mv, a.k_pages, a.v_pages, a.num_pages, a.page_size,
                        a.num_kv_heads, a.layout))
    return cudaErrorNotSupported;
  PrefixParams p;
  p.q = static_cast<const uint16_t *>(a.q);
  p.k = static_cast<const uint16_t *>(a.k_pages);
  p.v = static_cast<const uint16_t *>(a.v_pages);
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
  alignas(64) CUtensorMap mq;
  p.q_tma = query_tensor_map(&mq, a.q, a.batch, a.num_qo_heads, p.group) ? 1 : 0;
  if (!p.q_tma) std::memset(&mq, 0, sizeof(mq));
  const int grid = a.num_kv_heads * a.row_tiles * a.chunks;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  return a.dtype == PKD_BF16 ? launch_typed<__nv_bfloat16>(p, mk, mv, mq, grid, st)
                             : launch_typed<__half>(p, mk, mv, mq, grid, st);
}

}  // namespace pkd

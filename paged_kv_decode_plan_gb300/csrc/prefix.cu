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
//   warps 8, 9 one thread each issues the S = Q K^T MMAs of tile 0 / tile 1;
//              warp 8 also allocates tensor memory
//   warps 10, 11  one thread each issues the O += P V MMAs of tile 0 / 1 (an
//              issuing thread spends ~80 cycles per tcgen05.mma and ~200 per
//              barrier wait, so each chain gets its own thread)
//   warps 12, 13  loaders of K and of V: TMA tiled loads of head h, 64-token
//              stages, 16-token boxes, 128-byte swizzle; the prefix's ragged
//              last box is copied with plain loads, zeros past the end.  K and
//              V have their own full / empty barriers: K of a stage is free
//              once both S MMAs have read it, well before P V frees V.
// Per query tile q and 64-token tile i (S double-buffered in tensor memory):
//   S[i&1] = Q_q K_i^T           M 128, N 64, K 128 (A, B from shared memory)
//   P      = exp2(S * c - ref)   softmax threads; P (f16 / bf16 pairs) is
//                                stored over the S columns it came from
//   O     += P V_i               M 128, N 128, K 64 (A = P from tensor memory)
// bf16 P is split as hi + lo (two MMAs into the same accumulators).  The row
// sum l is kept in fp32 registers.  The running reference moves only when a
// row maximum grows by > 2^8; then O and l are rescaled (after P V of the
// previous tile has completed).  With two S buffers the tensor core computes
// S of tile i + 1 while the softmax works on tile i; S of tile i + 2 reuses
// the columns of P_i and is issued once P_i V_i has completed.  Tensor memory
// per query tile: 2 x 64 (S / P) + 128 (O) = 256 columns, 512 in all.
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
constexpr int kPTile = 64;                         // tokens per stage (MMA N of S)
constexpr int kPHalfRegion = kPTile * 128;         // one 64-column block: 64 rows x 128 B
constexpr int kPTensorBytes = 2 * kPHalfRegion;    // K (or V) of one stage
constexpr int kPOffV = kPTensorBytes;              // V after K in a stage
constexpr int kPStageBytes = 2 * kPTensorBytes;
constexpr int kPStages = 4;
constexpr int kPQBytes = kPQRows * 256;            // [d-half][row][128 B]
constexpr int kSoftmaxThreads = 128;
constexpr int kMmaWarp = 8, kLoadWarp = 12;  // warps 8 .. 11 issue MMAs; 12, 13 load
constexpr int kPThreads = 32 * 14;
constexpr uint32_t kTmemCols = 512;

// Tensor-memory columns of query tile q: two 64-column S buffers, then O
// (128).  P of a tile is stored over its S buffer: hi pairs in the first 32
// columns, bf16 lo pairs in the next 32.
__host__ __device__ constexpr uint32_t col_s(int q, int b) { return 256u * q + 64u * b; }
__host__ __device__ constexpr uint32_t col_o(int q) { return 256u * q + 128u; }
static_assert(col_o(1) + kHeadDim <= kTmemCols, "tensor-memory budget");

constexpr int kOffQ = kPStages * kPStageBytes;
constexpr int kOffBars = kOffQ + 2 * kPQBytes;
// full[tensor][S], empty[tensor][S], then per query tile and S buffer
// s_full, p_full, p_free, then per query tile q_full and the two drains
constexpr int kNumBars = 4 * kPStages + 18;
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
  // per query tile q and S buffer b (each completes once every two tiles)
  __device__ uint32_t s_full(int q, int b) const { return base + 8 * (4 * kPStages + 2 * q + b); }
  __device__ uint32_t p_full(int q, int b) const { return base + 8 * (4 * kPStages + 4 + 2 * q + b); }
  __device__ uint32_t p_free(int q, int b) const { return base + 8 * (4 * kPStages + 8 + 2 * q + b); }
  __device__ uint32_t q_full(int q) const { return base + 8 * (4 * kPStages + 12 + q); }
  // completion of every MMA issued by the S (role 0) or P V (role 1) thread of tile q
  __device__ uint32_t drain(int q, int role) const {
    return base + 8 * (4 * kPStages + 14 + 2 * q + role);
  }
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
// it % S with tokens [64 t, 64 t + 64) of head h.
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
      // rows [16 nfull, 64): plain copies up to the prefix end, zeros after
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

// Issuing threads of query tile q.  Tile i uses S buffer i & 1; the s_full /
// p_full / p_free barriers of a buffer complete once per two tiles, so tile i
// waits for their phase (i >> 1) & 1.  Neither thread can run two phases
// ahead of a waiter: S of tile i + 2 needs P V of tile i, which needs P of
// tile i.
//
// Warp kMmaWarp + q: S[i & 1] = Q_q K_i^T, eight K = 16 steps over the head
// dim.  S of tile i overwrites P of tile i - 2, so it waits for P V of tile
// i - 2 to complete (p_free).
template <typename T>
__device__ void issue_qk(const PrefixParams &p, int n, int q, uint8_t *smem, uint32_t tmem,
                         const Bars &bars, volatile int *abort) {
  constexpr bool kSplit = std::is_same<T, __nv_bfloat16>::value;
  constexpr uint32_t kIdescQK = tc::idesc_f16(kSplit, kPQRows, kPTile, false);
  const uint32_t base = ptx::smem_u32(smem);
  // Descriptors are built once; a k-step adds its byte offset / 16 to the
  // start-address field (no carry: shared addresses stay below 256 KB).
  const uint64_t q_desc = tc::smem_desc_sw128(base + kOffQ + q * kPQBytes, 16, 1024);
  const uint64_t k_desc = tc::smem_desc_sw128(base, 16, 1024);
  bool ok = wait_phase(bars.q_full(q), 0, abort);
  bool issued = false;
  for (int i = 0; ok && i < n; ++i) {
    const int b = i & 1;
    if (i >= 2 && !(ok = wait_phase(bars.p_free(q, b), ((i - 2) >> 1) & 1, abort))) break;
    if (!(ok = wait_phase(bars.full(0, i % kPStages), (i / kPStages) & 1, abort))) break;
    tc::fence_after_sync();
    issued = true;
    const uint64_t kd = k_desc + (((i % kPStages) * kPStageBytes) >> 4);
    const uint32_t t_s = tmem + col_s(q, b);
#pragma unroll
    for (int kk = 0; kk < kHeadDim / 16; ++kk) {
      const uint32_t off = ((kk >> 2) * kPQRows * 128 + (kk & 3) * 32) >> 4;
      const uint32_t koff = ((kk >> 2) * kPHalfRegion + (kk & 3) * 32) >> 4;
      tc::mma_f16(t_s, q_desc + off, kd + koff, kIdescQK, kk > 0);
    }
    tc::commit(bars.s_full(q, b));
    tc::commit(bars.empty(0, i % kPStages));  // one arrival per query tile
  }
  if (!ok) give_up(p, abort);
  if (issued) {
    // every MMA of this thread completes before tensor memory is released
    tc::commit(bars.drain(q, 0));
    wait_phase(bars.drain(q, 0), 0, abort, true);
  }
}

// Warp kMmaWarp + 2 + q: O += P_i V_i once the softmax has written P_i over
// S[i & 1] (p_full); k-steps of 16 tokens, V rows 16 j .. 16 j + 15 are two
// 8-row groups (SBO 1024), V's d-halves one half region apart (LBO).
template <typename T>
__device__ void issue_pv(const PrefixParams &p, int n, int q, uint8_t *smem, uint32_t tmem,
                         const Bars &bars, volatile int *abort) {
  constexpr bool kSplit = std::is_same<T, __nv_bfloat16>::value;
  constexpr uint32_t kIdescPV = tc::idesc_f16(kSplit, kPQRows, kHeadDim, true);
  const uint64_t v_desc = tc::smem_desc_sw128(ptx::smem_u32(smem) + kPOffV, kPHalfRegion, 1024);
  const uint32_t t_o = tmem + col_o(q);
  bool ok = true, issued = false;
  for (int i = 0; i < n; ++i) {
    const int b = i & 1;
    // V is normally resident long before P: wait for it first so the MMAs
    // follow the P wait at once
    if (!(ok = wait_phase(bars.full(1, i % kPStages), (i / kPStages) & 1, abort))) break;
    if (!(ok = wait_phase(bars.p_full(q, b), (i >> 1) & 1, abort))) break;
    tc::fence_after_sync();
    issued = true;
    const uint64_t vd = v_desc + (((i % kPStages) * kPStageBytes) >> 4);
#pragma unroll
    for (int j = 0; j < kPTile / 16; ++j) {
      const uint32_t a = tmem + col_s(q, b) + 8 * j;
      tc::mma_f16_tmem_a(t_o, a, vd + ((j * 2048) >> 4), kIdescPV, i > 0 || j > 0);
      if (kSplit) tc::mma_f16_tmem_a(t_o, a + 32, vd + ((j * 2048) >> 4), kIdescPV, true);
    }
    tc::commit(bars.p_free(q, b));
    tc::commit(bars.empty(1, i % kPStages));  // one arrival per query tile
  }
  if (!ok) give_up(p, abort);
  if (issued) {
    tc::commit(bars.drain(q, 1));
    wait_phase(bars.drain(q, 1), 0, abort, true);
  }
}

// One 64-token tile of one query row (warp-collective): row maximum, lazy
// reference move, P stored over S, row sum.  When the reference moves and O
// holds earlier tiles, O is rescaled once P V of the previous tile has
// completed (barrier o_bar, parity o_par); false if that wait gave up.
// kFull: every token of the tile is in the prefix.
template <typename T, bool kFull>
__device__ __forceinline__ bool softmax_tile(uint32_t t_s, uint32_t t_o, int valid, float cs,
                                             bool rescale_o, uint32_t o_bar, uint32_t o_par,
                                             volatile int *abort, float &ref, float &l) {
  constexpr bool kSplit = std::is_same<T, __nv_bfloat16>::value;
  float s[kPTile];
  tc::ld64(t_s, s);
  float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
  if (kFull) {
#pragma unroll
    for (int j = 0; j < kPTile; j += 2) m4[(j >> 1) & 3] = ptx::fmax3(m4[(j >> 1) & 3], s[j], s[j + 1]);
  } else {
#pragma unroll
    for (int j = 0; j < kPTile; ++j)
      if (j < valid) m4[j & 3] = fmaxf(m4[j & 3], s[j]);
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
      if (!warp_wait(o_bar, o_par, abort)) return false;
      tc::fence_after_sync();
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
  const float2 cs2 = make_float2(cs, cs), nrc2 = make_float2(-rc, -rc);
  float2 lsum[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
  // 16 tokens (8 pairs, 8 tensor-memory columns of P) at a time, so few
  // packed pairs are live; every S value is already in registers, so the
  // bf16 lo pairs may overwrite S columns of later tokens
#pragma unroll
  for (int c8 = 0; c8 < kPTile / 16; ++c8) {
    float hi[8], lo[8];  // packed pairs, carried as float bit patterns
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int pair = 8 * c8 + j, k = 2 * pair;
      const float2 x = ptx::ffma2(make_float2(s[k], s[k + 1]), cs2, nrc2);
      float2 e = make_float2(ptx::ex2(x.x), ptx::ex2(x.y));
      if (!kFull) {
        e.x = k < valid ? e.x : 0.f;
        e.y = k + 1 < valid ? e.y : 0.f;
      }
      const uint32_t h2 = ptx::pack2<T>(e.x, e.y);
      hi[j] = __uint_as_float(h2);
      if (kSplit) {
        const float2 r = ptx::fsub2(e, ptx::unpack2<T>(h2));
        lo[j] = __uint_as_float(ptx::pack2<T>(r.x, r.y));
      }
      lsum[j & 1] = ptx::fadd2(lsum[j & 1], e);
    }
    tc::st8(t_s + 8 * c8, hi);
    if (kSplit) tc::st8(t_s + 32 + 8 * c8, lo);
  }
  const float2 ls = ptx::fadd2(lsum[0], lsum[1]);
  l += ls.x + ls.y;
  return true;
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

// 256-bit global store (sm_100 and later); p must be 32-byte aligned.
__device__ __forceinline__ void store8(float *p, float a, float b, float c, float d, float e,
                                       float f, float g, float h) {
  asm volatile("st.global.v8.f32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};\n" ::"l"(p), "f"(a),
               "f"(b), "f"(c), "f"(d), "f"(e), "f"(f), "f"(g), "f"(h)
               : "memory");
}

// Warps 4q .. 4q + 3: query tile q, softmax, and the chunk's partial states.
template <typename T>
__device__ void softmax_rows(const PrefixParams &p, int q, int h, int rt, int c, int t_begin,
                             int n, uint8_t *smem, uint32_t tmem, const Bars &bars,
                             volatile int *abort) {
  const int r = threadIdx.x & (kSoftmaxThreads - 1);
  const int lane = r & 31;
  const uint32_t lane_base = static_cast<uint32_t>(r & ~31) << 16;
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
    const int sb = i & 1;
    if (!warp_wait(bars.s_full(q, sb), (i >> 1) & 1, abort)) {
      failed = true;
      break;
    }
    tc::fence_after_sync();
    // S of tile i may be ready before P V of tile i - 1 has completed (it was
    // issued into the other buffer); a rescale of O waits for that P V, whose
    // completion is phase ((i - 1) >> 1) & 1 of p_free of the other buffer
    const uint32_t t_s = tmem + lane_base + col_s(q, sb);
    const uint32_t o_bar = bars.p_free(q, sb ^ 1);
    const uint32_t o_par = ((i - 1) >> 1) & 1;
    const int valid = min(kPTile, p.length - (t_begin + i) * kPTile);
    const bool ok =
        valid == kPTile
            ? softmax_tile<T, true>(t_s, t_o, valid, cs, i > 0, o_bar, o_par, abort, ref, l)
            : softmax_tile<T, false>(t_s, t_o, valid, cs, i > 0, o_bar, o_par, abort, ref, l);
    if (!ok) {
      failed = true;
      break;
    }
    tc::wait_st();
    tc::fence_before_sync();
    ptx::mbar_arrive(bars.p_full(q, sb));
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
  if (!warp_wait(bars.p_free(q, (n - 1) & 1), ((n - 1) >> 1) & 1, abort)) {
    if (lane == 0) give_up(p, abort);
    return;
  }
  tc::fence_after_sync();
  const float inv = l > 0.f ? 1.f / l : 0.f;
  // Each thread writes its own row: whole 32-byte sectors (256-bit stores)
  // where the row is 32-byte aligned, which halves the sector writes of
  // 16-byte stores and leaves none half-filled.
  const bool wide = (reinterpret_cast<uintptr_t>(o) & 31u) == 0;
#pragma unroll 1
  for (int half = 0; half < 2; ++half) {
    float v[64];
    tc::ld64(t_o + 64 * half, v);
    if (!live) continue;
    float *dst = o + 64 * half;
    if (wide) {
#pragma unroll
      for (int e = 0; e < 64; e += 8)
        store8(dst + e, v[e] * inv, v[e + 1] * inv, v[e + 2] * inv, v[e + 3] * inv,
               v[e + 4] * inv, v[e + 5] * inv, v[e + 6] * inv, v[e + 7] * inv);
    } else {
#pragma unroll
      for (int e = 0; e < 64; e += 4)
        *reinterpret_cast<float4 *>(dst + e) =
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
      for (int b = 0; b < 2; ++b) {
        ptx::mbar_init(bars.s_full(q, b), 1);
        ptx::mbar_init(bars.p_full(q, b), kSoftmaxThreads);
        ptx::mbar_init(bars.p_free(q, b), 1);
      }
      ptx::mbar_init(bars.q_full(q), p.q_tma ? 1 : kSoftmaxThreads);
      ptx::mbar_init(bars.drain(q, 0), 1);
      ptx::mbar_init(bars.drain(q, 1), 1);
    }
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
    const int q = warp < kMmaWarp ? warp >> 2 : (warp - kMmaWarp) & 1;
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
      if ((threadIdx.x & 31) == 0 && n > 0 && q < nq) {
        if (warp < kMmaWarp + 2)
          issue_qk<T>(p, n, q, smem, tmem, bars, abort);
        else
          issue_pv<T>(p, n, q, smem, tmem, bars, abort);
      }
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
  CUtensorMap mk;
  CUtensorMap mv;
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
  CUtensorMap mq;
  p.q_tma = query_tensor_map(&mq, a.q, a.batch, a.num_qo_heads, p.group) ? 1 : 0;
  if (!p.q_tma) std::memset(&mq, 0, sizeof(mq));
  const int grid = a.num_kv_heads * a.row_tiles * a.chunks;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  return a.dtype == PKD_BF16 ? launch_typed<__nv_bfloat16>(p, mk, mv, mq, grid, st)
                             : launch_typed<__half>(p, mk, mv, mq, grid, st);
}

}  // namespace pkd

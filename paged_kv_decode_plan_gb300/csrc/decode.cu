// Split-KV paged decode attention kernel (warp-specialised).
//
// One persistent CTA per SM walks its contiguous share of the plan's work
// list.  A unit is a token range [t0, t1) of one request.  Tiles are 16
// tokens of every key/value head (16 * Hkv * 512 bytes of K and V).
//
// Roles inside a CTA:
//  * loader warp(s) fill a ring of shared-memory stages.  When a page holds
//    whole 16-token tiles (page_size % 16 == 0) one warp issues TMA tiled
//    loads (cp.async.bulk.tensor, 128-byte swizzle), one 16 x 64-element box
//    per (tensor, head, d-half), completing on the stage's "full" mbarrier.
//    Otherwise four warps copy 16-byte chunks with cp.async into the same
//    swizzled layout and arrive on the barrier when their copies land.
//  * eight consumer warps compute.  Warp w owns key/value head
//    w / (8 / Hkv) and a slice of that head's query group, so no two warps
//    share an output row.  With the query group as the N = 8 side of
//    mma.sync m16n8k16:
//        S^T = K Q^T    (16 tokens x 8 query heads, fp32 accumulate)
//        online softmax over tokens in fp32, base 2, maxima kept on the raw
//        logits and the scale sm_scale * log2(e) applied inside one fma;
//        the reference is only moved when the maximum grows by more than
//        2^8 (every p stays <= 256), so most tiles skip the rescale
//        O^T += V^T P^T (128 d x 8 query heads); P^T reaches the B operand
//        through movmatrix.  For bfloat16, P is split into hi + lo parts
//        (8 significant bits each) and multiplied twice; row sums are taken
//        over exactly the values multiplied.
// Every mbarrier wait is bounded; a wait that runs out records
// PKD_DEVICE_TIMEOUT in the status word and the CTA stops.
//
// Sources (page title, section):
//  - "FlashInfer" (aiwiki.ai/wiki/flashinfer), "Block-sparse cache
//    representation": pages reached through a page table.
//  - same page, "Custom attention templates": grouped-query heads.
//  - same page, "Attention states": a split request's units emit (output,
//    log-sum-exp) partial states, merged by the separate merge kernel.
//  - same page, "Extreme-negative-logit correction": the running maximum
//    starts at -infinity; differences are clamped so -inf - (-inf) never
//    reaches exp; an empty row yields (0, -infinity).
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstring>
#include <mutex>
#include <type_traits>

#include "pkd_internal.h"
#include "ptx.cuh"

namespace pkd {
namespace {

constexpr int kConsumerWarps = 8;
constexpr int kTile = 16;                           // tokens per tile
constexpr int kRowBytes = kHeadDim * 2;             // one token, one head
constexpr int kHalfBytes = kTile * 128;             // 16 rows x 64 elements
constexpr int kStageBudget = 3 * 64 * 1024;         // bytes of stages per CTA
constexpr float kLn2 = 0.69314718055994530942f;
constexpr float kLazy = 8.f;                        // log2 of the largest p
constexpr long long kWaitPolls = 1ll << 22;         // bounded mbarrier waits

enum Loader : int { kLoaderTma = 0, kLoaderCpAsync = 1 };

template <int L>
__host__ __device__ constexpr int loader_warps() { return L == kLoaderTma ? 1 : 4; }
__host__ __device__ constexpr int head_bytes() { return 2 * kHalfBytes; }  // one head
template <int HKV>
__host__ __device__ constexpr int tensor_bytes() { return HKV * head_bytes(); }
template <int HKV>
__host__ __device__ constexpr int stage_bytes() { return 2 * tensor_bytes<HKV>(); }
template <int HKV>
__host__ __device__ constexpr int num_stages() { return kStageBudget / stage_bytes<HKV>(); }

struct Params {
  const uint16_t *q, *k, *v;
  const int32_t *indptr, *indices, *last;
  int32_t *image;
  float *partials;
  uint16_t *out;
  float *lse;
  float scale_log2;
  long long num_pages;
  int batch, hq, group, page_size;
  int max_partials;   // partial slots the float workspace holds
  int image_words;    // int32 words of the plan image
  int grid;           // CTAs launched
};

struct Unit {
  int req, t0, t1, slot, pbase;
};

__device__ __forceinline__ void flag(int32_t *image, unsigned bit) {
  atomicOr(reinterpret_cast<unsigned int *>(image + kHStatus), bit);
}

// Reads unit u and checks it against the device page table.  Every thread
// computes the same result; a unit that fails is reduced to an empty range
// (and, if its request id is invalid, to req = -1: nothing is written).
__device__ Unit read_unit(const Params &p, const int32_t *units, int u,
                          int num_partials) {
  const int32_t *w = units + kUnitWords * u;
  Unit r;
  r.req = __ldg(w);
  r.t0 = __ldg(w + 1);
  r.t1 = __ldg(w + 2);
  r.slot = __ldg(w + 3);
  r.pbase = 0;
  if (r.req < 0 || r.req >= p.batch || r.slot < -1 || r.slot >= num_partials ||
      r.t0 < 0 || r.t1 < r.t0) {
    if (threadIdx.x == 0) flag(p.image, PKD_DEVICE_BAD_PLAN);
    r.req = -1;
    r.t0 = r.t1 = 0;
    return r;
  }
  const int pb = __ldg(p.indptr + r.req);
  const int pe = __ldg(p.indptr + r.req + 1);
  long long len = 0;
  if (pe > pb) {
    const int last = min(max(__ldg(p.last + r.req), 1), p.page_size);
    len = static_cast<long long>(pe - pb - 1) * p.page_size + last;
  }
  if (r.t1 > len) {
    if (threadIdx.x == 0) flag(p.image, PKD_DEVICE_BAD_LENGTH);
    r.t1 = static_cast<int>(len);
    if (r.t0 > r.t1) r.t0 = r.t1;
  }
  r.pbase = pb;
  return r;
}

__device__ __forceinline__ int unit_tiles(const Unit &u) {
  return (u.t1 - u.t0 + kTile - 1) / kTile;
}

// Polls an mbarrier phase; gives up (false) after kWaitPolls polls or once
// another warp has given up.  `patient` waits ignore the abort flag.
__device__ __forceinline__ bool wait_phase(uint32_t bar, uint32_t parity,
                                           volatile int *abort, bool patient = false) {
  for (long long i = 0; i < kWaitPolls; ++i) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    if (!patient && (i & 63) == 63 && *abort) return false;
  }
  return false;
}

__device__ __forceinline__ void give_up(const Params &p, volatile int *abort) {
  *abort = 1;
  flag(p.image, PKD_DEVICE_TIMEOUT);
}

// Byte offset of 16-byte chunk c (0..15) of token row r (0..15) within one
// head's K or V tile: [d-half][row][128 B], chunks XOR-swizzled by row as the
// TMA 128-byte swizzle lays them out.
__device__ __forceinline__ uint32_t tile_offset(int r, int c) {
  return (c >> 3) * kHalfBytes + r * 128 + (((c & 7) ^ (r & 7)) << 4);
}

// ----------------------------------------------------------------- loaders

template <int HKV>
__device__ void load_tma(const Params &p, const CUtensorMap *map_k,
                         const CUtensorMap *map_v, const int32_t *units,
                         int num_partials, int u_begin, int u_end, uint8_t *stages,
                         uint32_t full0, uint32_t empty0, volatile int *abort) {
  constexpr int kStages = num_stages<HKV>();
  const int lane = threadIdx.x & 31;
  const uint32_t stage0 = ptx::smem_u32(stages);
  int it = 0;
  bool ok = true;
  for (int u = u_begin; u < u_end && ok; ++u) {
    const Unit unit = read_unit(p, units, u, num_partials);
    const int ntiles = unit_tiles(unit);
    for (int t = 0; t < ntiles; ++t) {
      const int s = it % kStages;
      if (!wait_phase(empty0 + 8 * s, ((it / kStages) & 1) ^ 1, abort)) {
        if (lane == 0) give_up(p, abort);
        ok = false;
        break;
      }
      const int tok0 = unit.t0 + t * kTile;
      const int pi = tok0 / p.page_size;
      const int slot0 = tok0 - pi * p.page_size;
      int page = __ldg(p.indices + unit.pbase + pi);
      if (static_cast<unsigned long long>(page) >=
          static_cast<unsigned long long>(p.num_pages)) {
        if (lane == 0) flag(p.image, PKD_DEVICE_BAD_PAGE);
        page = 0;
      }
      if (lane == 0) ptx::mbar_arrive_expect_tx(full0 + 8 * s, stage_bytes<HKV>());
      __syncwarp();
      if (lane < 4 * HKV) {
        const int tensor = lane / (2 * HKV);
        const int head = (lane >> 1) % HKV;
        const int half = lane & 1;
        const uint32_t dst = stage0 + s * stage_bytes<HKV>() +
                             tensor * tensor_bytes<HKV>() + head * head_bytes() +
                             half * kHalfBytes;
        ptx::tma_load_3d(dst, tensor ? map_v : map_k, half * 64, head,
                         page * p.page_size + slot0, full0 + 8 * s);
      }
      ++it;
    }
  }
  // the CTA must not retire while this warp's copies are still landing
  for (int j = max(0, it - kStages); j < it; ++j)
    wait_phase(full0 + 8 * (j % kStages), (j / kStages) & 1, abort, true);
}

template <int HKV>
struct CpAsyncLoader {
  static constexpr int kRows = 2 * HKV;  // (token, head) rows per thread per tensor

  const Params &p;
  const int32_t *units;
  int num_partials, u, u_end, t;
  Unit unit;
  bool have;
  int tok0, t1;
  int page[kRows], slot[kRows];

  __device__ CpAsyncLoader(const Params &p_, const int32_t *units_, int np, int ub,
                           int ue)
      : p(p_), units(units_), num_partials(np), u(ub), u_end(ue), t(0), have(false) {
    if (u < u_end) unit = read_unit(p, units, u, num_partials);
    describe();
  }

  __device__ __forceinline__ static int lt() {
    return static_cast<int>(threadIdx.x) - 32 * kConsumerWarps;
  }
  __device__ __forceinline__ static int row_token(int j) { return ((lt() >> 4) + 8 * j) / HKV; }
  __device__ __forceinline__ static int row_head(int j) { return ((lt() >> 4) + 8 * j) % HKV; }

  // Moves to the next tile and starts the page-id loads it needs.
  __device__ void describe() {
    while (u < u_end && unit.t0 + t * kTile >= unit.t1) {
      ++u;
      t = 0;
      if (u < u_end) unit = read_unit(p, units, u, num_partials);
    }
    have = u < u_end;
    if (!have) return;
    tok0 = unit.t0 + t * kTile;
    t1 = unit.t1;
#pragma unroll
    for (int j = 0; j < kRows; ++j) {
      const int tok = tok0 + row_token(j);
      int pg = 0, sl = 0;
      if (tok < t1) {
        const int pi = tok / p.page_size;
        sl = tok - pi * p.page_size;
        pg = __ldg(p.indices + unit.pbase + pi);
      }
      page[j] = pg;
      slot[j] = sl;
    }
    ++t;
  }

  // Copies the described tile into the stage at `dst` (zero rows past the
  // unit's end).
  __device__ void issue(uint32_t dst) {
    const int c = lt() & 15;
#pragma unroll
    for (int j = 0; j < kRows; ++j) {
      const int tl = row_token(j);
      const int head = row_head(j);
      bool valid = tok0 + tl < t1;
      if (valid && static_cast<unsigned long long>(page[j]) >=
                       static_cast<unsigned long long>(p.num_pages)) {
        flag(p.image, PKD_DEVICE_BAD_PAGE);
        valid = false;
      }
      const long long row =
          valid ? (static_cast<long long>(page[j]) * p.page_size + slot[j]) * HKV + head
                : 0;
      const uint32_t off = head * head_bytes() + tile_offset(tl, c);
      const uint32_t n = valid ? 16u : 0u;
      ptx::cp_async_16(dst + off, p.k + row * kHeadDim + c * 8, n);
      ptx::cp_async_16(dst + tensor_bytes<HKV>() + off, p.v + row * kHeadDim + c * 8, n);
    }
  }
};

template <int HKV>
__device__ void load_cp_async(const Params &p, const int32_t *units, int num_partials,
                              int u_begin, int u_end, uint8_t *stages, uint32_t full0,
                              uint32_t empty0, volatile int *abort) {
  constexpr int kStages = num_stages<HKV>();
  const uint32_t stage0 = ptx::smem_u32(stages);
  CpAsyncLoader<HKV> ld(p, units, num_partials, u_begin, u_end);
  int it = 0;
  while (ld.have) {
    const int s = it % kStages;
    if (!wait_phase(empty0 + 8 * s, ((it / kStages) & 1) ^ 1, abort)) {
      give_up(p, abort);
      break;
    }
    ld.issue(stage0 + s * stage_bytes<HKV>());
    ptx::cp_async_mbar_arrive_noinc(full0 + 8 * s);
    ld.describe();
    ++it;
  }
  ptx::cp_async_wait_all();
}

// ---------------------------------------------------------------- consumer

template <typename T, int HKV, int NG>
__device__ void consume(const Params &p, const int32_t *units, int num_partials,
                        int u_begin, int u_end, const uint8_t *stages, uint32_t full0,
                        uint32_t empty0, volatile int *abort) {
  constexpr int kStages = num_stages<HKV>();
  constexpr int kQw = kConsumerWarps / HKV;       // warps per key/value head
  constexpr bool kSplitP = std::is_same<T, __nv_bfloat16>::value;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int hk = warp / kQw, qpart = warp % kQw;
  const int gid = lane >> 2, tq = lane & 3;
  const int gq = (p.group + kQw - 1) / kQw;       // query heads per warp
  const int col_lo = qpart * gq;
  const int col_hi = min(p.group, col_lo + gq);   // this warp's columns
  const float c = p.scale_log2;
  const uint32_t stage0 = ptx::smem_u32(stages);
  const int slot_floats = static_cast<int>(partial_slot_floats(p.hq, kHeadDim));
  // ldmatrix row addresses: K as the A operand (non-transposed), V^T as the
  // A operand (transposed load of V rows)
  const int a_row = (lane & 7) + (((lane >> 3) & 1) << 3);
  const int a_hi = lane >> 4;
  const int v_row = (lane & 7) + ((lane >> 4) << 3);
  const int v_hi = (lane >> 3) & 1;

  int it = 0;
  for (int u = u_begin; u < u_end; ++u) {
    const Unit unit = read_unit(p, units, u, num_partials);
    const int ntiles = unit_tiles(unit);

    // Q^T as the B operand: column n*8 + gid is query head col_lo + n*8 + gid
    uint32_t qb[NG][8][2];
#pragma unroll
    for (int n = 0; n < NG; ++n) {
      const int col = col_lo + 8 * n + gid;
      const bool ok = unit.req >= 0 && col < col_hi;
      const uint16_t *qrow =
          p.q + (static_cast<long long>(max(unit.req, 0)) * p.hq + hk * p.group +
                 min(col, p.group - 1)) * kHeadDim;
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        qb[n][kk][0] =
            ok ? __ldg(reinterpret_cast<const uint32_t *>(qrow + 16 * kk + 2 * tq)) : 0u;
        qb[n][kk][1] =
            ok ? __ldg(reinterpret_cast<const uint32_t *>(qrow + 16 * kk + 8 + 2 * tq)) : 0u;
      }
    }

    float ref[NG][2], l[NG][2], acc[NG][8][4];
#pragma unroll
    for (int n = 0; n < NG; ++n) {
      ref[n][0] = ref[n][1] = -INFINITY;
      l[n][0] = l[n][1] = 0.f;
#pragma unroll
      for (int mt = 0; mt < 8; ++mt)
        acc[n][mt][0] = acc[n][mt][1] = acc[n][mt][2] = acc[n][mt][3] = 0.f;
    }

    bool stop = false;
    for (int t = 0; t < ntiles; ++t, ++it) {
      const int s = it % kStages;
      if (!wait_phase(full0 + 8 * s, (it / kStages) & 1, abort)) {
        if (lane == 0) give_up(p, abort);
        stop = true;
        break;
      }
      const uint32_t kb = stage0 + s * stage_bytes<HKV>() + hk * head_bytes();
      const uint32_t vb = kb + tensor_bytes<HKV>();
      const int valid = min(kTile, unit.t1 - unit.t0 - t * kTile);

      // S^T = K Q^T: rows are tokens, columns this warp's query heads
      float sc[NG][4];
#pragma unroll
      for (int n = 0; n < NG; ++n) sc[n][0] = sc[n][1] = sc[n][2] = sc[n][3] = 0.f;
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        uint32_t a[4];
        ptx::ldmatrix_x4(kb + tile_offset(a_row, 2 * kk + a_hi), a[0], a[1], a[2], a[3]);
#pragma unroll
        for (int n = 0; n < NG; ++n) ptx::mma_16816<T>(sc[n], a, qb[n][kk][0], qb[n][kk][1]);
      }

      // online softmax over tokens, per query-head column
      bool need = false;
      float cand[NG][2];
#pragma unroll
      for (int n = 0; n < NG; ++n) {
        if (gid >= valid) sc[n][0] = sc[n][1] = -INFINITY;
        if (gid + 8 >= valid) sc[n][2] = sc[n][3] = -INFINITY;
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          float mx = fmaxf(sc[n][j], sc[n][j + 2]);
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
          cand[n][j] = mx * c;
          need |= cand[n][j] > ref[n][j] + kLazy;
        }
      }
      if (__any_sync(0xffffffffu, need)) {
#pragma unroll
        for (int n = 0; n < NG; ++n)
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            float alpha = 1.f;
            if (cand[n][j] > ref[n][j] + kLazy) {
              alpha = exp2f(ref[n][j] - cand[n][j]);  // ref = -inf gives 0
              ref[n][j] = cand[n][j];
            }
            l[n][j] *= alpha;
#pragma unroll
            for (int mt = 0; mt < 8; ++mt) {
              acc[n][mt][j] *= alpha;
              acc[n][mt][j + 2] *= alpha;
            }
          }
      }

      // P^T as the B operand of O^T += V^T P^T
      uint32_t pb[NG][2], pl[NG][2];
#pragma unroll
      for (int n = 0; n < NG; ++n) {
        const float r0 = ref[n][0] == -INFINITY ? 0.f : ref[n][0];  // clamp
        const float r1 = ref[n][1] == -INFINITY ? 0.f : ref[n][1];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const float e0 = exp2f(fmaf(sc[n][2 * h], c, -r0));
          const float e1 = exp2f(fmaf(sc[n][2 * h + 1], c, -r1));
          const uint32_t hi = ptx::pack2<T>(e0, e1);
          const float2 bh = ptx::unpack2<T>(hi);
          pb[n][h] = ptx::movmatrix_trans(hi);
          if (kSplitP) {
            const uint32_t lo = ptx::pack2<T>(e0 - bh.x, e1 - bh.y);
            const float2 bl = ptx::unpack2<T>(lo);
            pl[n][h] = ptx::movmatrix_trans(lo);
            l[n][0] += bh.x + bl.x;
            l[n][1] += bh.y + bl.y;
          } else {
            pl[n][h] = 0u;
            l[n][0] += bh.x;
            l[n][1] += bh.y;
          }
        }
      }

      // V rows past the unit's end may hold anything: zero them in the A
      // fragments (tokens 2tq, 2tq+1 and 2tq+8, 2tq+9 of this lane)
      uint32_t m01 = 0xffffffffu, m89 = 0xffffffffu;
      if (valid < kTile) {
        m01 = (2 * tq < valid ? 0x0000ffffu : 0u) | (2 * tq + 1 < valid ? 0xffff0000u : 0u);
        m89 = (2 * tq + 8 < valid ? 0x0000ffffu : 0u) |
              (2 * tq + 9 < valid ? 0xffff0000u : 0u);
      }
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) {
        uint32_t a[4];
        ptx::ldmatrix_x4_trans(vb + tile_offset(v_row, 2 * mt + v_hi), a[0], a[1], a[2],
                               a[3]);
        a[0] &= m01;
        a[1] &= m01;
        a[2] &= m89;
        a[3] &= m89;
#pragma unroll
        for (int n = 0; n < NG; ++n) {
          ptx::mma_16816<T>(acc[n][mt], a, pb[n][0], pb[n][1]);
          if (kSplitP) ptx::mma_16816<T>(acc[n][mt], a, pl[n][0], pl[n][1]);
        }
      }
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(empty0 + 8 * s);
    }
    if (stop) return;

    // column sums across the eight token rows of the fragment
#pragma unroll
    for (int n = 0; n < NG; ++n)
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        l[n][j] += __shfl_xor_sync(0xffffffffu, l[n][j], 4);
        l[n][j] += __shfl_xor_sync(0xffffffffu, l[n][j], 8);
        l[n][j] += __shfl_xor_sync(0xffffffffu, l[n][j], 16);
      }
    if (unit.req < 0) continue;
#pragma unroll
    for (int n = 0; n < NG; ++n)
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int col = col_lo + 8 * n + 2 * tq + j;
        if (col >= col_hi) continue;
        const int head = hk * p.group + col;
        const float inv = l[n][j] > 0.f ? 1.f / l[n][j] : 0.f;
        const float lse_h =
            l[n][j] > 0.f ? (ref[n][j] + log2f(l[n][j])) * kLn2 : -INFINITY;
        if (unit.slot < 0) {
          uint16_t *o = p.out + (static_cast<long long>(unit.req) * p.hq + head) * kHeadDim;
#pragma unroll
          for (int mt = 0; mt < 8; ++mt) {
            const uint32_t pair =
                ptx::pack2<T>(acc[n][mt][j] * inv, acc[n][mt][j + 2] * inv);
            o[16 * mt + gid] = static_cast<uint16_t>(pair & 0xffffu);
            o[16 * mt + gid + 8] = static_cast<uint16_t>(pair >> 16);
          }
          if (gid == 0) p.lse[static_cast<long long>(unit.req) * p.hq + head] = lse_h;
        } else {
          float *base = p.partials + static_cast<long long>(unit.slot) * slot_floats;
          float *o = base + head * kHeadDim;
#pragma unroll
          for (int mt = 0; mt < 8; ++mt) {
            o[16 * mt + gid] = acc[n][mt][j] * inv;
            o[16 * mt + gid + 8] = acc[n][mt][j + 2] * inv;
          }
          if (gid == 0) base[p.hq * kHeadDim + head] = lse_h;
        }
      }
  }
}

// ------------------------------------------------------------------ kernel

template <typename T, int HKV, int NG, int LOADER>
__global__ void __launch_bounds__(32 * (kConsumerWarps + loader_warps<LOADER>()), 1)
    decode_kernel(const __grid_constant__ Params p,
                  const __grid_constant__ CUtensorMap map_k,
                  const __grid_constant__ CUtensorMap map_v) {
  constexpr int kStages = num_stages<HKV>();
  extern __shared__ uint8_t smem_raw[];
  uint8_t *stages = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t *bars = reinterpret_cast<uint64_t *>(stages + kStages * stage_bytes<HKV>());
  volatile int *abort = reinterpret_cast<volatile int *>(bars + 2 * kStages);
  const uint32_t full0 = ptx::smem_u32(bars);
  const uint32_t empty0 = full0 + 8 * kStages;

  // the image must be the one the host planned for this launch
  const int32_t *img = p.image;
  const int num_ctas = img[kHNumCtas];
  const int num_units = img[kHNumUnits];
  const int num_partials = img[kHNumPartials];
  if (img[kHMagic] != kMagic || img[kHVersion] != kLayoutVersion ||
      img[kHBatch] != p.batch || img[kHTileTokens] != kTile ||
      img[kHNumQoHeads] != p.hq || img[kHPageSize] != p.page_size ||
      num_ctas != p.grid || num_units < 0 || num_partials < 0 ||
      num_partials > p.max_partials || img[kHNumSplit] < 0 ||
      image_offsets(num_ctas, num_units, img[kHNumSplit]).end > p.image_words) {
    if (threadIdx.x == 0 && blockIdx.x == 0) flag(p.image, PKD_DEVICE_BAD_PLAN);
    return;
  }
  const int32_t *cta_ptr = img + kHeaderWords;
  const int32_t *units = cta_ptr + num_ctas + 1;
  const int u_begin = cta_ptr[blockIdx.x], u_end = cta_ptr[blockIdx.x + 1];
  if (u_begin < 0 || u_end > num_units || u_begin > u_end) {
    if (threadIdx.x == 0) flag(p.image, PKD_DEVICE_BAD_PLAN);
    return;
  }
  // a merge kernel launched after this one may be scheduled from now on; it
  // waits for this grid to finish before it reads any partial state
  ptx::launch_dependents();
  if (u_begin == u_end) return;

  if (threadIdx.x == 0) {
    const uint32_t full_count =
        LOADER == kLoaderTma ? 1u : 32u * loader_warps<kLoaderCpAsync>();
    for (int s = 0; s < kStages; ++s) {
      ptx::mbar_init(full0 + 8 * s, full_count);
      ptx::mbar_init(empty0 + 8 * s, kConsumerWarps);
    }
    *abort = 0;
    ptx::fence_mbar_init();
    ptx::fence_proxy_async();
  }
  __syncthreads();

  if (threadIdx.x >= 32 * kConsumerWarps) {
    if (LOADER == kLoaderTma)
      load_tma<HKV>(p, &map_k, &map_v, units, num_partials, u_begin, u_end, stages,
                    full0, empty0, abort);
    else
      load_cp_async<HKV>(p, units, num_partials, u_begin, u_end, stages, full0,
                         empty0, abort);
  } else {
    consume<T, HKV, NG>(p, units, num_partials, u_begin, u_end, stages, full0,
                        empty0, abort);
  }
}

template <int HKV>
__host__ __device__ constexpr int smem_bytes() {
  return 1024 + num_stages<HKV>() * stage_bytes<HKV>() + 16 * num_stages<HKV>() + 16;
}

template <typename T, int HKV, int NG, int LOADER>
int launch_typed(const Params &prm, const CUtensorMap &mk, const CUtensorMap &mv,
                 void *stream) {
  auto kernel = decode_kernel<T, HKV, NG, LOADER>;
  const int smem = smem_bytes<HKV>();
  cudaError_t e =
      cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  kernel<<<prm.grid, 32 * (kConsumerWarps + loader_warps<LOADER>()), smem,
           static_cast<cudaStream_t>(stream)>>>(prm, mk, mv);
  return cudaGetLastError();
}

template <typename T, int HKV, int NG>
int launch_loader(const Params &prm, bool tma, const CUtensorMap &mk,
                  const CUtensorMap &mv, void *stream) {
  if (tma) return launch_typed<T, HKV, NG, kLoaderTma>(prm, mk, mv, stream);
  return launch_typed<T, HKV, NG, kLoaderCpAsync>(prm, mk, mv, stream);
}

template <typename T, int HKV>
int launch_group(const Params &prm, bool tma, const CUtensorMap &mk,
                 const CUtensorMap &mv, void *stream) {
  constexpr int kQw = kConsumerWarps / HKV;
  const int gq = (prm.group + kQw - 1) / kQw;
  if (gq > 8) return launch_loader<T, HKV, 2>(prm, tma, mk, mv, stream);
  return launch_loader<T, HKV, 1>(prm, tma, mk, mv, stream);
}

template <typename T>
int launch_heads(const Params &prm, int hkv, bool tma, const CUtensorMap &mk,
                 const CUtensorMap &mv, void *stream) {
  switch (hkv) {
    case 1: return launch_group<T, 1>(prm, tma, mk, mv, stream);
    case 2: return launch_group<T, 2>(prm, tma, mk, mv, stream);
    case 4: return launch_group<T, 4>(prm, tma, mk, mv, stream);
    default: return launch_group<T, 8>(prm, tma, mk, mv, stream);
  }
}

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                         cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

// K or V pages viewed as [token row][head][d] with d innermost; boxes of 16
// token rows x 1 head x 64 elements, 128-byte swizzle.
bool encode_pages(CUtensorMap *map, const void *base, long long num_pages,
                  int page_size, int hkv) {
  PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
  if (!encode) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(kHeadDim), static_cast<cuuint64_t>(hkv),
                        static_cast<cuuint64_t>(num_pages) * page_size};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(kRowBytes),
                           static_cast<cuuint64_t>(kRowBytes) * hkv};
  cuuint32_t box[3] = {64, 1, kTile};
  cuuint32_t estr[3] = {1, 1, 1};
  return encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT16, 3, const_cast<void *>(base), dims,
                strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

int launch_decode(const DecodeArgs &a, void *stream) {
  Params prm;
  prm.q = static_cast<const uint16_t *>(a.q);
  prm.k = static_cast<const uint16_t *>(a.k_pages);
  prm.v = static_cast<const uint16_t *>(a.v_pages);
  prm.indptr = a.kv_indptr;
  prm.indices = a.kv_indices;
  prm.last = a.kv_last_page_len;
  prm.image = a.image;
  prm.partials = a.partials;
  prm.out = static_cast<uint16_t *>(a.out);
  prm.lse = a.lse;
  prm.scale_log2 = a.sm_scale_log2;
  prm.num_pages = a.num_pages;
  prm.batch = a.batch;
  prm.hq = a.num_qo_heads;
  prm.group = a.num_qo_heads / a.num_kv_heads;
  prm.page_size = a.page_size;
  prm.max_partials = a.max_partials;
  prm.image_words = a.image_words;
  prm.grid = a.num_ctas;

  alignas(64) CUtensorMap mk;
  alignas(64) CUtensorMap mv;
  std::memset(&mk, 0, sizeof(mk));
  std::memset(&mv, 0, sizeof(mv));
  // TMA when every tile lies inside one page and token rows fit in int32
  const bool tma = a.page_size % kTile == 0 && a.num_pages > 0 &&
                   a.num_pages * static_cast<long long>(a.page_size) < (1ll << 31) &&
                   encode_pages(&mk, a.k_pages, a.num_pages, a.page_size, a.num_kv_heads) &&
                   encode_pages(&mv, a.v_pages, a.num_pages, a.page_size, a.num_kv_heads);
  if (a.dtype == PKD_BF16)
    return launch_heads<__nv_bfloat16>(prm, a.num_kv_heads, tma, mk, mv, stream);
  return launch_heads<__half>(prm, a.num_kv_heads, tma, mk, mv, stream);
}

}  // namespace pkd

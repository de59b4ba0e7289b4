// Split-KV paged decode attention kernel.
//
// One persistent CTA per SM walks its contiguous share of the plan's work
// list.  A unit is a token range [t0, t1) of one request; the CTA covers every
// key/value head of that range, so each tile it loads is whole tokens (all
// heads, NHD-contiguous in memory).  Tiles of 128 (token, head) rows of K and
// V (64 KB) flow through a 3-stage cp.async pipeline into XOR-swizzled shared
// memory; page ids are looked up one tile ahead of the copies that use them.
//
// Warp w handles key/value head w / (8 / Hkv) and 16 tokens of each tile.
// The query group (g <= 16 heads) is the M = 16 side of mma.sync m16n8k16:
//   S = Q K^T  (fp32 accumulate), online softmax in fp32 (base 2, with the
//   scale sm_scale * log2(e) applied inside the exponent), O = O * alpha + P V.
// P enters the second product in the input type (for bfloat16 as a hi + lo
// pair); the row sums are taken over exactly the values multiplied, so O / l
// stays a convex combination of the value rows.
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
#include <cuda_runtime.h>

#include <cmath>
#include <type_traits>

#include "pkd_internal.h"
#include "ptx.cuh"

namespace pkd {
namespace {

constexpr int kWarps = 8;
constexpr int kThreads = 32 * kWarps;
constexpr int kStages = 3;
constexpr int kRowBytes = kHeadDim * 2;                  // one token, one head
constexpr int kTileRows = 128;                           // (token, head) rows
constexpr int kTensorTileBytes = kTileRows * kRowBytes;  // 32 KB
constexpr int kStageBytes = 2 * kTensorTileBytes;        // K then V
constexpr int kRowsPerThread = kTileRows * 16 / kThreads;  // 16-byte chunks
constexpr float kLn2 = 0.69314718055994530942f;

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

// A tile ready to be copied: its first token, the unit's end, and the page id
// and in-page slot of each of this thread's rows.
struct TileDesc {
  int tok0, t1;
  int page[kRowsPerThread];
  int slot[kRowsPerThread];
};

template <int HKV>
struct Pipeline {
  static constexpr int kTile = kTileRows / HKV;  // tokens per tile

  const Params &p;
  const int32_t *units;
  int num_partials;
  int u, u_end, t;  // cursor: next tile to describe is tile t of unit u
  Unit unit;
  bool have;        // desc holds a tile
  TileDesc desc;

  __device__ Pipeline(const Params &p_, const int32_t *units_, int num_partials_,
                      int u_begin, int u_end_)
      : p(p_), units(units_), num_partials(num_partials_), u(u_begin),
        u_end(u_end_), t(0), have(false) {
    if (u < u_end) unit = read_unit(p, units, u, num_partials);
    describe();
  }

  // First token of this thread's row j within the tile, and its head.
  __device__ __forceinline__ static int row_token(int j) {
    return ((threadIdx.x >> 4) + 16 * j) / HKV;
  }
  __device__ __forceinline__ static int row_head() {
    return (threadIdx.x >> 4) % HKV;
  }

  // Advances the cursor to the next tile and loads its page ids.
  __device__ void describe() {
    while (u < u_end && unit.t0 + t * kTile >= unit.t1) {
      ++u;
      t = 0;
      if (u < u_end) unit = read_unit(p, units, u, num_partials);
    }
    have = u < u_end;
    if (!have) return;
    desc.tok0 = unit.t0 + t * kTile;
    desc.t1 = unit.t1;
#pragma unroll
    for (int j = 0; j < kRowsPerThread; ++j) {
      const int tok = desc.tok0 + row_token(j);
      int page = 0, slot = 0;
      if (tok < desc.t1) {
        const int pi = tok / p.page_size;
        slot = tok - pi * p.page_size;
        page = __ldg(p.indices + unit.pbase + pi);
      }
      desc.page[j] = page;
      desc.slot[j] = slot;
    }
    ++t;
  }

  // Copies the described tile into `stage` (zero rows past the unit's end),
  // then describes the next one.  Always commits one cp.async group.
  __device__ void issue(uint8_t *stage) {
    if (have) {
      const int c = threadIdx.x & 15;
      const int head = row_head();
      const uint32_t k_dst = ptx::smem_u32(stage);
      const uint32_t v_dst = k_dst + kTensorTileBytes;
#pragma unroll
      for (int j = 0; j < kRowsPerThread; ++j) {
        const int tl = row_token(j);
        const int tok = desc.tok0 + tl;
        bool valid = tok < desc.t1;
        const int page = desc.page[j];
        if (valid && static_cast<unsigned long long>(page) >=
                         static_cast<unsigned long long>(p.num_pages)) {
          flag(p.image, PKD_DEVICE_BAD_PAGE);
          valid = false;
        }
        const long long row =
            valid ? ((static_cast<long long>(page) * p.page_size + desc.slot[j]) *
                         HKV + head)
                  : 0;
        const uint32_t off =
            (head * kTile + tl) * kRowBytes + ((c ^ (tl & 7)) << 4);
        const uint32_t n = valid ? 16u : 0u;
        ptx::cp_async_16(k_dst + off, p.k + row * kHeadDim + c * 8, n);
        ptx::cp_async_16(v_dst + off, p.v + row * kHeadDim + c * 8, n);
      }
      describe();
    }
    ptx::cp_async_commit();
  }
};

template <typename T, int HKV>
__global__ void __launch_bounds__(kThreads, 1) decode_kernel(const Params p) {
  constexpr int kWph = kWarps / HKV;  // warps per key/value head
  constexpr int kTile = kTileRows / HKV;
  extern __shared__ __align__(1024) uint8_t smem[];
  float *red_m = reinterpret_cast<float *>(smem + kStages * kStageBytes);
  float *red_l = red_m + kWarps * 16;
  float *red_acc = red_l + HKV * 16;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int hk = warp / kWph, sub = warp % kWph;
  const int gid = lane >> 2, tq = lane & 3;

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
    if (tid == 0 && blockIdx.x == 0) flag(p.image, PKD_DEVICE_BAD_PLAN);
    return;
  }
  const int32_t *cta_ptr = img + kHeaderWords;
  const int32_t *units = cta_ptr + num_ctas + 1;
  const int u_begin = cta_ptr[blockIdx.x], u_end = cta_ptr[blockIdx.x + 1];
  if (u_begin < 0 || u_end > num_units || u_begin > u_end) {
    if (tid == 0) flag(p.image, PKD_DEVICE_BAD_PLAN);
    return;
  }
  if (u_begin == u_end) return;

  if (kWph > 1) {
    for (int i = tid; i < HKV * 16 * (kHeadDim + 1); i += kThreads) red_l[i] = 0.f;
  }

  Pipeline<HKV> pipe(p, units, num_partials, u_begin, u_end);
#pragma unroll
  for (int s = 0; s < kStages - 1; ++s) pipe.issue(smem + s * kStageBytes);

  // per-lane ldmatrix addressing (token within the warp's 16, swizzle key)
  const int k_tok = (lane & 7) + ((lane >> 4) << 3);
  const int k_hi = (lane >> 3) & 1;
  const int v_tok = (lane & 7) + (((lane >> 3) & 1) << 3);
  const int v_hi = lane >> 4;
  const int sw = lane & 7;
  const int slot_floats = static_cast<int>(partial_slot_floats(p.hq, kHeadDim));

  int stage = 0;
  for (int u = u_begin; u < u_end; ++u) {
    const Unit unit = read_unit(p, units, u, num_partials);

    // query fragments: rows are the group's heads (zero past g)
    uint32_t qf[8][4];
    {
      const int r0 = gid, r1 = gid + 8;
      const uint16_t *q0 = p.q + (static_cast<long long>(max(unit.req, 0)) * p.hq +
                                  hk * p.group + r0) * kHeadDim;
      const uint16_t *q1 = q0 + 8 * kHeadDim;
      const bool ok0 = unit.req >= 0 && r0 < p.group;
      const bool ok1 = unit.req >= 0 && r1 < p.group;
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        const int d = kk * 16 + 2 * tq;
        qf[kk][0] = ok0 ? __ldg(reinterpret_cast<const uint32_t *>(q0 + d)) : 0u;
        qf[kk][1] = ok1 ? __ldg(reinterpret_cast<const uint32_t *>(q1 + d)) : 0u;
        qf[kk][2] = ok0 ? __ldg(reinterpret_cast<const uint32_t *>(q0 + d + 8)) : 0u;
        qf[kk][3] = ok1 ? __ldg(reinterpret_cast<const uint32_t *>(q1 + d + 8)) : 0u;
      }
    }

    float m[2] = {-INFINITY, -INFINITY};  // running max of the raw logits
    float l[2] = {0.f, 0.f};              // this lane's share of the row sums
    float acc[16][4];
#pragma unroll
    for (int j = 0; j < 16; ++j) acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.f;

    const int ntiles = (unit.t1 - unit.t0 + kTile - 1) / kTile;
    for (int it = 0; it < ntiles; ++it) {
      ptx::cp_async_wait<kStages - 2>();
      __syncthreads();
      pipe.issue(smem + ((stage + kStages - 1) % kStages) * kStageBytes);

      const uint8_t *sk = smem + stage * kStageBytes;
      const uint32_t kbase =
          ptx::smem_u32(sk) + (hk * kTile + sub * 16) * kRowBytes;
      const uint32_t vbase = kbase + kTensorTileBytes;
      const int valid = min(kTile, unit.t1 - unit.t0 - it * kTile) - sub * 16;

      // S = Q K^T over this warp's 16 tokens
      float s[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        uint32_t b0, b1, b2, b3;
        ptx::ldmatrix_x4(kbase + k_tok * kRowBytes + (((2 * kk + k_hi) ^ sw) << 4),
                         b0, b1, b2, b3);
        ptx::mma_16816<T>(s[0], qf[kk], b0, b1);
        ptx::mma_16816<T>(s[1], qf[kk], b2, b3);
      }

      // online softmax (rows gid and gid + 8).  Maxima are kept on the raw
      // logits; the scaled difference s * c - m * c is formed inside one fma so
      // only that small difference is rounded, and a row whose maximum is
      // still -inf uses reference 0 (clamp: no -inf - (-inf)).
      float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
      for (int n = 0; n < 2; ++n)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int tok = n * 8 + 2 * tq + (i & 1);
          if (tok >= valid) s[n][i] = -INFINITY;
          mx[i >> 1] = fmaxf(mx[i >> 1], s[n][i]);
        }
      float ref[2], alpha[2];
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 1));
        mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 2));
        const float mn = fmaxf(m[r], mx[r]);
        ref[r] = mn == -INFINITY ? 0.f : mn * p.scale_log2;
        alpha[r] = exp2f(fmaf(m[r], p.scale_log2, -ref[r]));
        m[r] = mn;
      }
      // P as the A operand of P V.  bfloat16 keeps only 8 significant bits,
      // so for it P is split into hi + lo (both bf16) and multiplied twice;
      // half P is used once.  Row sums are taken over the values multiplied.
      constexpr bool kSplitP = std::is_same<T, __nv_bfloat16>::value;
      uint32_t pa[4], pb[4];
      float rs[2] = {0.f, 0.f};
#pragma unroll
      for (int n = 0; n < 2; ++n)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const float e0 = exp2f(fmaf(s[n][2 * h], p.scale_log2, -ref[h]));
          const float e1 = exp2f(fmaf(s[n][2 * h + 1], p.scale_log2, -ref[h]));
          const uint32_t hi = ptx::pack2<T>(e0, e1);
          const float2 back = ptx::unpack2<T>(hi);
          pa[2 * n + h] = hi;
          if (kSplitP) {
            const uint32_t lo = ptx::pack2<T>(e0 - back.x, e1 - back.y);
            const float2 back_lo = ptx::unpack2<T>(lo);
            pb[2 * n + h] = lo;
            rs[h] += (back.x + back_lo.x) + (back.y + back_lo.y);
          } else {
            pb[2 * n + h] = 0u;
            rs[h] += back.x + back.y;
          }
        }
#pragma unroll
      for (int r = 0; r < 2; ++r) l[r] = l[r] * alpha[r] + rs[r];
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        acc[j][0] *= alpha[0];
        acc[j][1] *= alpha[0];
        acc[j][2] *= alpha[1];
        acc[j][3] *= alpha[1];
      }

      // O += P V
#pragma unroll
      for (int jj = 0; jj < 16; jj += 2) {
        uint32_t b0, b1, b2, b3;
        ptx::ldmatrix_x4_trans(
            vbase + v_tok * kRowBytes + (((jj + v_hi) ^ sw) << 4), b0, b1, b2, b3);
        ptx::mma_16816<T>(acc[jj], pa, b0, b1);
        ptx::mma_16816<T>(acc[jj + 1], pa, b2, b3);
        if (kSplitP) {
          ptx::mma_16816<T>(acc[jj], pb, b0, b1);
          ptx::mma_16816<T>(acc[jj + 1], pb, b2, b3);
        }
      }
      stage = (stage + 1) % kStages;
    }

    // row totals of l across the quad
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      l[r] += __shfl_xor_sync(0xffffffffu, l[r], 1);
      l[r] += __shfl_xor_sync(0xffffffffu, l[r], 2);
    }

    bool writer = true;
    if (kWph > 1) {
      // combine the warps that share this head: rescale to the common max
      if (tq == 0) {
        red_m[warp * 16 + gid] = m[0];
        red_m[warp * 16 + gid + 8] = m[1];
      }
      __syncthreads();
      float f[2];
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        float mm = -INFINITY;
#pragma unroll
        for (int w = 0; w < kWph; ++w)
          mm = fmaxf(mm, red_m[(hk * kWph + w) * 16 + gid + 8 * r]);
        const float rf = mm == -INFINITY ? 0.f : mm * p.scale_log2;
        f[r] = exp2f(fmaf(m[r], p.scale_log2, -rf));
        m[r] = mm;
      }
      float *acc_h = red_acc + hk * 16 * kHeadDim;
#pragma unroll
      for (int j = 0; j < 16; ++j)
#pragma unroll
        for (int i = 0; i < 4; ++i)
          atomicAdd(acc_h + (gid + 8 * (i >> 1)) * kHeadDim + 8 * j + 2 * tq + (i & 1),
                    acc[j][i] * f[i >> 1]);
      if (tq == 0) {
        atomicAdd(red_l + hk * 16 + gid, l[0] * f[0]);
        atomicAdd(red_l + hk * 16 + gid + 8, l[1] * f[1]);
      }
      __syncthreads();
      writer = sub == 0;
      if (writer) {
#pragma unroll
        for (int j = 0; j < 16; ++j)
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            float *cell =
                acc_h + (gid + 8 * (i >> 1)) * kHeadDim + 8 * j + 2 * tq + (i & 1);
            acc[j][i] = *cell;
            *cell = 0.f;
          }
        l[0] = red_l[hk * 16 + gid];
        l[1] = red_l[hk * 16 + gid + 8];
      }
      __syncthreads();
      if (writer && tq == 0) {
        red_l[hk * 16 + gid] = 0.f;
        red_l[hk * 16 + gid + 8] = 0.f;
      }
    }

    if (writer && unit.req >= 0) {
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        const int row = gid + 8 * r;
        if (row >= p.group) continue;
        const int head = hk * p.group + row;
        const float inv = l[r] > 0.f ? 1.f / l[r] : 0.f;
        const float lse_r =
            l[r] > 0.f ? fmaf(m[r], p.scale_log2, log2f(l[r])) * kLn2 : -INFINITY;
        if (unit.slot < 0) {
          uint16_t *o = p.out + (static_cast<long long>(unit.req) * p.hq + head) * kHeadDim;
#pragma unroll
          for (int j = 0; j < 16; ++j)
            *reinterpret_cast<uint32_t *>(o + 8 * j + 2 * tq) =
                ptx::pack2<T>(acc[j][2 * r] * inv, acc[j][2 * r + 1] * inv);
          if (tq == 0) p.lse[static_cast<long long>(unit.req) * p.hq + head] = lse_r;
        } else {
          float *base = p.partials + static_cast<long long>(unit.slot) * slot_floats;
          float *o = base + head * kHeadDim;
#pragma unroll
          for (int j = 0; j < 16; ++j)
            *reinterpret_cast<float2 *>(o + 8 * j + 2 * tq) =
                make_float2(acc[j][2 * r] * inv, acc[j][2 * r + 1] * inv);
          if (tq == 0) base[p.hq * kHeadDim + head] = lse_r;
        }
      }
    }
  }
  ptx::cp_async_wait<0>();
}

template <typename T, int HKV>
int launch_typed(const Params &prm, int grid, void *stream) {
  constexpr int kWph = kWarps / HKV;
  const int smem = kStages * kStageBytes +
                   (kWph > 1 ? (kWarps * 16 + HKV * 16 * (1 + kHeadDim)) * 4 : 0);
  auto kernel = decode_kernel<T, HKV>;
  cudaError_t e = cudaFuncSetAttribute(
      kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  kernel<<<grid, kThreads, smem, static_cast<cudaStream_t>(stream)>>>(prm);
  return cudaGetLastError();
}

template <typename T>
int launch_heads(const Params &prm, int hkv, int grid, void *stream) {
  switch (hkv) {
    case 1: return launch_typed<T, 1>(prm, grid, stream);
    case 2: return launch_typed<T, 2>(prm, grid, stream);
    case 4: return launch_typed<T, 4>(prm, grid, stream);
    default: return launch_typed<T, 8>(prm, grid, stream);
  }
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
  if (a.dtype == PKD_BF16)
    return launch_heads<__nv_bfloat16>(prm, a.num_kv_heads, a.num_ctas, stream);
  return launch_heads<__half>(prm, a.num_kv_heads, a.num_ctas, stream);
}

}  // namespace pkd

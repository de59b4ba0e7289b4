// Device helpers shared by the attention kernels.
#pragma once

#include <cstdint>

#include "pkd_internal.h"
#include "ptx.cuh"

namespace pkd {

constexpr int kTile = 16;                 // tokens per 16-row mma tile
constexpr int kRowBytes = kHeadDim * 2;   // one token of one head
constexpr int kHalfBytes = kTile * 128;   // 16 rows x 64 elements
constexpr float kLn2 = 0.69314718055994530942f;
constexpr float kLazy = 8.f;              // log2 of the largest unnormalised p
constexpr long long kWaitPolls = 1ll << 22;  // bounded mbarrier waits

// Records a failed check in a plan image's status word.
__device__ __forceinline__ void flag(int32_t *image, unsigned bit) {
  atomicOr(reinterpret_cast<unsigned int *>(image + kHStatus), bit);
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

// Byte offset of 16-byte chunk c (0..15) of token row r (0..15) within one
// head's 16-token K or V tile: [d-half][row][128 B], chunks XOR-swizzled by
// row as the TMA 128-byte swizzle lays them out.
__device__ __forceinline__ uint32_t tile_offset(int r, int c) {
  return (c >> 3) * kHalfBytes + r * 128 + (((c & 7) ^ (r & 7)) << 4);
}

}  // namespace pkd

// bwd_tiles.cuh -- the query-tile walk shared by the head_dim 64/128 backward
// kernels (one CTA per key tile, and CTA pairs over two key tiles).
#pragma once

#include "ring_attn_internal.h"

namespace ra {

// Query tiles of the CTA's pairs.  Tiles of a range start at the range start
// rounded down to a multiple of 4, so the LSE/Delta slice of every tile is a
// 16-byte aligned TMA load; columns before the range start are masked.
struct PairList {
  int qb0, qe0, qb1, qe1, n0, nt, G, hbase;
  __device__ __forceinline__ int tile(int i) const { return i % nt; }
  __device__ __forceinline__ int head(int i) const { return hbase + i / nt; }
  __device__ __forceinline__ int start(int i) const {
    const int t = tile(i);
    return t < n0 ? (qb0 & ~3) + 128 * t : (qb1 & ~3) + 128 * (t - n0);
  }
  __device__ __forceinline__ int lo(int i) const { return tile(i) < n0 ? qb0 : qb1; }
  __device__ __forceinline__ int end(int i) const { return tile(i) < n0 ? qe0 : qe1; }
};

__device__ __forceinline__ int ceil128(int a, int b) { return b > a ? (b - a + 127) / 128 : 0; }

__device__ __forceinline__ void red_add_v4(float* addr, float a, float b, float c, float d) {
  asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(addr), "f"(a), "f"(b), "f"(c), "f"(d)
               : "memory");
}

}  // namespace ra

// The 16-query tile of the main branch: union of the tile's block selections.
//
// A tile is 16 consecutive queries of one KV group (they always fall in the same 64-token
// block); with G <= 8 heads their rows fill one 128-row UMMA tile.  The tile's selections are
// sorted as (block, query, slot) keys by one warp; the distinct blocks form the tile's union and
// each gets a mask of the queries that selected it.  A block selected by kSharedMin or more of
// the tile's queries is "shared" and is processed once for the tile; the selections of any other
// block are "private" and go to the block-major (KV-outer) pass.
#pragma once

#include <climits>
#include <type_traits>

#include "msa_device.cuh"

namespace msa {

constexpr int kTileQ = 16;         // queries per tile
constexpr int kMaxSel = 64;        // largest k supported
constexpr int kMaxKeys = kTileQ * kMaxSel;
// A block is processed once for the tile ("shared") when at least kSharedMin of the tile's
// queries selected it; otherwise each of its selections goes to the block-major pass, which
// packs full 128-row tiles (main branch at 128K: 7.10 ms with 3, 8.00 ms with 2, 6.94-6.95 ms
// with 4, 5, 6 or 8).
constexpr int kSharedMin = 4;
constexpr int kMaxShared = kMaxKeys / 2;   // a shared block holds at least two selections

// Keys per lane for a tile's 16*k selections (a power of two, 32*EPL >= 16*k).
template <typename F>
__device__ __forceinline__ auto with_epl(int kk, F&& f) {
  if (kk <= 2) return f(std::integral_constant<int, 1>());
  if (kk <= 4) return f(std::integral_constant<int, 2>());
  if (kk <= 8) return f(std::integral_constant<int, 4>());
  if (kk <= 16) return f(std::integral_constant<int, 8>());
  if (kk <= 32) return f(std::integral_constant<int, 16>());
  return f(std::integral_constant<int, 32>());
}
constexpr unsigned kAllLanes = 0xffffffffu;

// Ascending bitonic sort of the 32*EPL keys a warp holds lane-major (element EPL*lane + j).
template <int EPL>
__device__ __forceinline__ void warp_sort(int (&x)[EPL]) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int size = 2; size <= 32 * EPL; size <<= 1) {
#pragma unroll
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      int nx[EPL];
#pragma unroll
      for (int j = 0; j < EPL; ++j) {
        const int e = EPL * lane + j;
        const int other =
            stride < EPL ? x[j ^ stride] : __shfl_xor_sync(kAllLanes, x[j], stride / EPL);
        const bool lower = (e & stride) == 0, asc = (e & size) == 0;
        nx[j] = (lower == asc) ? min(x[j], other) : max(x[j], other);
      }
#pragma unroll
      for (int j = 0; j < EPL; ++j) x[j] = nx[j];
    }
  }
}

// Sorted selection keys of one tile: key = block << 10 | query-in-tile << 6 | slot, INT_MAX for
// padding, -1 entries and blocks after the query's own block (block < 2^21).  Queries at or
// after i_end are not part of the tile.
struct TileKeys {
  __device__ static int block(int key) { return key >> 10; }
  __device__ static int query(int key) { return (key >> 6) & 15; }
  __device__ static int slot(int key) { return key & 63; }
};

// Loads and sorts the tile's keys, then builds the union: s_U[0..nU) ascending distinct blocks,
// s_mask[u] = queries that selected s_U[u].  rank[j] is the union slot of key x[j].  Whole warp.
template <int EPL>
__device__ __forceinline__ int tile_union(const int32_t* __restrict__ idx, int r, int64_t i0,
                                          int64_t i_end, int64_t N, int kk, int (&x)[EPL],
                                          int (&rank)[EPL], int* s_U, unsigned* s_mask) {
  const int lane = threadIdx.x & 31;
  const int n = kTileQ * kk;
#pragma unroll
  for (int j = 0; j < EPL; ++j) {
    const int e = EPL * lane + j;
    int key = INT_MAX;
    if (e < n) {
      const int w = e / kk, t = e - w * kk;
      const int64_t i = i0 + w;
      if (i < i_end) {
        const int b = __ldg(idx + ((int64_t)r * N + i) * kk + t);
        if (b >= 0 && (int64_t)b <= (i >> 6)) key = (b << 10) | (w << 6) | t;
      }
    }
    x[j] = key;
  }
  warp_sort<EPL>(x);
  int prev = __shfl_up_sync(kAllLanes, x[EPL - 1], 1);
  if (lane == 0) prev = INT_MIN;
  int head[EPL], cnt = 0;
#pragma unroll
  for (int j = 0; j < EPL; ++j) {
    const int pk = j ? x[j - 1] : prev;
    head[j] = x[j] != INT_MAX && (pk == INT_MIN || (pk >> 10) != (x[j] >> 10));
    cnt += head[j];
  }
  int incl = cnt;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int t = __shfl_up_sync(kAllLanes, incl, o);
    if (lane >= o) incl += t;
  }
  const int nU = __shfl_sync(kAllLanes, incl, 31);
  int run = incl - cnt;
#pragma unroll
  for (int j = 0; j < EPL; ++j) {
    run += head[j];
    rank[j] = run - 1;
    if (head[j]) {
      s_U[rank[j]] = x[j] >> 10;
      s_mask[rank[j]] = 0u;
    }
  }
  __syncwarp();
#pragma unroll
  for (int j = 0; j < EPL; ++j)
    if (x[j] != INT_MAX) atomicOr(&s_mask[rank[j]], 1u << ((x[j] >> 6) & 15));
  __syncwarp();
  return nU;
}

}  // namespace msa

// Work planning of the sparse main branch («MiniMax-M3：MSA 技术报告速读», section 主分支
// eq. O^(h)_i; the kernel section's pre-scheduled work with a two-stage merge and no atomic
// updates of results).
//
//   k_attn_plan (pass 0)  per 16-query tile: count each private selection in its (group, block)
//                         bucket (a block that fewer than kSharedMin of the tile's queries
//                         selected)
//   k_attn_scan           exclusive scans: entry offsets and work-tile offsets per bucket
//   k_attn_plan (pass 1)  scatter private selections into their buckets, and record per tile its
//                         shared blocks (block << 16 | query mask) and per query its private
//                         slots, which the shared-block pass reads instead of rebuilding them
// The block-major pass writes the partial of (row, slot) at a fixed position of that row and
// slot; the merge itself is the epilogue of k_attn_shared, which finds a row's private slots
// from its own union of the tile.  Bucket order is decided by integer atomics and does not
// affect any result: every partial is computed independently and the merge visits partials in
// slot order.
#include <cmath>

#include "attn_tile.cuh"
#include "msa_internal.h"

namespace msa {
namespace {

constexpr int kPlanWarps = 4;

template <int EPL>
__device__ __forceinline__ void plan_tile(const int32_t* __restrict__ idx, int r, int64_t i0,
                                          int64_t q0, int64_t q1, int64_t N, int kk,
                                          int64_t nblk, int pass, int* s_U, unsigned* s_mask,
                                          unsigned long long* s_pm, int* count, const int* offset,
                                          int* cursor, int* entries, int* tile_list,
                                          unsigned long long* tile_priv) {
  const int lane = threadIdx.x & 31;
  int x[EPL], rank[EPL];
  if (pass == 1 && lane < kTileQ) s_pm[lane] = 0ull;
  const int nU = tile_union<EPL>(idx, r, i0, q1, N, kk, x, rank, s_U, s_mask);
  if (pass == 1) {
    const int64_t tix = (int64_t)r * ((q1 - q0 + kTileQ - 1) / kTileQ) + (i0 - q0) / kTileQ;
    int* lst = tile_list + tix * (kMaxShared + 1);
    int nS = 0;
    for (int base = 0; base < nU; base += 32) {
      const int u = base + lane;
      const unsigned m = u < nU ? s_mask[u] : 0u;
      const bool keep = __popc(m) >= kSharedMin;
      const unsigned kb = __ballot_sync(kAllLanes, keep);
      if (keep) lst[1 + nS + __popc(kb & ((1u << lane) - 1u))] = (s_U[u] << 16) | (int)m;
      nS += __popc(kb);
    }
    if (lane == 0) lst[0] = nS;
#pragma unroll
    for (int j = 0; j < EPL; ++j)
      if (x[j] != INT_MAX && __popc(s_mask[rank[j]]) < kSharedMin)
        atomicOr(&s_pm[TileKeys::query(x[j])], 1ull << TileKeys::slot(x[j]));
    __syncwarp();
    if (lane < kTileQ) tile_priv[tix * kTileQ + lane] = s_pm[lane];
  }
#pragma unroll
  for (int j = 0; j < EPL; ++j) {
    const int key = x[j];
    if (key == INT_MAX || __popc(s_mask[rank[j]]) >= kSharedMin) continue;
    const int b = TileKeys::block(key), w = TileKeys::query(key), t = TileKeys::slot(key);
    const int64_t bucket = (int64_t)r * nblk + b;
    if (pass == 0) {
      atomicAdd(count + bucket, 1);
    } else {
      const int pos = offset[bucket] + atomicAdd(cursor + bucket, 1);
      const int64_t li = i0 - q0 + w;
      entries[pos] = (int)((li << 6) | t);
    }
  }
}

__global__ void __launch_bounds__(32 * kPlanWarps)
    k_attn_plan(const int32_t* __restrict__ idx, int64_t N, int kk, int64_t q0, int64_t q1,
                int64_t nblk, int pass, int* count, const int* offset, int* cursor,
                int* entries, int* tile_list, unsigned long long* tile_priv) {
  __shared__ int s_U[kPlanWarps][kMaxKeys];
  __shared__ unsigned s_mask[kPlanWarps][kMaxKeys];
  __shared__ unsigned long long s_pm[kPlanWarps][kTileQ];
  const int warp = threadIdx.x >> 5;
  const int r = blockIdx.y;
  const int64_t i0 = q0 + ((int64_t)blockIdx.x * kPlanWarps + warp) * kTileQ;
  if (i0 >= q1) return;
  int* U = s_U[warp];
  unsigned* Mk = s_mask[warp];
  with_epl(kk, [&](auto e) {
    plan_tile<decltype(e)::value>(idx, r, i0, q0, q1, N, kk, nblk, pass, U, Mk, s_pm[warp], count,
                                  offset, cursor, entries, tile_list, tile_priv);
    return 0;
  });
}

// One CTA: offset[b] = sum_{b'<b} count[b'], tile_off[b] = sum_{b'<b} ceil(count[b'] / ept),
// with the totals in entry nb; cursor[] cleared for pass 1.
constexpr int kScanThreads = 1024;

__global__ void __launch_bounds__(kScanThreads)
    k_attn_scan(const int* __restrict__ count, int* offset, int* tile_off, int* cursor, int nb,
                int ept) {
  __shared__ int s_a[kScanThreads], s_t[kScanThreads];
  const int tid = threadIdx.x;
  const int per = (nb + kScanThreads - 1) / kScanThreads;
  const int beg = min(nb, tid * per), end = min(nb, beg + per);
  int sa = 0, st = 0;
  for (int b = beg; b < end; ++b) {
    const int c = count[b];
    sa += c;
    st += (c + ept - 1) / ept;
  }
  s_a[tid] = sa;
  s_t[tid] = st;
  __syncthreads();
  for (int o = 1; o < kScanThreads; o <<= 1) {        // inclusive Hillis-Steele scan
    const int va = tid >= o ? s_a[tid - o] : 0;
    const int vt = tid >= o ? s_t[tid - o] : 0;
    __syncthreads();
    s_a[tid] += va;
    s_t[tid] += vt;
    __syncthreads();
  }
  int ra = s_a[tid] - sa, rt = s_t[tid] - st;
  for (int b = beg; b < end; ++b) {
    const int c = count[b];
    offset[b] = ra;
    tile_off[b] = rt;
    cursor[b] = 0;
    ra += c;
    rt += (c + ept - 1) / ept;
  }
  if (tid == kScanThreads - 1) {
    offset[nb] = s_a[tid];
    tile_off[nb] = s_t[tid];
  }
}

}  // namespace

cudaError_t launch_attn_plan(const int32_t* idx, int64_t N, int H_kv, int kk, int64_t q0,
                             int64_t q1, int64_t nblk, int pass, int* count, const int* offset,
                             int* cursor, int* entries, int* tile_list,
                             unsigned long long* tile_priv, cudaStream_t st) {
  const int64_t tiles = (q1 - q0 + kTileQ - 1) / kTileQ;
  const dim3 grid((unsigned)((tiles + kPlanWarps - 1) / kPlanWarps), (unsigned)H_kv);
  k_attn_plan<<<grid, 32 * kPlanWarps, 0, st>>>(idx, N, kk, q0, q1, nblk, pass, count, offset,
                                                cursor, entries, tile_list, tile_priv);
  return cudaGetLastError();
}

cudaError_t launch_attn_scan(const int* count, int* offset, int* tile_off, int* cursor, int nb,
                             int ept, cudaStream_t st) {
  k_attn_scan<<<1, kScanThreads, 0, st>>>(count, offset, tile_off, cursor, nb, ept);
  return cudaGetLastError();
}

}  // namespace msa

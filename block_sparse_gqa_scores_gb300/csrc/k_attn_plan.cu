// Work planning of the sparse main branch («MiniMax-M3：MSA 技术报告速读», section 主分支
// eq. O^(h)_i; the kernel section's pre-scheduled work with a two-stage merge and no atomic
// updates of results).
//
//   k_attn_plan      per 16-query tile (one warp): sort the tile's selections and build its
//                    union; record its shared blocks (block << 16 | query mask) and per query
//                    its private slots, which the shared-block pass reads instead of rebuilding
//                    them; give each private selection (a block that fewer than kSharedMin of
//                    the tile's queries selected) its rank in its (group, block) bucket and note
//                    (bucket, rank, entry) in the tile's own scratch region
//   k_attn_scan      exclusive scans: entry offsets and work-tile offsets per bucket
//   k_attn_scatter   per tile: entries[offset[bucket] + rank] = entry
// The block-major pass writes the partial of (row, slot) at a fixed position of that row and
// slot; the merge itself is the epilogue of k_attn_shared.  The order inside a bucket is decided
// by integer atomics and does not affect any result: every partial is computed independently
// and the merge visits partials in slot order.
#include <cmath>

#include "attn_tile.cuh"
#include "msa_internal.h"

namespace msa {
namespace {

constexpr int kPlanWarps = 4;

// One warp per tile; the kernel is instantiated per keys-per-lane EPL (32 EPL >= 16 k), so its
// registers and shared memory fit the k in use.
template <int EPL>
__global__ void __launch_bounds__(32 * kPlanWarps)
    k_attn_plan(const int32_t* __restrict__ idx, int64_t N, int kk, int64_t q0, int64_t q1,
                int64_t nblk, int* count, int* tile_list, unsigned long long* tile_priv,
                int* sc, int* sc_n) {
  __shared__ int s_U[kPlanWarps][32 * EPL];
  __shared__ unsigned s_mask[kPlanWarps][32 * EPL];
  __shared__ unsigned long long s_pm[kPlanWarps][kTileQ];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r = blockIdx.y;
  const int64_t ntl = (q1 - q0 + kTileQ - 1) / kTileQ;          // tiles per group
  const int64_t tl = (int64_t)blockIdx.x * kPlanWarps + warp;
  const int64_t i0 = q0 + tl * kTileQ;
  if (tl >= ntl) return;
  const int64_t tix = (int64_t)r * ntl + tl;
  int* U = s_U[warp];
  unsigned* Mk = s_mask[warp];
  unsigned long long* pm = s_pm[warp];
  int x[EPL], rank[EPL];
  if (lane < kTileQ) pm[lane] = 0ull;
  const int nU = tile_union<EPL>(idx, r, i0, q1, N, kk, x, rank, U, Mk);
  // shared blocks
  int* lst = tile_list + tix * (kMaxShared + 1);
  int nS = 0;
  for (int base = 0; base < nU; base += 32) {
    const int u = base + lane;
    const unsigned m = u < nU ? Mk[u] : 0u;
    const bool keep = __popc(m) >= kSharedMin;
    const unsigned kb = __ballot_sync(kAllLanes, keep);
    if (keep) lst[1 + nS + __popc(kb & ((1u << lane) - 1u))] = (U[u] << 16) | (int)m;
    nS += __popc(kb);
  }
  if (lane == 0) lst[0] = nS;
  // private selections: slot masks, bucket ranks, scratch triples
  int* tsc = sc + tix * (int64_t)(kTileQ * kk) * 3;
  int np = 0;
#pragma unroll
  for (int j = 0; j < EPL; ++j) {
    const int key = x[j];
    const bool priv = key != INT_MAX && __popc(Mk[rank[j]]) < kSharedMin;
    const unsigned pb = __ballot_sync(kAllLanes, priv);
    if (priv) {
      const int b = TileKeys::block(key), w = TileKeys::query(key), t = TileKeys::slot(key);
      atomicOr(&pm[w], 1ull << t);
      const int bucket = (int)((int64_t)r * nblk + b);
      const int li = np + __popc(pb & ((1u << lane) - 1u));
      tsc[3 * li] = bucket;
      tsc[3 * li + 1] = atomicAdd(count + bucket, 1);
      tsc[3 * li + 2] = (int)(((i0 - q0 + w) << 6) | t);
    }
    np += __popc(pb);
  }
  __syncwarp();
  if (lane < kTileQ) tile_priv[tix * kTileQ + lane] = pm[lane];
  if (lane == 0) sc_n[tix] = np;
}

// One CTA: offset[b] = sum_{b'<b} count[b'], tile_off[b] = sum_{b'<b} ceil(count[b'] / ept),
// with the totals in entry nb.
constexpr int kScanThreads = 1024;

__global__ void __launch_bounds__(kScanThreads)
    k_attn_scan(const int* __restrict__ count, int* offset, int* tile_off, int nb, int ept) {
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
    ra += c;
    rt += (c + ept - 1) / ept;
  }
  if (tid == kScanThreads - 1) {
    offset[nb] = s_a[tid];
    tile_off[nb] = s_t[tid];
  }
}

// One warp per tile: each private selection to its place in its bucket.
constexpr int kScatterWarps = 8;

__global__ void __launch_bounds__(32 * kScatterWarps)
    k_attn_scatter(const int* __restrict__ sc, const int* __restrict__ sc_n,
                   const int* __restrict__ offset, int* entries, int64_t ntiles, int per_tile) {
  const int64_t t = (int64_t)blockIdx.x * kScatterWarps + (threadIdx.x >> 5);
  if (t >= ntiles) return;
  const int n = sc_n[t];
  const int* tsc = sc + t * (int64_t)per_tile * 3;
  for (int x = threadIdx.x & 31; x < n; x += 32)
    entries[offset[tsc[3 * x]] + tsc[3 * x + 1]] = tsc[3 * x + 2];
}

}  // namespace

cudaError_t launch_attn_plan(const int32_t* idx, int64_t N, int H_kv, int kk, int64_t q0,
                             int64_t q1, int64_t nblk, int* count, int* tile_list,
                             unsigned long long* tile_priv, int* sc, int* sc_n, cudaStream_t st) {
  const int64_t tiles = (q1 - q0 + kTileQ - 1) / kTileQ;
  const dim3 grid((unsigned)((tiles + kPlanWarps - 1) / kPlanWarps), (unsigned)H_kv);
  auto run = [&](auto kern) {
    kern<<<grid, 32 * kPlanWarps, 0, st>>>(idx, N, kk, q0, q1, nblk, count, tile_list, tile_priv,
                                           sc, sc_n);
    return cudaGetLastError();
  };
  if (kk <= 2) return run(k_attn_plan<1>);
  if (kk <= 4) return run(k_attn_plan<2>);
  if (kk <= 8) return run(k_attn_plan<4>);
  if (kk <= 16) return run(k_attn_plan<8>);
  if (kk <= 32) return run(k_attn_plan<16>);
  return run(k_attn_plan<32>);
}

cudaError_t launch_attn_scan(const int* count, int* offset, int* tile_off, int nb, int ept,
                             cudaStream_t st) {
  k_attn_scan<<<1, kScanThreads, 0, st>>>(count, offset, tile_off, nb, ept);
  return cudaGetLastError();
}

cudaError_t launch_attn_scatter(const int* sc, const int* sc_n, const int* offset, int* entries,
                                int64_t ntiles, int kk, cudaStream_t st) {
  const unsigned grid = (unsigned)((ntiles + kScatterWarps - 1) / kScatterWarps);
  k_attn_scatter<<<grid, 32 * kScatterWarps, 0, st>>>(sc, sc_n, offset, entries, ntiles,
                                                      kTileQ * kk);
  return cudaGetLastError();
}

}  // namespace msa

// Per-group top-k block selection with the forced local block («MiniMax-M3：MSA 技术报告速读»,
// section 索引分支: eq. I^(r)_i = TopK_b(M^idx,(r)_{i,.}, k) and the always-kept local block).
//
// Prefill: one warp per (group, query) row; decode: one CTA per row, its warps taking segments of
// the row (below).  Only comparisons, no exponentials.  Let l = floor(i/64)
// and K1 = k-1.  If l+1 <= k every visible block is taken.  Otherwise:
//   1. one coalesced pass keeps each lane's two largest scores among blocks b < l; the K1-th
//      largest of those 64 values (a warp bitonic sort) is an actual score with at least K1
//      scores >= it, so it bounds the K1-th best score from below;
//   2. a second pass appends every score >= that bound to a per-warp buffer in block order
//      (ballot compaction keeps the order);
//   3. the exact K1 best are those whose rank under (score desc, block asc) is < K1; if the
//      buffer would overflow, it is first reduced to its K1 best and later blocks must then
//      beat the K1-th kept score strictly (a later block loses every tie).
// The buffer stays in block order, so the K1 kept blocks come out ascending; l is appended.
#include <math.h>

#include "msa_device.cuh"
#include "msa_internal.h"

namespace msa {
namespace {

constexpr int kSelWarps = 8;
constexpr int kBuf = 160;          // candidate buffer entries per warp (5 per lane)
constexpr int kPerLane = kBuf / 32;
constexpr unsigned kFull = 0xffffffffu;

struct SelScratch {
  float v[kBuf];
  int b[kBuf];
};

// Value of the K1-th largest (1 <= K1 <= 64) of the 64 values held as (x0, x1) per lane.
__device__ __forceinline__ float kth_largest64(float x0, float x1, int K1) {
  const int lane = threadIdx.x & 31;
  float x[2] = {x0, x1};
#pragma unroll
  for (int size = 2; size <= 64; size <<= 1) {
#pragma unroll
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      float nx[2];
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int e = j * 32 + lane;
        const float other = stride == 32 ? x[j ^ 1] : __shfl_xor_sync(kFull, x[j], stride);
        const bool lower = (e & stride) == 0;
        const bool desc = (e & size) == 0;             // the final merge sorts descending
        nx[j] = (lower == desc) ? fmaxf(x[j], other) : fminf(x[j], other);
      }
      x[0] = nx[0];
      x[1] = nx[1];
    }
  }
  const int t = K1 - 1;
  return __shfl_sync(kFull, (t >> 5) ? x[1] : x[0], t & 31);
}

// Keeps the K1 best of buf[0..cnt) (score desc, position asc), in position order.
// Returns the score of the K1-th best (the weakest kept).
__device__ __forceinline__ float compact(SelScratch& sc, int cnt, int K1) {
  const int lane = threadIdx.x & 31;
  float mv[kPerLane];
  int mb[kPerLane], rank[kPerLane];
#pragma unroll
  for (int t = 0; t < kPerLane; ++t) {
    const int c = lane + 32 * t;
    mv[t] = c < cnt ? sc.v[c] : -INFINITY;
    mb[t] = c < cnt ? sc.b[c] : 0;
    rank[t] = 0;
  }
  for (int d = 0; d < cnt; ++d) {
    const float vd = sc.v[d];
#pragma unroll
    for (int t = 0; t < kPerLane; ++t) {
      const int c = lane + 32 * t;
      rank[t] += (vd > mv[t]) || (vd == mv[t] && d < c);
    }
  }
  __syncwarp();
  int base = 0;
  float tau = -INFINITY;
#pragma unroll
  for (int t = 0; t < kPerLane; ++t) {
    const int c = lane + 32 * t;
    const bool keep = c < cnt && rank[t] < K1;
    const unsigned m = __ballot_sync(kFull, keep);
    if (keep) {
      const int pos = base + __popc(m & ((1u << lane) - 1u));
      sc.v[pos] = mv[t];
      sc.b[pos] = mb[t];
    }
    base += __popc(m);
    const unsigned w = __ballot_sync(kFull, c < cnt && rank[t] == K1 - 1);
    if (w) tau = __shfl_sync(kFull, mv[t], __ffs(w) - 1);
  }
  __syncwarp();
  return tau;
}

// The K1 best of blocks [b0, b1) of a row (score desc, block asc), left in sc.v / sc.b in block
// order; returns how many (min(K1, b1 - b0)).  Whole warp.
__device__ int select_segment(const float* __restrict__ Mrow, int b0, int b1, int K1,
                              SelScratch& sc) {
  const int lane = threadIdx.x & 31;
  float a1 = -INFINITY, a2 = -INFINITY;
  for (int b = b0 + lane; b < b1; b += 32) {
    const float v = __ldg(Mrow + b);
    if (v > a1) {
      a2 = a1;
      a1 = v;
    } else if (v > a2) {
      a2 = v;
    }
  }
  // fewer than K1 candidates: the bound is -inf and every block is kept
  float tau = b1 - b0 > K1 ? kth_largest64(a1, a2, K1) : -INFINITY;
  bool strict = false;
  int cnt = 0;
  for (int base = b0; base < b1; base += 32) {
    const int b = base + lane;
    const float v = b < b1 ? __ldg(Mrow + b) : -INFINITY;
    bool pred = b < b1 && (strict ? v > tau : v >= tau);
    unsigned m = __ballot_sync(kFull, pred);
    if (cnt + __popc(m) > kBuf) {
      tau = compact(sc, cnt, K1);
      cnt = K1;
      strict = true;
      pred = b < b1 && v > tau;
      m = __ballot_sync(kFull, pred);
    }
    if (pred) {
      const int pos = cnt + __popc(m & ((1u << lane) - 1u));
      sc.v[pos] = v;
      sc.b[pos] = b;
    }
    cnt += __popc(m);
  }
  __syncwarp();
  if (cnt > K1) {
    compact(sc, cnt, K1);
    cnt = K1;
  }
  return cnt;
}

__device__ void select_row(const float* __restrict__ Mrow, int64_t l, int k,
                           int32_t* __restrict__ out, SelScratch& sc) {
  const int lane = threadIdx.x & 31;
  if (l + 1 <= k) {
    for (int c = lane; c < k; c += 32) out[c] = c <= l ? c : -1;
    return;
  }
  const int K1 = k - 1;
  const int n = (int)l;                                  // candidates: blocks 0 .. l-1
  float a1 = -INFINITY, a2 = -INFINITY;
  for (int b = lane; b < n; b += 32) {
    const float v = __ldg(Mrow + b);
    if (v > a1) {
      a2 = a1;
      a1 = v;
    } else if (v > a2) {
      a2 = v;
    }
  }
  float tau = kth_largest64(a1, a2, K1);
  bool strict = false;
  int cnt = 0;
  for (int base = 0; base < n; base += 32) {
    const int b = base + lane;
    const float v = b < n ? __ldg(Mrow + b) : -INFINITY;
    bool pred = b < n && (strict ? v > tau : v >= tau);
    unsigned m = __ballot_sync(kFull, pred);
    if (cnt + __popc(m) > kBuf) {
      tau = compact(sc, cnt, K1);
      cnt = K1;
      strict = true;
      pred = b < n && v > tau;
      m = __ballot_sync(kFull, pred);
    }
    if (pred) {
      const int pos = cnt + __popc(m & ((1u << lane) - 1u));
      sc.v[pos] = v;
      sc.b[pos] = b;
    }
    cnt += __popc(m);
  }
  __syncwarp();
  if (cnt > K1) {
    compact(sc, cnt, K1);
    cnt = K1;
  }
  for (int c = lane; c < K1; c += 32) out[c] = c < cnt ? sc.b[c] : -1;
  if (lane == 0) out[K1] = (int32_t)l;
}

__global__ void __launch_bounds__(32 * kSelWarps)
    k_select_prefill(const float* __restrict__ M, int32_t* __restrict__ idx, int64_t N, int k,
                     int64_t q_start, int64_t q_count, int64_t nrows, int64_t nblk) {
  __shared__ SelScratch sc[kSelWarps];
  const int warp = threadIdx.x >> 5;
  const int64_t row = (int64_t)blockIdx.x * kSelWarps + warp;   // row = r*q_count + t
  if (row >= nrows) return;
  const int64_t r = row / q_count, t = row - r * q_count, i = q_start + t;
  select_row(M + row * nblk, i >> 6, k, idx + (r * N + i) * k, sc[warp]);
}

// Decode: one CTA per (sequence, group) row.  The row's candidate blocks 0 .. l-1 are cut into
// up to kSelWarps segments; each warp keeps its segment's K1 best (select_segment), and warp 0
// keeps the K1 best of those, gathered in segment order (= block order), so the result is exactly
// the single-warp selection: every block of the row's K1 best is among its segment's K1 best
// under the same (score desc, block asc) order.
__global__ void __launch_bounds__(32 * kSelWarps)
    k_select_decode(const float* __restrict__ Mdec, int32_t* __restrict__ idx,
                    const CacheMap cm, int S, int H_kv, int k, int64_t max_len,
                    int64_t nblk_max) {
  __shared__ SelScratch sc[kSelWarps];
  __shared__ int s_cnt[kSelWarps];
  pdl_launch_dependents();
  pdl_wait();                                                   // the block scores are written
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t row = blockIdx.x;                               // row = s*H_kv + r
  const int64_t s = row / H_kv;
  const int64_t L = cm.pages ? cm.len<true>(s, max_len) : cm.len<false>(s, max_len);
  const int64_t l = (L - 1) >> 6;
  const float* Mrow = Mdec + row * nblk_max;
  int32_t* out = idx + row * k;
  if (l + 1 <= k) {
    if (warp == 0)
      for (int c = lane; c < k; c += 32) out[c] = c <= l ? c : -1;
    return;
  }
  const int K1 = k - 1;
  const int n = (int)l;
  // segments: as many as the merge buffer holds K1-long lists of, at most one per warp
  int nseg = kBuf / K1;
  nseg = nseg > kSelWarps ? kSelWarps : (nseg < 1 ? 1 : nseg);
  const int seg = (n + nseg - 1) / nseg;
  if (warp < nseg) {
    const int b0 = min(n, warp * seg), b1 = min(n, b0 + seg);
    const int cnt = b1 > b0 ? select_segment(Mrow, b0, b1, K1, sc[warp]) : 0;
    if (lane == 0) s_cnt[warp] = cnt;
  }
  __syncthreads();
  if (warp == 0) {
    // gather the segments' survivors after warp 0's own, in segment order
    int cnt = s_cnt[0];
    for (int w = 1; w < nseg; ++w) {
      const int c = s_cnt[w];
      for (int x = lane; x < c; x += 32) {
        sc[0].v[cnt + x] = sc[w].v[x];
        sc[0].b[cnt + x] = sc[w].b[x];
      }
      cnt += c;
    }
    __syncwarp();
    if (cnt > K1) {
      compact(sc[0], cnt, K1);
      cnt = K1;
    }
    for (int c = lane; c < K1; c += 32) out[c] = c < cnt ? sc[0].b[c] : -1;
    if (lane == 0) out[K1] = (int32_t)l;
  }
}

}  // namespace

cudaError_t launch_select_prefill(const float* M, int32_t* idx, int64_t N, int H_kv, int k,
                                  int64_t q_start, int64_t q_count, cudaStream_t stream) {
  const int64_t nrows = (int64_t)H_kv * q_count;
  const int64_t nblk = (N + kBlock - 1) / kBlock;
  const int64_t grid = (nrows + kSelWarps - 1) / kSelWarps;
  k_select_prefill<<<(unsigned)grid, 32 * kSelWarps, 0, stream>>>(M, idx, N, k, q_start, q_count,
                                                                  nrows, nblk);
  return cudaGetLastError();
}

cudaError_t launch_select_decode(const float* Mdec, int32_t* idx, const CacheMap& cm, int S,
                                 int H_kv, int k, int64_t max_len, int64_t nblk_max,
                                 cudaStream_t stream) {
  const int64_t nrows = (int64_t)S * H_kv;
  return launch_pdl(k_select_decode, dim3((unsigned)nrows), dim3(32 * kSelWarps), 0, stream, Mdec,
                    idx, cm, S, H_kv, k, max_len, nblk_max);
}

}  // namespace msa

// Top-k machinery of the block selection («MiniMax-M3：MSA 技术报告速读», section 索引分支:
// eq. I^(r)_i = TopK_b(M^idx,(r)_{i,.}, k)), shared by the prefill selection and the decode tail.
// Comparisons only; ties under (score desc, block asc) go to the lower block.
#pragma once

#include <math.h>

#include "msa_device.cuh"

namespace msa {
namespace sel {

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

// A lower bound on the K1-th best score of blocks [b0, b1) of a row: the K1-th largest of every
// lane's two best, all of them scores of the segment; -inf when the segment has at most K1
// blocks.  Whole warp.  SMEM: the row is a copy in shared memory (plain loads), else in global
// memory (read-only loads).
template <bool SMEM = false>
static __device__ float segment_bound(const float* __restrict__ Mrow, int b0, int b1, int K1) {
  const int lane = threadIdx.x & 31;
  float a1 = -INFINITY, a2 = -INFINITY;
  for (int b = b0 + lane; b < b1; b += 32) {
    const float v = SMEM ? Mrow[b] : __ldg(Mrow + b);
    if (v > a1) {
      a2 = a1;
      a1 = v;
    } else if (v > a2) {
      a2 = v;
    }
  }
  return b1 - b0 > K1 ? kth_largest64(a1, a2, K1) : -INFINITY;
}

// The K1 best (score desc, block asc) of the blocks of [b0, b1) that score at least tau0, left
// in sc.v / sc.b in block order; returns how many.  tau0 must not exceed the K1-th best score of
// the whole row, so that the row's K1 best blocks in this segment all pass.  Whole warp.
template <bool SMEM = false>
static __device__ int select_segment_from(const float* __restrict__ Mrow, int b0, int b1, int K1,
                                          float tau0, SelScratch& sc) {
  const int lane = threadIdx.x & 31;
  float tau = tau0;
  bool strict = false;
  int cnt = 0;
  for (int base = b0; base < b1; base += 32) {
    const int b = base + lane;
    const float v = b < b1 ? (SMEM ? Mrow[b] : __ldg(Mrow + b)) : -INFINITY;
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

// The K1 best of blocks [b0, b1) of a row (score desc, block asc), left in sc.v / sc.b in block
// order; returns how many (min(K1, b1 - b0)).  Whole warp.
template <bool SMEM = false>
static __device__ int select_segment(const float* __restrict__ Mrow, int b0, int b1, int K1,
                              SelScratch& sc) {
  return select_segment_from<SMEM>(Mrow, b0, b1, K1, segment_bound<SMEM>(Mrow, b0, b1, K1), sc);
}

}  // namespace sel
}  // namespace msa

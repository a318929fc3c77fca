// Per-group top-k block selection with the forced local block («MiniMax-M3：MSA 技术报告速读»,
// section 索引分支: eq. I^(r)_i = TopK_b(M^idx,(r)_{i,.}, k) and the always-kept local block).
//
// One warp per (group, query) row (the decode tail, k_attn.cu, runs the same machinery over
// segments of a row).  Only comparisons, no exponentials.  Let l = floor(i/64)
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

#include "msa_internal.h"
#include "select_core.cuh"

namespace msa {
namespace {

constexpr int kSelWarps = 8;
using namespace sel;

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

}  // namespace msa

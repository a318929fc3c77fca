// Work planning and the final merge of the sparse main branch («MiniMax-M3：MSA 技术报告速读»,
// section 主分支 eq. O^(h)_i; the kernel section's pre-scheduled work with a two-stage merge
// and no atomic updates of results).
//
//   k_attn_plan (pass 0)  per 8-query tile: count each private selection in its (group, block)
//                         bucket (a block that only one of the tile's queries selected)
//   k_attn_scan           exclusive scans: entry offsets and work-tile offsets per bucket
//   k_attn_plan (pass 1)  scatter private selections into their buckets; record, per (row,
//                         slot), where the block-major pass writes that slot's partial (-1 if the
//                         slot is empty or shared)
//   k_attn_merge          per (row, group): combine the shared-block partial and the private
//                         partials in slot order into O and the natural-log LSE
// Bucket order is decided by integer atomics and does not affect any result: every partial is
// computed independently and the merge visits partials in slot order.
#include <cmath>

#include "attn_tile.cuh"
#include "msa_internal.h"

namespace msa {
namespace {

constexpr int kPlanWarps = 4;

template <int EPL>
__device__ __forceinline__ void plan_tile(const int32_t* __restrict__ idx, int r, int64_t i0,
                                          int64_t q0, int64_t q1, int64_t N, int kk, int64_t qc,
                                          int64_t nblk, int pass, int* s_U, unsigned* s_mask,
                                          int* count, const int* offset, int* cursor, int* entries,
                                          int* slotmap) {
  const int lane = threadIdx.x & 31;
  int x[EPL], rank[EPL];
  tile_union<EPL>(idx, r, i0, q1, N, kk, x, rank, s_U, s_mask);
  if (pass == 1) {
    const int nq = (int)min((int64_t)kTileQ, q1 - i0);
    for (int e = lane; e < nq * kk; e += 32)
      slotmap[((int64_t)r * qc + (i0 - q0)) * kk + e] = -1;
    __syncwarp();
  }
#pragma unroll
  for (int j = 0; j < EPL; ++j) {
    const int key = x[j];
    if (key == INT_MAX || __popc(s_mask[rank[j]]) != 1) continue;
    const int b = TileKeys::block(key), w = TileKeys::query(key), t = TileKeys::slot(key);
    const int64_t bucket = (int64_t)r * nblk + b;
    if (pass == 0) {
      atomicAdd(count + bucket, 1);
    } else {
      const int pos = offset[bucket] + atomicAdd(cursor + bucket, 1);
      const int64_t li = i0 - q0 + w;
      entries[pos] = (int)((li << 6) | t);
      slotmap[((int64_t)r * qc + li) * kk + t] = pos;
    }
  }
}

__global__ void __launch_bounds__(32 * kPlanWarps)
    k_attn_plan(const int32_t* __restrict__ idx, int64_t N, int kk, int64_t q0, int64_t q1,
                int64_t qc, int64_t nblk, int pass, int* count, const int* offset, int* cursor,
                int* entries, int* slotmap) {
  __shared__ int s_U[kPlanWarps][kTileQ * kMaxSel];
  __shared__ unsigned s_mask[kPlanWarps][kTileQ * kMaxSel];
  const int warp = threadIdx.x >> 5;
  const int r = blockIdx.y;
  const int64_t i0 = q0 + ((int64_t)blockIdx.x * kPlanWarps + warp) * kTileQ;
  if (i0 >= q1) return;
  int* U = s_U[warp];
  unsigned* Mk = s_mask[warp];
  if (kk <= 4)
    plan_tile<1>(idx, r, i0, q0, q1, N, kk, qc, nblk, pass, U, Mk, count, offset, cursor, entries, slotmap);
  else if (kk <= 8)
    plan_tile<2>(idx, r, i0, q0, q1, N, kk, qc, nblk, pass, U, Mk, count, offset, cursor, entries, slotmap);
  else if (kk <= 16)
    plan_tile<4>(idx, r, i0, q0, q1, N, kk, qc, nblk, pass, U, Mk, count, offset, cursor, entries, slotmap);
  else if (kk <= 32)
    plan_tile<8>(idx, r, i0, q0, q1, N, kk, qc, nblk, pass, U, Mk, count, offset, cursor, entries, slotmap);
  else
    plan_tile<16>(idx, r, i0, q0, q1, N, kk, qc, nblk, pass, U, Mk, count, offset, cursor, entries, slotmap);
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

// One warp per (row, group).  Lane l owns EPL = G*D_H/32 consecutive elements of the group's
// [G, D_H] output, all inside head h = l*EPL / D_H.
template <int D_H, int G>
__global__ void __launch_bounds__(128)
    k_attn_merge(const __nv_bfloat16* __restrict__ tp_o, const float* __restrict__ tp_lse,
                 const int* __restrict__ slotmap, const __nv_bfloat16* __restrict__ part_o,
                 const float* __restrict__ part_lse, __nv_bfloat16* __restrict__ o,
                 float* __restrict__ lse, int64_t N, int H_q, int H_kv, int kk, int64_t q0,
                 int64_t q1) {
  constexpr int EPL = G * D_H / 32;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t qc = q1 - q0;
  const int64_t unit = (int64_t)blockIdx.x * 4 + warp;      // r * qc + li
  if (unit >= (int64_t)H_kv * qc) return;
  const int r = (int)(unit / qc);
  const int64_t li = unit - (int64_t)r * qc, i = q0 + li;
  const int h = lane * EPL / D_H, d0 = lane * EPL - h * D_H;
  const int* sm = slotmap + unit * kk;

  // pass 1: the largest partial LSE of this head
  float mx = tp_lse[unit * G + h];
  for (int t = 0; t < kk; ++t) {
    const int pos = sm[t];
    if (pos >= 0) mx = fmaxf(mx, part_lse[(int64_t)pos * G + h]);
  }
  // pass 2: weighted sum in slot order (the shared-block partial first)
  float acc[EPL];
#pragma unroll
  for (int e = 0; e < EPL; ++e) acc[e] = 0.f;
  float wsum = 0.f;
  // adds w * src[0..EPL) (bf16) to acc, 16-byte loads when the run allows it
  auto axpy = [&](float w, const __nv_bfloat16* src) {
    if constexpr (EPL % 8 == 0) {
#pragma unroll
      for (int e = 0; e < EPL; e += 8) {
        const uint4 u = *reinterpret_cast<const uint4*>(src + e);
        const uint32_t wd[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int k2 = 0; k2 < 4; ++k2) {
          const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&wd[k2]));
          acc[e + 2 * k2] += w * f.x;
          acc[e + 2 * k2 + 1] += w * f.y;
        }
      }
    } else {
#pragma unroll
      for (int e = 0; e < EPL; e += 2) {
        const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(src + e));
        acc[e] += w * f.x;
        acc[e + 1] += w * f.y;
      }
    }
  };
  {
    const float lt = tp_lse[unit * G + h];
    const float w = lt == -INFINITY ? 0.f : ex2(lt - mx);
    wsum += w;
    if (w > 0.f) axpy(w, tp_o + (unit * G + h) * D_H + d0);
  }
  for (int t = 0; t < kk; ++t) {
    const int pos = sm[t];
    if (pos < 0) continue;
    const float w = ex2(part_lse[(int64_t)pos * G + h] - mx);
    wsum += w;
    axpy(w, part_o + ((int64_t)pos * G + h) * D_H + d0);
  }
  const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
  __nv_bfloat16* dst = o + (i * H_q + (int64_t)r * G + h) * D_H + d0;
#pragma unroll
  for (int e = 0; e < EPL; e += 2)
    *reinterpret_cast<uint32_t*>(dst + e) = pack_bf16x2(acc[e] * inv, acc[e + 1] * inv);
  if (d0 == 0)
    lse[((int64_t)r * G + h) * N + i] = (mx + __log2f(wsum)) * 0.69314718055994531f;
}

template <int D_H>
cudaError_t merge_dispatch(int G, dim3 grid, cudaStream_t st, const void* tp_o, const float* tp_lse,
                           const int* slotmap, const void* part_o, const float* part_lse, void* o,
                           float* lse, int64_t N, int H_q, int H_kv, int kk, int64_t q0, int64_t q1) {
  auto a = static_cast<const __nv_bfloat16*>(tp_o);
  auto p = static_cast<const __nv_bfloat16*>(part_o);
  auto out = static_cast<__nv_bfloat16*>(o);
  switch (G) {
    case 1: k_attn_merge<D_H, 1><<<grid, 128, 0, st>>>(a, tp_lse, slotmap, p, part_lse, out, lse, N, H_q, H_kv, kk, q0, q1); break;
    case 2: k_attn_merge<D_H, 2><<<grid, 128, 0, st>>>(a, tp_lse, slotmap, p, part_lse, out, lse, N, H_q, H_kv, kk, q0, q1); break;
    case 4: k_attn_merge<D_H, 4><<<grid, 128, 0, st>>>(a, tp_lse, slotmap, p, part_lse, out, lse, N, H_q, H_kv, kk, q0, q1); break;
    default: k_attn_merge<D_H, 8><<<grid, 128, 0, st>>>(a, tp_lse, slotmap, p, part_lse, out, lse, N, H_q, H_kv, kk, q0, q1); break;
  }
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attn_plan(const int32_t* idx, int64_t N, int H_kv, int kk, int64_t q0,
                             int64_t q1, int64_t qc_stride, int64_t nblk, int pass, int* count,
                             const int* offset, int* cursor, int* entries, int* slotmap,
                             cudaStream_t st) {
  const int64_t tiles = (q1 - q0 + kTileQ - 1) / kTileQ;
  const dim3 grid((unsigned)((tiles + kPlanWarps - 1) / kPlanWarps), (unsigned)H_kv);
  k_attn_plan<<<grid, 32 * kPlanWarps, 0, st>>>(idx, N, kk, q0, q1, qc_stride, nblk, pass, count,
                                                offset, cursor, entries, slotmap);
  return cudaGetLastError();
}

cudaError_t launch_attn_scan(const int* count, int* offset, int* tile_off, int* cursor, int nb,
                             int ept, cudaStream_t st) {
  k_attn_scan<<<1, kScanThreads, 0, st>>>(count, offset, tile_off, cursor, nb, ept);
  return cudaGetLastError();
}

cudaError_t launch_attn_merge(const void* tp_o, const float* tp_lse, const int* slotmap,
                              const void* part_o, const float* part_lse, void* o, float* lse,
                              int64_t N, int H_q, int H_kv, int d_h, int kk, int64_t q0, int64_t q1,
                              cudaStream_t st) {
  const int64_t units = (int64_t)H_kv * (q1 - q0);
  const dim3 grid((unsigned)((units + 3) / 4));
  const int G = H_q / H_kv;
  if (d_h == 128)
    return merge_dispatch<128>(G, grid, st, tp_o, tp_lse, slotmap, part_o, part_lse, o, lse, N, H_q,
                               H_kv, kk, q0, q1);
  return merge_dispatch<64>(G, grid, st, tp_o, tp_lse, slotmap, part_o, part_lse, o, lse, N, H_q,
                            H_kv, kk, q0, q1);
}

}  // namespace msa

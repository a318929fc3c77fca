// Variable-length prefill batches («MiniMax-M3：MSA 技术报告速读», section 索引分支 and section
// 主分支, applied to each sequence of a packed batch on its own): one launch per stage for the
// whole batch.
//
// The sequences are laid out in a virtual row space in which every sequence starts on a multiple
// of max(128, the rows of one index-branch CTA).  There no 64-token block, 16-query tile or
// index-branch CTA spans two sequences, so the single-sequence kernels run on the whole virtual
// batch:
//   * the index branch starts each CTA's key loop at the first key tile of its sequence (ktab),
//     so a row's candidate blocks are its own sequence's blocks before its local block;
//   * the main branch needs nothing more: every selected block lies in the row's own sequence
//     and causality inside it is the virtual causality.
// Rows past a sequence's end (padding) are zero on input, select no block, and are dropped on
// output.  When every sequence length is already a multiple of the alignment, the virtual rows
// are the packed rows and Q, K, V, O are used in place; only the selections (to per-sequence
// block numbers and layout) and the LSE (to the per-sequence layout) are rewritten.
#include "msa_internal.h"

namespace msa {
namespace {

// sequence of virtual row v: the s with vstart[s] <= v < vstart[s+1]
__device__ __forceinline__ int find_seq(const int64_t* __restrict__ vstart, int nseq, int64_t v) {
  int lo = 0, hi = nseq;                                  // vstart[lo] <= v < vstart[hi]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (__ldg(vstart + mid) <= v) lo = mid; else hi = mid;
  }
  return lo;
}

__global__ void k_varlen_ktab(const int64_t* __restrict__ vstart, int nseq, int64_t ngroups,
                              int* ktab) {
  const int64_t g = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (g >= ngroups) return;
  const int s = find_seq(vstart, nseq, g * 128);
  ktab[g] = (int)(__ldg(vstart + s) / 128);
}

// 16-byte rows copies: dst row v (virtual) <- src row p (packed) or zeros for padding rows
__device__ __forceinline__ void copy_row(uint4* dst, const uint4* src, int n16, bool real) {
  for (int x = threadIdx.x; x < n16; x += blockDim.x) dst[x] = real ? __ldg(src + x) : make_uint4(0, 0, 0, 0);
}

struct VarlenIo {
  const uint4 *q, *k, *v, *qi, *ki;     // packed inputs
  uint4 *qv, *kv, *vv, *qiv, *kiv;      // virtual copies
  int nq16, nkv16, nqi16, nki16;        // 16-byte chunks per row of each tensor
};

__global__ void __launch_bounds__(256)
    k_varlen_gather(const int64_t* __restrict__ vstart, const int64_t* __restrict__ pstart,
                    int nseq, const VarlenIo io) {
  const int64_t v = blockIdx.x;
  const int s = find_seq(vstart, nseq, v);
  const int64_t il = v - __ldg(vstart + s);
  const bool real = il < __ldg(pstart + s + 1) - __ldg(pstart + s);
  const int64_t p = real ? __ldg(pstart + s) + il : 0;
  copy_row(io.qv + v * io.nq16, io.q + p * io.nq16, io.nq16, real);
  copy_row(io.kv + v * io.nkv16, io.k + p * io.nkv16, io.nkv16, real);
  copy_row(io.vv + v * io.nkv16, io.v + p * io.nkv16, io.nkv16, real);
  copy_row(io.qiv + v * io.nqi16, io.qi + p * io.nqi16, io.nqi16, real);
  copy_row(io.kiv + v * io.nki16, io.ki + p * io.nki16, io.nki16, real);
}

// Padding rows select nothing: a 16-query tile that holds a sequence's last rows then counts
// only real queries when it sorts its blocks into shared and private ones, exactly as the
// single-sequence call on those rows does.
__global__ void __launch_bounds__(256)
    k_varlen_clear_padding(const int64_t* __restrict__ vstart, const int64_t* __restrict__ pstart,
                           int nseq, int64_t Tv, int H_kv, int kk, int32_t* idx_v) {
  const int64_t v = (int64_t)blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5);
  if (v >= Tv) return;
  const int s = find_seq(vstart, nseq, v);
  if (v - __ldg(vstart + s) < __ldg(pstart + s + 1) - __ldg(pstart + s)) return;
  for (int x = threadIdx.x & 31; x < H_kv * kk; x += 32) {
    const int r = x / kk, t = x - r * kk;
    idx_v[((int64_t)r * Tv + v) * kk + t] = -1;
  }
}

// Per real virtual row: its selections (virtual block numbers -> the sequence's own, layout
// [H_kv, N_s, k] at element cu_seqlens[s] * H_kv * k), its LSEs (layout [H_q, N_s] at
// cu_seqlens[s] * H_q) and, unless the output was written in place, its O row.
__global__ void __launch_bounds__(256)
    k_varlen_scatter(const int64_t* __restrict__ vstart, const int64_t* __restrict__ pstart,
                     int nseq, int64_t Tv, int H_q, int H_kv, int kk,
                     const int32_t* __restrict__ idx_v, const float* __restrict__ lse_v,
                     const uint4* __restrict__ o_v, int no16, int32_t* idx, float* lse,
                     uint4* o) {
  const int64_t v = blockIdx.x;
  const int s = find_seq(vstart, nseq, v);
  const int64_t v0 = __ldg(vstart + s), t0 = __ldg(pstart + s);
  const int64_t n = __ldg(pstart + s + 1) - t0, il = v - v0;
  if (il >= n) return;
  const int fb = (int)(v0 >> 6);                           // the sequence's first block
  for (int x = threadIdx.x; x < H_kv * kk; x += blockDim.x) {
    const int r = x / kk, t = x - r * kk;
    const int32_t b = __ldg(idx_v + ((int64_t)r * Tv + v) * kk + t);
    idx[t0 * H_kv * kk + ((int64_t)r * n + il) * kk + t] = b >= 0 ? b - fb : -1;
  }
  for (int h = threadIdx.x; h < H_q; h += blockDim.x)
    lse[t0 * H_q + (int64_t)h * n + il] = __ldg(lse_v + (int64_t)h * Tv + v);
  if (o_v != nullptr)
    for (int x = threadIdx.x; x < no16; x += blockDim.x) o[(t0 + il) * no16 + x] = __ldg(o_v + v * no16 + x);
}

size_t a256(size_t x) { return (x + 255) & ~size_t(255); }

}  // namespace

VarlenLayout varlen_layout(const int64_t* cu_seqlens, int nseq, int H_q, int H_kv, int d_h,
                           int d_idx, int k) {
  VarlenLayout w{};
  const int64_t align = std::max<int64_t>(128, index_rows_per_cta(H_kv));
  w.align = align;
  int64_t tv = 0;
  for (int s = 0; s < nseq; ++s) {
    const int64_t n = cu_seqlens[s + 1] - cu_seqlens[s];
    tv += (n + align - 1) / align * align;
  }
  w.Tv = tv;
  w.in_place = tv == cu_seqlens[nseq];      // every length is a multiple of the alignment
  size_t off = 0;
  auto take = [&](size_t bytes) { const size_t o = off; off = a256(off + bytes); return o; };
  w.main = take(sparse_attn_ws_bytes(tv, H_q, H_kv, d_h, k));
  w.starts = take(2 * 8 * (size_t)(nseq + 1));
  w.ktab = take(4 * (size_t)(tv / 128));
  w.idx = take(4 * (size_t)H_kv * tv * k);
  w.lse = take(4 * (size_t)H_q * tv);
  if (!w.in_place) {
    w.q = take(2 * (size_t)tv * H_q * d_h);
    w.k = take(2 * (size_t)tv * H_kv * d_h);
    w.v = take(2 * (size_t)tv * H_kv * d_h);
    w.qi = take(2 * (size_t)tv * H_kv * d_idx);
    w.ki = take(2 * (size_t)tv * d_idx);
    w.o = take(2 * (size_t)tv * H_q * d_h);
  }
  w.total = off;
  return w;
}

cudaError_t launch_prefill_varlen(const void* q, const void* k, const void* v, const void* q_idx,
                                  const void* k_idx, const int64_t* cu_seqlens, int nseq,
                                  int H_q, int H_kv, int d_h, int d_idx, int kk, int32_t* idx,
                                  void* o, float* lse, void* ws, cudaStream_t st) {
  const VarlenLayout w = varlen_layout(cu_seqlens, nseq, H_q, H_kv, d_h, d_idx, kk);
  char* base = static_cast<char*>(ws);
  int64_t* vstart = reinterpret_cast<int64_t*>(base + w.starts);
  int64_t* pstart = vstart + (nseq + 1);
  // the two start tables (host -> device; the host copies are staged before the call returns)
  std::vector<int64_t> h(2 * (size_t)(nseq + 1));
  h[0] = 0;
  for (int s = 0; s < nseq; ++s) {
    const int64_t n = cu_seqlens[s + 1] - cu_seqlens[s];
    h[s + 1] = h[s] + (n + w.align - 1) / w.align * w.align;
  }
  for (int s = 0; s <= nseq; ++s) h[nseq + 1 + s] = cu_seqlens[s];
  cudaError_t e = cudaMemcpyAsync(vstart, h.data(), h.size() * 8, cudaMemcpyHostToDevice, st);
  if (e != cudaSuccess) return e;
  int* ktab = reinterpret_cast<int*>(base + w.ktab);
  const int64_t ng = w.Tv / 128;
  k_varlen_ktab<<<(unsigned)((ng + 255) / 256), 256, 0, st>>>(vstart, nseq, ng, ktab);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  const void *qv = q, *kv = k, *vv = v, *qiv = q_idx, *kiv = k_idx;
  void* ov = o;
  if (!w.in_place) {
    VarlenIo io{};
    io.q = static_cast<const uint4*>(q);
    io.k = static_cast<const uint4*>(k);
    io.v = static_cast<const uint4*>(v);
    io.qi = static_cast<const uint4*>(q_idx);
    io.ki = static_cast<const uint4*>(k_idx);
    io.qv = reinterpret_cast<uint4*>(base + w.q);
    io.kv = reinterpret_cast<uint4*>(base + w.k);
    io.vv = reinterpret_cast<uint4*>(base + w.v);
    io.qiv = reinterpret_cast<uint4*>(base + w.qi);
    io.kiv = reinterpret_cast<uint4*>(base + w.ki);
    io.nq16 = H_q * d_h / 8;
    io.nkv16 = H_kv * d_h / 8;
    io.nqi16 = H_kv * d_idx / 8;
    io.nki16 = d_idx / 8;
    k_varlen_gather<<<(unsigned)w.Tv, 256, 0, st>>>(vstart, pstart, nseq, io);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    qv = io.qv, kv = io.kv, vv = io.vv, qiv = io.qiv, kiv = io.kiv;
    ov = base + w.o;
  }
  int32_t* idx_v = reinterpret_cast<int32_t*>(base + w.idx);
  float* lse_v = reinterpret_cast<float*>(base + w.lse);
  if ((e = launch_index_select(qiv, kiv, idx_v, w.Tv, H_kv, d_idx, kk, 0, w.Tv, st, ktab)) !=
      cudaSuccess)
    return e;
  if (!w.in_place) {
    k_varlen_clear_padding<<<(unsigned)((w.Tv + 7) / 8), 256, 0, st>>>(vstart, pstart, nseq, w.Tv,
                                                                      H_kv, kk, idx_v);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  if ((e = launch_sparse_attn_fwd(qv, kv, vv, idx_v, ov, lse_v, w.Tv, H_q, H_kv, d_h, kk,
                                  base + w.main, st)) != cudaSuccess)
    return e;
  k_varlen_scatter<<<(unsigned)w.Tv, 256, 0, st>>>(
      vstart, pstart, nseq, w.Tv, H_q, H_kv, kk, idx_v, lse_v,
      w.in_place ? nullptr : static_cast<const uint4*>(ov), H_q * d_h / 8, idx, lse,
      static_cast<uint4*>(o));
  return cudaGetLastError();
}

}  // namespace msa

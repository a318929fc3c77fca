// Main branch of prefill («MiniMax-M3：MSA 技术报告速读», section 主分支, eq. O^(h)_i): the
// launch sequence over query chunks and its workspace.
//
// Per chunk of at most 16384 query rows:
//   plan (count) -> scan -> plan (scatter)   bucket the private selections (attn_tile.cuh)
//   k_attn_kvouter                           block-major tcgen05 pass over private selections
//   k_attn_shared                            16-query tiles over their shared blocks; its
//                                            epilogue merges the private partials in slot
//                                            order and writes O and LSE
// Nothing here allocates or synchronises; the caller provides the workspace.
#include "attn_tile.cuh"
#include "msa_internal.h"

namespace msa {
namespace {

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

constexpr int64_t kChunkRows = 16384;     // query rows per pass (bounds the workspace)

struct AttnWs {
  size_t count, offset, tile_off, cursor, entries, part_o, part_lse, total;
  int64_t qc;
  int nb;
};

AttnWs attn_layout(int64_t N, int H_q, int H_kv, int d_h, int kk) {
  AttnWs w{};
  const int G = H_q / H_kv;
  w.qc = ((N < kChunkRows ? N : kChunkRows) + kTileQ - 1) / kTileQ * kTileQ;
  const int64_t nblk = (N + kBlock - 1) / kBlock;
  w.nb = (int)(H_kv * nblk);
  const size_t sel = (size_t)H_kv * w.qc * kk;            // selections of one chunk
  size_t off = 0;
  auto take = [&](size_t bytes) { const size_t o = off; off = align256(off + bytes); return o; };
  w.count = take(4 * (size_t)(w.nb + 1));
  w.offset = take(4 * (size_t)(w.nb + 1));
  w.tile_off = take(4 * (size_t)(w.nb + 1));
  w.cursor = take(4 * (size_t)(w.nb + 1));
  w.entries = take(4 * sel);
  w.part_o = take(2 * sel * G * d_h);
  w.part_lse = take(4 * sel * G);
  w.total = off;
  return w;
}

}  // namespace

size_t sparse_attn_ws_bytes(int64_t N, int H_q, int H_kv, int d_h, int kk) {
  return attn_layout(N, H_q, H_kv, d_h, kk).total;
}

// The main branch over query chunks: plan (count) -> scan -> plan (scatter) -> block-major pass
// over private selections -> shared-block pass (which also merges).  Everything is enqueued on
// `stream`.
cudaError_t launch_sparse_attn_fwd(const void* q, const void* k, const void* v, const int32_t* idx,
                                   void* o, float* lse, int64_t N, int H_q, int H_kv, int d_h,
                                   int kk, void* ws, cudaStream_t stream) {
  const AttnWs w = attn_layout(N, H_q, H_kv, d_h, kk);
  char* base = static_cast<char*>(ws);
  int* count = reinterpret_cast<int*>(base + w.count);
  int* offset = reinterpret_cast<int*>(base + w.offset);
  int* tile_off = reinterpret_cast<int*>(base + w.tile_off);
  int* cursor = reinterpret_cast<int*>(base + w.cursor);
  int* entries = reinterpret_cast<int*>(base + w.entries);
  void* part_o = base + w.part_o;
  float* part_lse = reinterpret_cast<float*>(base + w.part_lse);

  CUtensorMap tk, tv;
  cudaError_t e = make_tma_3d_bf16(&tk, k, (uint64_t)d_h, (uint64_t)H_kv, (uint64_t)N, 64, 1, 32, 128);
  if (e != cudaSuccess) return e;
  e = make_tma_3d_bf16(&tv, v, (uint64_t)d_h, (uint64_t)H_kv, (uint64_t)N, 64, 1, 32, 128);
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 148;
  if (cudaGetDevice(&dev) == cudaSuccess)
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int64_t nblk = (N + kBlock - 1) / kBlock;
  const int G = H_q / H_kv;
  for (int64_t q0 = 0; q0 < N; q0 += w.qc) {
    const int64_t q1 = q0 + w.qc < N ? q0 + w.qc : N;
    if ((e = cudaMemsetAsync(count, 0, 4 * (size_t)w.nb, stream)) != cudaSuccess) return e;
    if ((e = launch_attn_plan(idx, N, H_kv, kk, q0, q1, nblk, 0, count, offset, cursor, entries,
                              stream)) != cudaSuccess) return e;
    if ((e = launch_attn_scan(count, offset, tile_off, cursor, w.nb, 128 / G, stream)) != cudaSuccess)
      return e;
    if ((e = launch_attn_plan(idx, N, H_kv, kk, q0, q1, nblk, 1, count, offset, cursor, entries,
                              stream)) != cudaSuccess) return e;
    if ((e = launch_attn_kvouter(q, k, v, entries, offset, tile_off, w.nb, nblk, N, q0, q1, H_q,
                                 H_kv, d_h, kk, 3 * sms, part_o, part_lse, stream)) != cudaSuccess)
      return e;
    if ((e = launch_attn_shared(tk, tv, q, idx, part_o, part_lse, o, lse, N, q0, q1, H_q,
                                H_kv, d_h, kk, stream)) != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace msa

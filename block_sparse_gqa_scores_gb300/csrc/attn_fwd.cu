// Main branch of prefill («MiniMax-M3：MSA 技术报告速读», section 主分支, eq. O^(h)_i): the
// launch sequence over query chunks and its workspace.
//
// Per chunk of at most 65536 query rows:
//   plan -> scan -> scatter                  bucket the private selections (attn_tile.cuh) and
//                                            record each tile's shared blocks
//   k_attn_kvouter                           block-major tcgen05 pass over private selections
//   k_attn_shared                            16-query tiles over their shared blocks; its
//                                            epilogue merges the private partials in slot
//                                            order and writes O and LSE
// The two passes stress different units (the block-major pass moves the partials and the
// gathered query rows through HBM; the shared-block pass is bound by its softmax chain), so
// chunks are pipelined over two streams: the plan and block-major pass of chunk c+1 run on a
// library-owned side stream while the shared-block pass of chunk c runs on the caller's
// stream, with two workspace sets used alternately and events ordering each hand-over.  All
// work of the call is complete when the caller's stream reaches the end of it.
// Nothing here allocates device memory or synchronises the host; the caller provides the
// workspace.
#include <mutex>

#include "attn_tile.cuh"
#include "msa_internal.h"

namespace msa {
namespace {

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// query rows per pass: bounds the workspace (about 8.8 GB per set at the 128K shape); larger
// chunks fill the (group, block) buckets of the block-major pass better and leave fewer passes
// (main branch at 128K: 6.66 ms with 65536 rows, 6.94 ms with 32768, 6.74 ms with one chunk of
// 131072)
constexpr int64_t kChunkRows = 65536;
constexpr int kKvoCtasPerSm = 1;         // block-major pass: persistent, one CTA per SM (TMEM)

struct AttnWs {
  size_t count, offset, tile_off, sc, sc_n, entries, tile_list, tile_priv, part_o, part_lse,
      set_bytes;
  int64_t qc;
  int nb, sets;
};

// One workspace set per chunk in flight: two when there is more than one chunk.
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
  w.entries = take(4 * sel);
  const size_t tiles = (size_t)H_kv * (w.qc / kTileQ);            // 16-query tiles of a chunk
  w.sc = take(12 * sel);                 // per tile: (bucket, rank, entry) of its private selections
  w.sc_n = take(4 * tiles);
  w.tile_list = take(4 * tiles * (kMaxShared + 1));
  w.tile_priv = take(8 * tiles * kTileQ);
  w.part_o = take(2 * sel * G * d_h);
  w.part_lse = take(4 * sel * G);
  w.set_bytes = off;
  w.sets = N > w.qc ? 2 : 1;
  return w;
}

// The side stream of each device, created on first use.
std::mutex g_side_mutex;
cudaStream_t g_side[64] = {};

cudaError_t side_stream(cudaStream_t* out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_side_mutex);
  if (!g_side[dev] && (e = cudaStreamCreateWithFlags(&g_side[dev], cudaStreamNonBlocking)) != cudaSuccess)
    return e;
  *out = g_side[dev];
  return cudaSuccess;
}

// Events of one call (released once the device has passed them).
struct CallEvents {
  cudaEvent_t start = nullptr, ready[2] = {nullptr, nullptr}, freed[2] = {nullptr, nullptr};
  cudaError_t create() {
    cudaError_t e = cudaEventCreateWithFlags(&start, cudaEventDisableTiming);
    for (int s = 0; s < 2 && e == cudaSuccess; ++s) {
      e = cudaEventCreateWithFlags(&ready[s], cudaEventDisableTiming);
      if (e == cudaSuccess) e = cudaEventCreateWithFlags(&freed[s], cudaEventDisableTiming);
    }
    return e;
  }
  ~CallEvents() {
    if (start) cudaEventDestroy(start);
    for (int s = 0; s < 2; ++s) {
      if (ready[s]) cudaEventDestroy(ready[s]);
      if (freed[s]) cudaEventDestroy(freed[s]);
    }
  }
};

}  // namespace

size_t sparse_attn_ws_bytes(int64_t N, int H_q, int H_kv, int d_h, int kk) {
  const AttnWs w = attn_layout(N, H_q, H_kv, d_h, kk);
  return w.set_bytes * w.sets;
}

// The main branch over query chunks: plan -> scan -> scatter -> block-major pass
// over private selections, then the shared-block pass (which also merges), pipelined as above.
cudaError_t launch_sparse_attn_fwd(const void* q, const void* k, const void* v, const int32_t* idx,
                                   void* o, float* lse, int64_t N, int H_q, int H_kv, int d_h,
                                   int kk, void* ws, cudaStream_t stream) {
  const AttnWs w = attn_layout(N, H_q, H_kv, d_h, kk);
  const int G = H_q / H_kv;
  CUtensorMap tq, tk, tv;
  cudaError_t e = make_tma_3d_bf16(&tq, q, (uint64_t)d_h, (uint64_t)H_q, (uint64_t)N, 64, G, kTileQ, 128);
  if (e != cudaSuccess) return e;
  e = make_tma_3d_bf16(&tk, k, (uint64_t)d_h, (uint64_t)H_kv, (uint64_t)N, 64, 1, 32, 128);
  if (e != cudaSuccess) return e;
  e = make_tma_3d_bf16(&tv, v, (uint64_t)d_h, (uint64_t)H_kv, (uint64_t)N, 64, 1, 32, 128);
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 148;
  if (cudaGetDevice(&dev) == cudaSuccess)
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int64_t nblk = (N + kBlock - 1) / kBlock;

  // one chunk: everything on the caller's stream
  cudaStream_t side = stream;
  CallEvents ev;
  if (w.sets == 2) {
    if ((e = side_stream(&side)) != cudaSuccess) return e;
    if ((e = ev.create()) != cudaSuccess) return e;
    if ((e = cudaEventRecord(ev.start, stream)) != cudaSuccess) return e;     // inputs ready
    if ((e = cudaStreamWaitEvent(side, ev.start, 0)) != cudaSuccess) return e;
  }
  int64_t c = 0;
  for (int64_t q0 = 0; q0 < N; q0 += w.qc, ++c) {
    const int64_t q1 = q0 + w.qc < N ? q0 + w.qc : N;
    const int s = (int)(c & 1) % w.sets;
    char* base = static_cast<char*>(ws) + (size_t)s * w.set_bytes;
    int* count = reinterpret_cast<int*>(base + w.count);
    int* offset = reinterpret_cast<int*>(base + w.offset);
    int* tile_off = reinterpret_cast<int*>(base + w.tile_off);
    int* sc = reinterpret_cast<int*>(base + w.sc);
    int* sc_n = reinterpret_cast<int*>(base + w.sc_n);
    int* entries = reinterpret_cast<int*>(base + w.entries);
    int* tile_list = reinterpret_cast<int*>(base + w.tile_list);
    auto* tile_priv = reinterpret_cast<unsigned long long*>(base + w.tile_priv);
    void* part_o = base + w.part_o;
    float* part_lse = reinterpret_cast<float*>(base + w.part_lse);
    // the block-major half of chunk c, once the shared-block pass of chunk c-2 has read set s
    if (w.sets == 2 && c >= 2 && (e = cudaStreamWaitEvent(side, ev.freed[s], 0)) != cudaSuccess)
      return e;
    if ((e = cudaMemsetAsync(count, 0, 4 * (size_t)w.nb, side)) != cudaSuccess) return e;
    if ((e = launch_attn_plan(idx, N, H_kv, kk, q0, q1, nblk, count, tile_list, tile_priv, sc,
                              sc_n, side)) != cudaSuccess) return e;
    if ((e = launch_attn_scan(count, offset, tile_off, w.nb, 128 / G, side)) != cudaSuccess)
      return e;
    if ((e = launch_attn_scatter(sc, sc_n, offset, entries,
                                 (int64_t)H_kv * ((q1 - q0 + kTileQ - 1) / kTileQ), kk, side)) != cudaSuccess)
      return e;
    if ((e = launch_attn_kvouter(q, k, v, entries, offset, tile_off, w.nb, nblk, N, q0, q1, H_q,
                                 H_kv, d_h, kk, kKvoCtasPerSm * sms, part_o, part_lse, side)) != cudaSuccess)
      return e;
    // the shared-block half (and the merge) of chunk c on the caller's stream
    if (w.sets == 2) {
      if ((e = cudaEventRecord(ev.ready[s], side)) != cudaSuccess) return e;
      if ((e = cudaStreamWaitEvent(stream, ev.ready[s], 0)) != cudaSuccess) return e;
    }
    if ((e = launch_attn_shared(tq, tk, tv, q, tile_list, tile_priv, part_o, part_lse, o, lse, N, q0, q1, H_q,
                                H_kv, d_h, kk, stream)) != cudaSuccess) return e;
    if (w.sets == 2 && (e = cudaEventRecord(ev.freed[s], stream)) != cudaSuccess) return e;
  }
  // every side-stream launch precedes a shared-block pass that waited for it, so the caller's
  // stream finishing the last pass means the whole call is done
  return cudaSuccess;
}

}  // namespace msa

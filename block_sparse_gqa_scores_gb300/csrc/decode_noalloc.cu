// msa_sparse_decode_noalloc: the decode path with its scratch in a fixed device array, so that
// neither the caller nor the library allocates anything for it.
//
// Who needs this: a caller that cannot create device buffers at the point where it decodes --
// for example a serving runtime that reserved all device memory for its own pool up front, or
// a latency-critical decode loop that must not call cudaMalloc/cudaFree because those calls can
// block on other work or synchronise the device.  Such a caller still owns and passes every
// input and output; only the temporary block scores and selections live in
// the array below.
//
// The array is part of the library image: every GPU that loads libmsa.so holds these bytes
// until the process exits.  Its device address is looked up once per device, on the first call
// made with that device current (cudaGetSymbolAddress); make that first call before capturing
// any stream.  The cached address belongs to the device's primary context: a device reset
// (cudaDeviceReset) re-creates that context and may load the library elsewhere, after which the
// cached address is stale, so this entry point must not be used on that device again.  All calls share the array and it keeps the last call's contents; nothing in it
// has to start at zero, because every entry a kernel reads was written earlier in the same
// call.  Two calls whose work overlaps on the GPU (different streams, or different host threads
// on one device) race on the array: serialise them.
#include <mutex>

#include "../../include/msa.h"
#include "msa_internal.h"

static __device__ __align__(256) unsigned char msa_decode_scratch[MSA_DECODE_NOALLOC_SCRATCH_BYTES];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mutex;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of msa_decode_scratch on the current device (looked up once per device).
cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, msa_decode_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return cudaSuccess;
}

bool al16(const void* p) { return p && ((uintptr_t)p & 15u) == 0; }
bool al4(const void* p) { return p && ((uintptr_t)p & 3u) == 0; }
bool pow2_le(int x, int hi) { return x >= 1 && x <= hi && (x & (x - 1)) == 0; }

}  // namespace

extern "C" __attribute__((visibility("default"))) msa_status_t msa_sparse_decode_noalloc(
    const void* q, const void* q_idx, const void* k_cache, const void* v_cache,
    const void* k_idx_cache, const int64_t* cu_seqlens, int S, int64_t max_len, int H_q, int H_kv,
    int d_h, int d_idx, int block_size, int k, void* o, float* lse, int32_t* idx_out,
    void* stream) {
  if (!al16(q) || !al16(q_idx) || !al16(k_cache) || !al16(v_cache) || !al16(k_idx_cache) ||
      !cu_seqlens || ((uintptr_t)cu_seqlens & 7u) || !al16(o) || !al4(lse) ||
      (idx_out && !al4(idx_out)))
    return MSA_ERR_INVALID_ARGUMENT;
  if (S < 1 || S > 65535 || max_len < 1 || H_q < 1 || H_kv < 1 || H_q % H_kv != 0 ||
      block_size != 64 || k < 1 || k > 64 || d_h < 1 || d_idx < 1)
    return MSA_ERR_INVALID_ARGUMENT;
  if (!pow2_le(H_kv, 8) || !pow2_le(H_q / H_kv, 8) || (d_h != 64 && d_h != 128) ||
      (d_idx != 32 && d_idx != 64))
    return MSA_ERR_UNSUPPORTED;
  const msa::DecodeWs w = msa::decode_layout(S, max_len, H_q, H_kv, d_h, k);
  if (w.total > (size_t)MSA_DECODE_NOALLOC_SCRATCH_BYTES) return MSA_ERR_WORKSPACE;
  void* scratch = nullptr;
  if (scratch_address(&scratch) != cudaSuccess) return MSA_ERR_CUDA;

  cudaStream_t st = (cudaStream_t)stream;
  char* base = static_cast<char*>(scratch);
  float* Mdec = reinterpret_cast<float*>(base + w.off_m);
  int32_t* idx = idx_out ? idx_out : reinterpret_cast<int32_t*>(base + w.off_idx);
  const int64_t nblk = (max_len + 63) / 64;
  const msa::CacheMap cm{cu_seqlens, nullptr, nullptr, 0, 0};
  cudaError_t e = msa::launch_decode_block_scores(q_idx, k_idx_cache, cm, Mdec, S, H_kv,
                                                  d_idx, max_len, nblk, st);
  if (e != cudaSuccess) return MSA_ERR_CUDA;
  e = msa::launch_decode_tail(q, k_cache, v_cache, Mdec, nblk, cm, S, max_len, H_q, H_kv, d_h,
                              k, idx, o, lse, st);
  return e == cudaSuccess ? MSA_OK : MSA_ERR_CUDA;
}

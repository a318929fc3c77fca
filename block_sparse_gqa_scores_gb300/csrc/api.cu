// C ABI of libmsa: host-side validation, workspace layout and dispatch to the kernels.
// Nothing here allocates device memory or synchronises, except msa_device_status().
#include <cudaTypedefs.h>

#include <algorithm>
#include <mutex>

#include "../../include/msa.h"
#include "msa_internal.h"

#define MSA_API extern "C" __attribute__((visibility("default")))

namespace msa {

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

cudaError_t make_tma_2d_bf16(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer,
                             int box_inner, int box_outer, int swizzle_bytes) {
  auto fn = encode_fn();
  if (!fn) return cudaErrorNotSupported;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {inner * 2};
  cuuint32_t box[2] = {(cuuint32_t)box_inner, (cuuint32_t)box_outer};
  cuuint32_t estr[2] = {1, 1};
  const CUtensorMapSwizzle sw = swizzle_bytes == 128  ? CU_TENSOR_MAP_SWIZZLE_128B
                                : swizzle_bytes == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                                                      : CU_TENSOR_MAP_SWIZZLE_NONE;
  const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t make_tma_3d_bf16(CUtensorMap* map, const void* base, uint64_t d0, uint64_t d1,
                             uint64_t d2, int box0, int box1, int box2, int swizzle_bytes) {
  auto fn = encode_fn();
  if (!fn) return cudaErrorNotSupported;
  cuuint64_t dims[3] = {d0, d1, d2};
  cuuint64_t strides[2] = {d0 * 2, d0 * d1 * 2};
  cuuint32_t box[3] = {(cuuint32_t)box0, (cuuint32_t)box1, (cuuint32_t)box2};
  cuuint32_t estr[3] = {1, 1, 1};
  const CUtensorMapSwizzle sw = swizzle_bytes == 128  ? CU_TENSOR_MAP_SWIZZLE_128B
                                : swizzle_bytes == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                                                      : CU_TENSOR_MAP_SWIZZLE_NONE;
  const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t make_tma_4d_bf16(CUtensorMap* map, const void* base, const uint64_t dims[4],
                             const uint64_t strides[3], const int box[4], int swizzle_bytes) {
  auto fn = encode_fn();
  if (!fn) return cudaErrorNotSupported;
  cuuint64_t d[4] = {dims[0], dims[1], dims[2], dims[3]};
  cuuint64_t st[3] = {strides[0], strides[1], strides[2]};
  cuuint32_t bx[4] = {(cuuint32_t)box[0], (cuuint32_t)box[1], (cuuint32_t)box[2], (cuuint32_t)box[3]};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  const CUtensorMapSwizzle sw = swizzle_bytes == 128  ? CU_TENSOR_MAP_SWIZZLE_128B
                                : swizzle_bytes == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                                                      : CU_TENSOR_MAP_SWIZZLE_NONE;
  const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), d, st,
                        bx, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace msa

namespace {

constexpr int64_t kMaxRows = (int64_t)1 << 31;   // TMA coordinates and grid.x are 32-bit

bool aligned16(const void* p) { return p && ((uintptr_t)p & 15u) == 0; }
bool aligned4(const void* p) { return p && ((uintptr_t)p & 3u) == 0; }
bool pow2_upto(int x, int hi) { return x >= 1 && x <= hi && (x & (x - 1)) == 0; }

msa_status_t from_cuda(cudaError_t e) { return e == cudaSuccess ? MSA_OK : MSA_ERR_CUDA; }

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

}  // namespace

namespace msa {

DecodeWs decode_layout(int S, int64_t max_len, int H_q, int H_kv, int d_h, int k) {
  (void)H_q;
  (void)d_h;
  DecodeWs w{};
  const int64_t nblk = (max_len + 63) / 64;
  size_t off = 0;
  w.off_m = off;
  off = align256(off + sizeof(float) * (size_t)S * H_kv * nblk);
  w.off_idx = off;
  off = align256(off + sizeof(int32_t) * (size_t)S * H_kv * k);
  w.total = off;
  return w;
}

}  // namespace msa

using msa::DecodeWs;
using msa::decode_layout;

MSA_API const char* msa_status_string(msa_status_t s) {
  switch (s) {
    case MSA_OK: return "MSA_OK";
    case MSA_ERR_INVALID_ARGUMENT: return "MSA_ERR_INVALID_ARGUMENT";
    case MSA_ERR_UNSUPPORTED: return "MSA_ERR_UNSUPPORTED";
    case MSA_ERR_WORKSPACE: return "MSA_ERR_WORKSPACE";
    case MSA_ERR_CUDA: return "MSA_ERR_CUDA";
    case MSA_ERR_TIMEOUT: return "MSA_ERR_TIMEOUT";
  }
  return "MSA_ERR_UNKNOWN";
}

MSA_API msa_status_t msa_index_block_scores(const void* q_idx, const void* k_idx, float* M,
                                            int64_t N, int H_kv, int d_idx, int block_size,
                                            int64_t q_start, int64_t q_count, void* stream) {
  if (!aligned16(q_idx) || !aligned16(k_idx) || !aligned16(M)) return MSA_ERR_INVALID_ARGUMENT;
  if (N < 1 || H_kv < 1 || d_idx < 1 || block_size != 64) return MSA_ERR_INVALID_ARGUMENT;
  if (q_start < 0 || q_count < 1 || q_start + q_count > N) return MSA_ERR_INVALID_ARGUMENT;
  if (!pow2_upto(H_kv, 8) || (d_idx != 32 && d_idx != 64)) return MSA_ERR_UNSUPPORTED;
  if (N * H_kv >= kMaxRows) return MSA_ERR_UNSUPPORTED;
  return from_cuda(msa::launch_index_block_scores(q_idx, k_idx, M, N, H_kv, d_idx, q_start,
                                                  q_count, (cudaStream_t)stream));
}

MSA_API msa_status_t msa_select_blocks(const float* M, int32_t* idx, int64_t N, int H_kv,
                                       int block_size, int k, int64_t q_start, int64_t q_count,
                                       void* stream) {
  if (!aligned16(M) || !aligned4(idx)) return MSA_ERR_INVALID_ARGUMENT;
  if (N < 1 || H_kv < 1 || block_size != 64 || k < 1 || k > 64) return MSA_ERR_INVALID_ARGUMENT;
  if (q_start < 0 || q_count < 1 || q_start + q_count > N) return MSA_ERR_INVALID_ARGUMENT;
  if (!pow2_upto(H_kv, 8)) return MSA_ERR_UNSUPPORTED;
  if (N * H_kv >= kMaxRows) return MSA_ERR_UNSUPPORTED;
  return from_cuda(
      msa::launch_select_prefill(M, idx, N, H_kv, k, q_start, q_count, (cudaStream_t)stream));
}

MSA_API msa_status_t msa_index_select(const void* q_idx, const void* k_idx, int32_t* idx,
                                      int64_t N, int H_kv, int d_idx, int block_size, int k,
                                      int64_t q_start, int64_t q_count, void* stream) {
  if (!aligned16(q_idx) || !aligned16(k_idx) || !aligned4(idx)) return MSA_ERR_INVALID_ARGUMENT;
  if (N < 1 || H_kv < 1 || d_idx < 1 || block_size != 64 || k < 1 || k > 64)
    return MSA_ERR_INVALID_ARGUMENT;
  if (q_start < 0 || q_count < 1 || q_start + q_count > N) return MSA_ERR_INVALID_ARGUMENT;
  if (!pow2_upto(H_kv, 8) || (d_idx != 32 && d_idx != 64) || k > MSA_INDEX_SELECT_MAX_K)
    return MSA_ERR_UNSUPPORTED;
  if (N * H_kv >= kMaxRows) return MSA_ERR_UNSUPPORTED;
  return from_cuda(msa::launch_index_select(q_idx, k_idx, idx, N, H_kv, d_idx, k, q_start,
                                            q_count, (cudaStream_t)stream));
}

MSA_API size_t msa_sparse_attn_fwd_workspace(int64_t N, int H_q, int H_kv, int d_h, int k) {
  if (N < 1 || H_kv < 1 || H_q < H_kv || H_q % H_kv != 0 || k < 1 || k > 64 || d_h < 1) return 0;
  return msa::sparse_attn_ws_bytes(N, H_q, H_kv, d_h, k);
}

MSA_API msa_status_t msa_sparse_attn_fwd(const void* q, const void* k, const void* v,
                                         const int32_t* idx, void* o, float* lse, int64_t N,
                                         int H_q, int H_kv, int d_h, int block_size, int k_blocks,
                                         void* ws, size_t ws_bytes, void* stream) {
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned4(idx) || !aligned16(o) ||
      !aligned4(lse) || !aligned16(ws))
    return MSA_ERR_INVALID_ARGUMENT;
  if (N < 1 || H_q < 1 || H_kv < 1 || H_q % H_kv != 0 || d_h < 1 || block_size != 64 ||
      k_blocks < 1 || k_blocks > 64)
    return MSA_ERR_INVALID_ARGUMENT;
  if (!pow2_upto(H_kv, 8) || !pow2_upto(H_q / H_kv, 8) || (d_h != 64 && d_h != 128))
    return MSA_ERR_UNSUPPORTED;
  if (N * H_kv >= kMaxRows || N > ((int64_t)1 << 21)) return MSA_ERR_UNSUPPORTED;
  if (ws_bytes < msa_sparse_attn_fwd_workspace(N, H_q, H_kv, d_h, k_blocks))
    return MSA_ERR_WORKSPACE;
  return from_cuda(msa::launch_sparse_attn_fwd(q, k, v, idx, o, lse, N, H_q, H_kv, d_h, k_blocks,
                                               ws, (cudaStream_t)stream));
}

MSA_API size_t msa_sparse_attn_bwd_workspace(int64_t N, int H_q, int H_kv, int d_h, int k) {
  if (N < 1 || H_kv < 1 || H_q < H_kv || H_q % H_kv != 0 || k < 1 || k > 64 || d_h < 1) return 0;
  return msa::sparse_attn_bwd_ws_bytes(N, H_q, H_kv, d_h, k);
}

MSA_API msa_status_t msa_sparse_attn_bwd(const void* q, const void* k, const void* v,
                                         const int32_t* idx, const void* o, const float* lse,
                                         const void* d_o, float* dq, float* dk, float* dv,
                                         int64_t N, int H_q, int H_kv, int d_h, int block_size,
                                         int k_blocks, void* ws, size_t ws_bytes, void* stream) {
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned4(idx) || !aligned16(o) ||
      !aligned4(lse) || !aligned16(d_o) || !aligned16(dq) || !aligned16(dk) || !aligned16(dv) ||
      !aligned16(ws))
    return MSA_ERR_INVALID_ARGUMENT;
  if (N < 1 || H_q < 1 || H_kv < 1 || H_q % H_kv != 0 || d_h < 1 || block_size != 64 ||
      k_blocks < 1 || k_blocks > 64)
    return MSA_ERR_INVALID_ARGUMENT;
  if (!pow2_upto(H_kv, 8) || !pow2_upto(H_q / H_kv, 8) || (d_h != 64 && d_h != 128))
    return MSA_ERR_UNSUPPORTED;
  if (N > ((int64_t)1 << 21) || N * H_kv * k_blocks >= kMaxRows) return MSA_ERR_UNSUPPORTED;
  if (ws_bytes < msa::sparse_attn_bwd_ws_bytes(N, H_q, H_kv, d_h, k_blocks))
    return MSA_ERR_WORKSPACE;
  return from_cuda(msa::launch_sparse_attn_bwd(q, k, v, idx, o, lse, d_o, dq, dk, dv, N, H_q,
                                               H_kv, d_h, k_blocks, ws, (cudaStream_t)stream));
}

MSA_API size_t msa_sparse_decode_workspace(int S, int64_t max_len, int H_q, int H_kv, int d_h,
                                           int d_idx, int k) {
  (void)d_idx;
  if (S < 1 || max_len < 1 || H_kv < 1 || H_q < H_kv || k < 1) return 0;
  return decode_layout(S, max_len, H_q, H_kv, d_h, k).total;
}

MSA_API msa_status_t msa_sparse_decode(const void* q, const void* q_idx, const void* k_cache,
                                       const void* v_cache, const void* k_idx_cache,
                                       const int64_t* cu_seqlens, int S, int64_t max_len, int H_q,
                                       int H_kv, int d_h, int d_idx, int block_size, int k,
                                       void* o, float* lse, int32_t* idx_out, void* ws,
                                       size_t ws_bytes, void* stream) {
  if (!aligned16(q) || !aligned16(q_idx) || !aligned16(k_cache) || !aligned16(v_cache) ||
      !aligned16(k_idx_cache) || !cu_seqlens || ((uintptr_t)cu_seqlens & 7u) || !aligned16(o) ||
      !aligned4(lse) || (idx_out && !aligned4(idx_out)) || !aligned16(ws))
    return MSA_ERR_INVALID_ARGUMENT;
  if (S < 1 || S > 65535 || max_len < 1 || H_q < 1 || H_kv < 1 || H_q % H_kv != 0 ||
      block_size != 64 || k < 1 || k > 64 || d_h < 1 || d_idx < 1)
    return MSA_ERR_INVALID_ARGUMENT;
  if (!pow2_upto(H_kv, 8) || !pow2_upto(H_q / H_kv, 8) || (d_h != 64 && d_h != 128) ||
      (d_idx != 32 && d_idx != 64))
    return MSA_ERR_UNSUPPORTED;
  const DecodeWs w = decode_layout(S, max_len, H_q, H_kv, d_h, k);
  if (ws_bytes < w.total) return MSA_ERR_WORKSPACE;
  cudaStream_t st = (cudaStream_t)stream;
  char* base = static_cast<char*>(ws);
  float* Mdec = reinterpret_cast<float*>(base + w.off_m);
  int32_t* idx = idx_out ? idx_out : reinterpret_cast<int32_t*>(base + w.off_idx);
  const int64_t nblk = (max_len + 63) / 64;
  const msa::CacheMap cm{cu_seqlens, nullptr, nullptr, 0, 0};
  cudaError_t e = msa::launch_decode_block_scores(q_idx, k_idx_cache, cm, Mdec, S, H_kv,
                                                  d_idx, max_len, nblk, st);
  if (e != cudaSuccess) return MSA_ERR_CUDA;
  e = msa::launch_decode_tail(q, k_cache, v_cache, Mdec, nblk, cm, S, max_len, H_q, H_kv, d_h, k,
                              idx, o, lse, st);
  return from_cuda(e);
}

// Varlen prefill: the whole packed batch in one launch per stage over a virtual row space in which
// each sequence starts on an aligned row (varlen.cu).  cu_seqlens is host memory: the launch
// sizes and the workspace layout depend on it.
namespace {
// the virtual row count of a valid batch, or -1
int64_t varlen_rows(const int64_t* cu_seqlens, int nseq, int H_kv) {
  if (!cu_seqlens || nseq < 1 || H_kv < 1 || cu_seqlens[0] != 0) return -1;
  const int64_t align = std::max<int64_t>(128, msa::index_rows_per_cta(H_kv));
  int64_t tv = 0;
  for (int s = 0; s < nseq; ++s) {
    const int64_t n = cu_seqlens[s + 1] - cu_seqlens[s];
    if (n < 1) return -1;
    tv += (n + align - 1) / align * align;
  }
  return tv;
}
}  // namespace

MSA_API size_t msa_prefill_varlen_workspace(const int64_t* cu_seqlens, int nseq, int H_q, int H_kv,
                                            int d_h, int k) {
  if (!cu_seqlens || nseq < 1 || H_kv < 1 || H_q < H_kv || H_q % H_kv != 0 || k < 1 || k > 64 ||
      d_h < 1)
    return 0;
  if (varlen_rows(cu_seqlens, nseq, H_kv) < 1) return 0;
  // d_idx is not an argument: the layout is sized for the largest supported index dim (64)
  return msa::varlen_layout(cu_seqlens, nseq, H_q, H_kv, d_h, 64, k).total;
}

MSA_API msa_status_t msa_prefill_varlen(const void* q, const void* k, const void* v,
                                        const void* q_idx, const void* k_idx,
                                        const int64_t* cu_seqlens, int nseq, int H_q, int H_kv,
                                        int d_h, int d_idx, int block_size, int k_blocks,
                                        int32_t* idx, void* o, float* lse, void* ws,
                                        size_t ws_bytes, void* stream) {
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(q_idx) || !aligned16(k_idx) ||
      !aligned4(idx) || !aligned16(o) || !aligned4(lse) || !aligned16(ws) || !cu_seqlens)
    return MSA_ERR_INVALID_ARGUMENT;
  if (nseq < 1 || H_q < 1 || H_kv < 1 || H_q % H_kv != 0 || d_h < 1 || d_idx < 1 ||
      block_size != 64 || k_blocks < 1 || k_blocks > 64 || cu_seqlens[0] != 0)
    return MSA_ERR_INVALID_ARGUMENT;
  for (int s = 0; s < nseq; ++s)
    if (cu_seqlens[s + 1] - cu_seqlens[s] < 1) return MSA_ERR_INVALID_ARGUMENT;
  if (!pow2_upto(H_kv, 8) || !pow2_upto(H_q / H_kv, 8) || (d_h != 64 && d_h != 128) ||
      (d_idx != 32 && d_idx != 64) || k_blocks > MSA_INDEX_SELECT_MAX_K)
    return MSA_ERR_UNSUPPORTED;
  const int64_t tv = varlen_rows(cu_seqlens, nseq, H_kv);
  if (tv * H_kv >= kMaxRows || tv > ((int64_t)1 << 21) || (int64_t)H_kv * tv * k_blocks >= kMaxRows)
    return MSA_ERR_UNSUPPORTED;
  if (ws_bytes < msa::varlen_layout(cu_seqlens, nseq, H_q, H_kv, d_h, 64, k_blocks).total)
    return MSA_ERR_WORKSPACE;
  return from_cuda(msa::launch_prefill_varlen(q, k, v, q_idx, k_idx, cu_seqlens, nseq, H_q, H_kv,
                                              d_h, d_idx, k_blocks, idx, o, lse, ws,
                                              (cudaStream_t)stream));
}

MSA_API msa_status_t msa_sparse_decode_paged(
    const void* q, const void* q_idx, const void* k_pages, const void* v_pages,
    const void* k_idx_pages, const int32_t* page_table, const int64_t* seq_lens, int S,
    int64_t max_pages, int64_t num_pages, int64_t max_len, int H_q, int H_kv, int d_h, int d_idx,
    int block_size, int k, void* o, float* lse, int32_t* idx_out, void* ws, size_t ws_bytes,
    void* stream) {
  if (!aligned16(q) || !aligned16(q_idx) || !aligned16(k_pages) || !aligned16(v_pages) ||
      !aligned16(k_idx_pages) || !aligned4(page_table) || !seq_lens ||
      ((uintptr_t)seq_lens & 7u) || !aligned16(o) || !aligned4(lse) ||
      (idx_out && !aligned4(idx_out)) || !aligned16(ws))
    return MSA_ERR_INVALID_ARGUMENT;
  if (S < 1 || S > 65535 || max_len < 1 || H_q < 1 || H_kv < 1 || H_q % H_kv != 0 ||
      block_size != 64 || k < 1 || k > 64 || d_h < 1 || d_idx < 1 || num_pages < 1 ||
      max_pages < 1 || max_pages * 64 < max_len)
    return MSA_ERR_INVALID_ARGUMENT;
  if (!pow2_upto(H_kv, 8) || !pow2_upto(H_q / H_kv, 8) || (d_h != 64 && d_h != 128) ||
      (d_idx != 32 && d_idx != 64))
    return MSA_ERR_UNSUPPORTED;
  const DecodeWs w = decode_layout(S, max_len, H_q, H_kv, d_h, k);
  if (ws_bytes < w.total) return MSA_ERR_WORKSPACE;
  cudaStream_t st = (cudaStream_t)stream;
  char* base = static_cast<char*>(ws);
  float* Mdec = reinterpret_cast<float*>(base + w.off_m);
  int32_t* idx = idx_out ? idx_out : reinterpret_cast<int32_t*>(base + w.off_idx);
  const int64_t nblk = (max_len + 63) / 64;
  const msa::CacheMap cm{nullptr, page_table, seq_lens, max_pages, num_pages};
  cudaError_t e = msa::launch_decode_block_scores(q_idx, k_idx_pages, cm, Mdec, S, H_kv, d_idx,
                                                  max_len, nblk, st);
  if (e != cudaSuccess) return MSA_ERR_CUDA;
  e = msa::launch_decode_tail(q, k_pages, v_pages, Mdec, nblk, cm, S, max_len, H_q, H_kv, d_h, k,
                              idx, o, lse, st);
  return from_cuda(e);
}

MSA_API size_t msa_kl_loss_fwd_workspace(int64_t N, int H_kv, int k) {
  if (N < 1 || H_kv < 1 || k < 1 || k > 64) return 0;
  return msa::kl_ws_bytes(N, H_kv, k);
}

MSA_API msa_status_t msa_kl_loss_fwd(const void* q, const void* k, const void* q_idx,
                                     const void* k_idx, const int32_t* idx, const float* lse,
                                     float* kl, float* lse_idx, float* p_sum, int64_t N, int H_q,
                                     int H_kv, int d_h, int d_idx, int block_size, int k_blocks,
                                     void* ws, size_t ws_bytes, void* stream) {
  if (!aligned16(q) || !aligned16(k) || !aligned16(q_idx) || !aligned16(k_idx) ||
      !aligned4(idx) || !aligned4(lse) || !aligned4(kl) || !aligned16(ws) ||
      (lse_idx && !aligned4(lse_idx)) || (p_sum && !aligned4(p_sum)))
    return MSA_ERR_INVALID_ARGUMENT;
  if (N < 1 || H_q < 1 || H_kv < 1 || H_q % H_kv != 0 || d_h < 1 || d_idx < 1 ||
      block_size != 64 || k_blocks < 1 || k_blocks > 64)
    return MSA_ERR_INVALID_ARGUMENT;
  if (!pow2_upto(H_kv, 8) || !pow2_upto(H_q / H_kv, 8) || (d_h != 64 && d_h != 128) ||
      (d_idx != 32 && d_idx != 64))
    return MSA_ERR_UNSUPPORTED;
  if (N > ((int64_t)1 << 21) || N * H_kv * k_blocks >= kMaxRows) return MSA_ERR_UNSUPPORTED;
  if (ws_bytes < msa::kl_ws_bytes(N, H_kv, k_blocks)) return MSA_ERR_WORKSPACE;
  return from_cuda(msa::launch_kl_loss_fwd(q, k, q_idx, k_idx, idx, lse, kl, lse_idx, p_sum, N,
                                           H_q, H_kv, d_h, d_idx, k_blocks, ws,
                                           (cudaStream_t)stream));
}

MSA_API size_t msa_kl_loss_bwd_workspace(int64_t N, int H_kv, int d_idx, int k) {
  if (N < 1 || H_kv < 1 || k < 1 || k > 64 || d_idx < 1) return 0;
  return msa::kl_bwd_ws_bytes(N, H_kv, d_idx, k);
}

MSA_API msa_status_t msa_kl_loss_bwd(const void* q, const void* k, const void* q_idx,
                                     const void* k_idx, const int32_t* idx, const float* lse,
                                     const float* lse_idx, const float* p_sum,
                                     const float* grad_kl, float* dq_idx, float* dk_idx, int64_t N,
                                     int H_q, int H_kv, int d_h, int d_idx, int block_size,
                                     int k_blocks, void* ws, size_t ws_bytes, void* stream) {
  if (!aligned16(q) || !aligned16(k) || !aligned16(q_idx) || !aligned16(k_idx) ||
      !aligned4(idx) || !aligned4(lse) || !aligned4(lse_idx) || !aligned4(p_sum) ||
      !aligned4(grad_kl) || !aligned16(dq_idx) || !aligned16(dk_idx) || !aligned16(ws))
    return MSA_ERR_INVALID_ARGUMENT;
  if (N < 1 || H_q < 1 || H_kv < 1 || H_q % H_kv != 0 || d_h < 1 || d_idx < 1 ||
      block_size != 64 || k_blocks < 1 || k_blocks > 64)
    return MSA_ERR_INVALID_ARGUMENT;
  if (!pow2_upto(H_kv, 8) || !pow2_upto(H_q / H_kv, 8) || (d_h != 64 && d_h != 128) ||
      (d_idx != 32 && d_idx != 64))
    return MSA_ERR_UNSUPPORTED;
  if (N > ((int64_t)1 << 21) || N * H_kv * k_blocks >= kMaxRows) return MSA_ERR_UNSUPPORTED;
  if (ws_bytes < msa::kl_bwd_ws_bytes(N, H_kv, d_idx, k_blocks)) return MSA_ERR_WORKSPACE;
  return from_cuda(msa::launch_kl_loss_bwd(q, k, q_idx, k_idx, idx, lse, lse_idx, p_sum, grad_kl,
                                           dq_idx, dk_idx, N, H_q, H_kv, d_h, d_idx, k_blocks, ws,
                                           (cudaStream_t)stream));
}

MSA_API msa_status_t msa_device_status(void) {
  unsigned v = 0, w = 0, x = 0, y = 0, z = 0;
  if (msa::read_reset_score_status(&v) != cudaSuccess) return MSA_ERR_CUDA;
  if (msa::read_reset_shared_status(&w) != cudaSuccess) return MSA_ERR_CUDA;
  if (msa::read_reset_kvo_status(&x) != cudaSuccess) return MSA_ERR_CUDA;
  if (msa::read_reset_kl_status(&y) != cudaSuccess) return MSA_ERR_CUDA;
  if (msa::read_reset_bwd_status(&z) != cudaSuccess) return MSA_ERR_CUDA;
  return (v | w | x | y | z) ? MSA_ERR_TIMEOUT : MSA_OK;
}

MSA_API msa_status_t msa_set_wait_limit_ns(uint64_t ns) {
  return from_cuda(msa::set_score_wait_limit((unsigned long long)ns));
}

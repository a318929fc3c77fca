// Internal launchers shared between the kernel translation units and the C ABI layer.
#pragma once

#include <algorithm>
#include <vector>

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace msa {

// Launches kernel<<<grid, block, smem, stream>>>(args...) with programmatic stream serialization:
// it may start while the previous kernel on the stream finishes, and must call pdl_wait() before
// reading that kernel's results.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// Byte offsets of the decode workspace: block scores [S, H_kv, ceil(max_len/64)] fp32 and
// selections [S, H_kv, k] int32 (when the caller passes no idx_out), each 256-byte aligned.
struct DecodeWs {
  size_t off_m, off_idx, total;
};
DecodeWs decode_layout(int S, int64_t max_len, int H_q, int H_kv, int d_h, int k);

// 2-D bf16 TMA descriptor over a row-major [outer, inner] tensor; box = box_inner x box_outer,
// swizzle_bytes in {0, 64, 128}.
cudaError_t make_tma_2d_bf16(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer,
                             int box_inner, int box_outer, int swizzle_bytes);

// 3-D bf16 TMA descriptor over a row-major [d2, d1, d0] tensor (d0 innermost); box
// box0 x box1 x box2, swizzle_bytes in {0, 64, 128}.
cudaError_t make_tma_3d_bf16(CUtensorMap* map, const void* base, uint64_t d0, uint64_t d1,
                             uint64_t d2, int box0, int box1, int box2, int swizzle_bytes);
// 4-D map with explicit byte strides of dims 1..3 (in any order: a box may gather dims whose
// strides are not increasing, e.g. the two 64-dim halves of G head rows)
cudaError_t make_tma_4d_bf16(CUtensorMap* map, const void* base, const uint64_t dims[4],
                             const uint64_t strides[3], const int box[4], int swizzle_bytes);

// Main branch of prefill: workspace bytes and the chunked launch sequence.
size_t sparse_attn_ws_bytes(int64_t N, int H_q, int H_kv, int d_h, int kk);
cudaError_t launch_sparse_attn_fwd(const void* q, const void* k, const void* v, const int32_t* idx,
                                   void* o, float* lse, int64_t N, int H_q, int H_kv, int d_h,
                                   int kk, void* ws, cudaStream_t stream);
cudaError_t read_reset_shared_status(unsigned* out);
cudaError_t read_reset_kvo_status(unsigned* out);
cudaError_t launch_attn_shared(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                               const void* q,
                               const int* tile_list, const unsigned long long* tile_priv,
                               const void* part_o,
                               const float* part_lse, void* o, float* lse, int64_t N, int64_t q0,
                               int64_t q1, int H_q, int H_kv, int d_h, int kk, cudaStream_t st);

cudaError_t launch_attn_plan(const int32_t* idx, int64_t N, int H_kv, int kk, int64_t q0,
                             int64_t q1, int64_t nblk, int* count, int* tile_list,
                             unsigned long long* tile_priv, int* sc, int* sc_n, cudaStream_t st);
cudaError_t launch_attn_scan(const int* count, int* offset, int* tile_off, int nb, int ept,
                             cudaStream_t st);
cudaError_t launch_attn_scatter(const int* sc, const int* sc_n, const int* offset, int* entries,
                                int64_t ntiles, int kk, cudaStream_t st);
cudaError_t launch_attn_kvouter(const void* q, const void* k, const void* v, const int* entries,
                                const int* offset, const int* tile_off, int nbuckets, int64_t nblk,
                                int64_t N, int64_t q0, int64_t q1, int H_q, int H_kv, int d_h,
                                int kk, int grid, void* part_o, float* part_lse,
                                cudaStream_t stream);
cudaError_t launch_index_block_scores(const void* q_idx, const void* k_idx, float* M, int64_t N,
                                      int H_kv, int d_idx, int64_t q_start, int64_t q_count,
                                      cudaStream_t stream);
// ktab (variable-length batches): per 128 rows, the first 128-key tile of the sequence that
// holds them; sequences then start on 128-row boundaries and no CTA's rows (index_rows_per_cta)
// span two of them.  Null: every row starts at key 0.
cudaError_t launch_index_select(const void* q_idx, const void* k_idx, int32_t* idx, int64_t N,
                                int H_kv, int d_idx, int k, int64_t q_start, int64_t q_count,
                                cudaStream_t stream, const int* ktab = nullptr);
int index_rows_per_cta(int H_kv);

// Variable-length prefill in one launch per stage (varlen.cu): the workspace layout over the
// virtual rows (each sequence padded to a multiple of `align` rows) and the launch sequence.
struct VarlenLayout {
  int64_t align, Tv;
  bool in_place;                       // virtual rows = packed rows: Q, K, V, O used in place
  size_t main, starts, ktab, idx, lse, q, k, v, qi, ki, o, total;
};
VarlenLayout varlen_layout(const int64_t* cu_seqlens, int nseq, int H_q, int H_kv, int d_h,
                           int d_idx, int k);
cudaError_t launch_prefill_varlen(const void* q, const void* k, const void* v, const void* q_idx,
                                  const void* k_idx, const int64_t* cu_seqlens, int nseq,
                                  int H_q, int H_kv, int d_h, int d_idx, int kk, int32_t* idx,
                                  void* o, float* lse, void* ws, cudaStream_t st);
cudaError_t read_reset_score_status(unsigned* out);
cudaError_t set_score_wait_limit(unsigned long long ns);

// KL alignment loss forward: workspace bytes and the launch sequence (plan, scan, block-major
// partials, merge).
size_t kl_ws_bytes(int64_t N, int H_kv, int kk);
size_t kl_bwd_ws_bytes(int64_t N, int H_kv, int d_idx, int kk);
cudaError_t launch_kl_loss_fwd(const void* q, const void* k, const void* q_idx, const void* k_idx,
                               const int32_t* idx, const float* lse, float* kl, float* lse_idx,
                               float* psum, int64_t N, int H_q, int H_kv, int d_h, int d_idx,
                               int kk, void* ws, cudaStream_t st);
cudaError_t launch_kl_loss_bwd(const void* q, const void* k, const void* q_idx, const void* k_idx,
                               const int32_t* idx, const float* lse, const float* lse_idx,
                               const float* psum, const float* grad_kl, float* dq_idx,
                               float* dk_idx, int64_t N, int H_q, int H_kv, int d_h, int d_idx,
                               int kk, void* ws, cudaStream_t st);
cudaError_t read_reset_kl_status(unsigned* out);
// Every selection of idx [H_kv, N, k] bucketed by (group, block) (entries (row << 6 | slot) in
// (16-query tile, query) order within a bucket; offsets and work-tile offsets of ept entries per
// tile, totals at index H_kv * ceil(N/64)).
cudaError_t launch_bucket_selections(const int32_t* idx, int64_t N, int H_kv, int kk, int ept,
                                     int* count, int* offset, int* tile_off, int* cursor,
                                     int* entries, cudaStream_t st);
// The same buckets with every bucket's entries in row order, independent of execution order;
// cnt_mat holds H_kv * ceil(N/64) * ordered_bucket_ranges(N) ints of scratch.
int ordered_bucket_ranges(int64_t N);
cudaError_t launch_bucket_selections_ordered(const int32_t* idx, int64_t N, int H_kv, int kk,
                                             int ept, int* count, int* offset, int* tile_off,
                                             int* cursor, int* cnt_mat, int* entries,
                                             cudaStream_t st);

// Backward of the main branch: workspace bytes and the launch sequence.
size_t sparse_attn_bwd_ws_bytes(int64_t N, int H_q, int H_kv, int d_h, int kk);
cudaError_t launch_sparse_attn_bwd(const void* q, const void* k, const void* v, const int32_t* idx,
                                   const void* o, const float* lse, const void* d_o, float* dq,
                                   float* dk, float* dv, int64_t N, int H_q, int H_kv, int d_h,
                                   int kk, void* ws, cudaStream_t st);
cudaError_t read_reset_bwd_status(unsigned* out);

cudaError_t launch_select_prefill(const float* M, int32_t* idx, int64_t N, int H_kv, int k,
                                  int64_t q_start, int64_t q_count, cudaStream_t stream);
// Where a decode sequence's cache rows live.  Packed: sequence s is rows cu[s] .. cu[s+1]-1 of the
// cache.  Paged: the cache is 64-token pages (one page per MSA block); token j of sequence s is
// row j % 64 of page pages[s * max_pages + j / 64], and the sequence is lens[s] tokens long.
// Lengths are clamped to [1, max_len] and page ids to [0, num_pages), so a bad length or page id
// gives wrong results, never an access outside the cache.  The packed layout trusts cu itself:
// its rows start at cu[s], so a cu[s] that is not a row of the cache addresses memory outside it.
struct CacheMap {
  const int64_t* cu;        // packed (nullptr when paged)
  const int32_t* pages;     // paged: [S, max_pages]
  const int64_t* lens;      // paged: [S]
  int64_t max_pages;
  int64_t num_pages;
#ifdef __CUDACC__
  // The kernels are instantiated per layout (PAGED), so the packed path carries no paged code.
  template <bool PAGED>
  __device__ __forceinline__ int64_t len(int64_t s, int64_t max_len) const {
    const int64_t L = PAGED ? __ldg(lens + s) : __ldg(cu + s + 1) - __ldg(cu + s);
    return L < 1 ? 1 : (L > max_len ? max_len : L);
  }
  // first cache row of sequence s when packed (0 when paged); read once per sequence
  template <bool PAGED>
  __device__ __forceinline__ int64_t seq_row(int64_t s) const { return PAGED ? 0 : __ldg(cu + s); }
  // cache row of token 64 * b of sequence s (the first token of its block b); row0 = seq_row(s)
  template <bool PAGED>
  __device__ __forceinline__ int64_t block_row(int64_t s, int64_t b, int64_t row0) const {
    if (!PAGED) return row0 + b * 64;
    int64_t pg = __ldg(pages + s * max_pages + b);
    pg = pg < 0 ? 0 : (pg >= num_pages ? num_pages - 1 : pg);
    return pg * 64;
  }
#endif
};

// The decode tail: per (sequence, group), the selection over the block scores Mdec and the
// attention of the group's heads over the selected blocks, writing o, lse and (if not null)
// idx_out.
cudaError_t launch_decode_tail(const void* q, const void* k_cache, const void* v_cache,
                               const float* Mdec, int64_t nblk_max, const CacheMap& cm, int S,
                               int64_t max_len, int H_q, int H_kv, int d_h, int kk,
                               int32_t* idx_out, void* o, float* lse, cudaStream_t stream);

cudaError_t launch_decode_block_scores(const void* q_idx, const void* k_idx_cache,
                                       const CacheMap& cm, float* Mdec, int S, int H_kv, int d_idx,
                                       int64_t max_len, int64_t nblk_max, cudaStream_t stream);

}  // namespace msa

/*
 * msa.h -- C ABI of the GB300 (sm_103a) MSA block-sparse GQA attention library
 * (libmsa.so).
 *
 * MSA (MiniMax Sparse Attention) as described in «MiniMax-M3：MSA 技术报告速读»
 * (MSA tech-report digest), section 核心机制：两个分支，先选后算:
 *   index branch:  S^{idx,(r)}_{i,j} = Q^idx(r)_i . K^idx_j / sqrt(d_idx)           (eq. S^idx)
 *                  M^{idx,(r)}_{i,b} = max_{j in block b, j <= i} S^{idx,(r)}_{i,j}   (eq. M^idx)
 *                  I^{(r)}_i = TopK_b(M^{idx,(r)}_{i,.}, k), local block always kept (eq. I^(r)_i)
 *   main branch:   O^{(h)}_i = softmax(Q^(h)_i K^(r)[I]^T / sqrt(d_h)) V^(r)[I]       (eq. O^(h)_i)
 *                  over the visible tokens (j <= i) of the selected blocks, shared by the
 *                  G = H_q/H_kv query heads of group r = h / G; the forward also emits the
 *                  per-row log-sum-exp (section Kernel).
 *   training:      the KL alignment loss between the main branch's group-averaged attention and
 *                  the index branch's softmax over the selected tokens (section 训练, eq. L_KL).
 *
 * Conventions (every entry point):
 *   - Pointers are DEVICE pointers owned by the caller; the library never allocates or
 *     frees memory and never synchronises.  Work is enqueued on `stream` (a cudaStream_t
 *     passed as void*; NULL = legacy default stream).
 *   - bf16 tensors are passed as `const void*` / `void*` (IEEE bfloat16 bit patterns),
 *     contiguous, row-major, 16-byte aligned base.
 *   - block_size must be 64.  Scales are fixed by the formulas (1/sqrt(d_idx), 1/sqrt(d_h)).
 *   - Supported shapes: H_kv in {1,2,4,8}; G = H_q/H_kv in {1,2,4,8}; d_h in {64,128};
 *     d_idx in {32,64}; 1 <= k <= 64.  Other valid shapes return MSA_ERR_UNSUPPORTED.
 *   - Inputs must be finite (no inf/NaN).
 *   - Host-side validation happens before any launch: a bad argument returns
 *     MSA_ERR_INVALID_ARGUMENT and enqueues nothing.  A launch failure returns
 *     MSA_ERR_CUDA.  Kernel-side waits are bounded; a wait that gives up records
 *     MSA_ERR_TIMEOUT in a device status word that msa_device_status() reports.
 *   - Selection ties go to the lower block index; selected indices are stored ascending
 *     and padded with -1 when fewer than k blocks are visible.
 *   - All functions are thread-safe (no mutable host state besides a lazily resolved
 *     driver entry point).
 */
#ifndef MSA_H_
#define MSA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    MSA_OK = 0,
    MSA_ERR_INVALID_ARGUMENT = 1, /* null/misaligned pointer, bad size, range outside [0,N) */
    MSA_ERR_UNSUPPORTED = 2,      /* valid shape this build has no kernel for            */
    MSA_ERR_WORKSPACE = 3,        /* ws_bytes smaller than the *_workspace() size         */
    MSA_ERR_CUDA = 4,             /* CUDA runtime/driver error at launch                  */
    MSA_ERR_TIMEOUT = 5           /* a bounded device-side wait gave up                   */
} msa_status_t;

/* Human-readable name of a status code (static string, never NULL). */
const char *msa_status_string(msa_status_t status);

/* Index branch: causal token scores max-pooled into block scores (eqs. S^idx and M^idx of
 * the digest's section 索引分支).  For query rows i in [q_start, q_start+q_count):
 *   M[r, i-q_start, b] = max_{j in [64b, min(64b+63, i)]} (q_idx[i,r,:] . k_idx[j,:]) / sqrt(d_idx)
 * and M = -inf for blocks b > floor(i/64) (max over an empty set).
 *   q_idx  bf16 [N, H_kv, d_idx]   one index query head per KV group
 *   k_idx  bf16 [N, d_idx]          one index key shared by all groups
 *   M      fp32 [H_kv, q_count, ceil(N/64)]  (written in full)
 * fp32 accumulation of bf16 products; on inputs whose products and sums are exact in
 * fp32 (small integers) M equals the exact value scaled and rounded once. */
msa_status_t msa_index_block_scores(const void *q_idx, const void *k_idx, float *M, int64_t N,
                                    int H_kv, int d_idx, int block_size, int64_t q_start,
                                    int64_t q_count, void *stream);

/* Per-group top-k block selection with the forced local block (eq. I^(r)_i and the local-
 * block rule of section 索引分支).  For each group r and row i in [q_start, q_start+q_count),
 * with l = floor(i/64):
 *   idx[r, i, :] = ascending( {l} U the k-1 blocks b < l with the largest M[r, i-q_start, b] )
 * ties broken toward the lower b; when l+1 <= k every visible block 0..l is selected and the
 * remaining k-(l+1) entries are -1.  Comparisons only (no exponentials).
 *   M    fp32 [H_kv, q_count, ceil(N/64)]  as written by msa_index_block_scores
 *   idx  int32 [H_kv, N, k]  only rows q_start..q_start+q_count-1 are written */
msa_status_t msa_select_blocks(const float *M, int32_t *idx, int64_t N, int H_kv, int block_size,
                               int k, int64_t q_start, int64_t q_count, void *stream);

/* Largest k msa_index_select supports (larger k: MSA_ERR_UNSUPPORTED; use
 * msa_index_block_scores + msa_select_blocks). */
#define MSA_INDEX_SELECT_MAX_K 32

/* The index branch in one pass: the block scores of msa_index_block_scores and the selection of
 * msa_select_blocks (eqs. S^idx, M^idx and I^(r)_i of section 索引分支), without writing M.
 * For each group r and row i in [q_start, q_start+q_count) it writes idx[r, i, :] exactly as
 * msa_select_blocks would from the M that msa_index_block_scores computes for the same inputs
 * (same fp32 block scores, same ordering (score desc, block asc), ascending, -1 padded).
 *   q_idx  bf16 [N, H_kv, d_idx];  k_idx bf16 [N, d_idx]
 *   idx    int32 [H_kv, N, k]  only rows q_start..q_start+q_count-1 are written
 * Needs no workspace.  k in [1, MSA_INDEX_SELECT_MAX_K]; other argument errors as
 * msa_index_block_scores and msa_select_blocks. */
msa_status_t msa_index_select(const void *q_idx, const void *k_idx, int32_t *idx, int64_t N,
                              int H_kv, int d_idx, int block_size, int k, int64_t q_start,
                              int64_t q_count, void *stream);

/* Workspace bytes msa_sparse_attn_fwd needs for these sizes (0 for invalid sizes).  It grows
 * with min(N, 65536) * H_q * k * d_h (the private-block partials of one 65536-row query chunk),
 * twice over when N > 65536 (two chunks in flight): 4.41 GB at H_q=32, k=16, d_h=128 for
 * N = 32768, 8.83 GB for N = 65536, 17.65 GB for any larger N. */
size_t msa_sparse_attn_fwd_workspace(int64_t N, int H_q, int H_kv, int d_h, int k);

/* Sparse main branch (eq. O^(h)_i of section 主分支, LSE of section Kernel).  For every row i
 * and query head h (group r = h / (H_q/H_kv)), over T = {j : floor(j/64) in idx[r,i,:], j <= i}:
 *   s_j = q[i,h,:] . k[j,r,:] / sqrt(d_h),   lse[h,i] = ln sum_{j in T} exp(s_j),
 *   o[i,h,:] = sum_{j in T} exp(s_j - lse[h,i]) v[j,r,:]
 *   q    bf16 [N, H_q, d_h];  k, v bf16 [N, H_kv, d_h];  idx int32 [H_kv, N, k]
 *        (entries -1 are skipped; entries must be distinct blocks <= floor(i/64) and must
 *        include floor(i/64), as msa_select_blocks writes them)
 *   o    bf16 [N, H_q, d_h] (fp32 accumulation, rounded to nearest even)
 *   lse  fp32 [H_q, N] (natural log)
 *   ws   device workspace, 16-byte aligned, of at least msa_sparse_attn_fwd_workspace() bytes
 *        (caller-owned; contents ignored on entry, unspecified on return; one call at a time
 *        per workspace).  Smaller: MSA_ERR_WORKSPACE.  N > 2^21: MSA_ERR_UNSUPPORTED.
 * Results do not depend on the launch order of work inside the call: the private-block
 * partials are merged per row in slot order, with no atomic updates of results.
 * With more than one 65536-row chunk, part of the work runs on a stream the library creates
 * once per device, ordered against `stream` by events; all of it has completed when `stream`
 * has passed the call. */
msa_status_t msa_sparse_attn_fwd(const void *q, const void *k, const void *v, const int32_t *idx,
                                 void *o, float *lse, int64_t N, int H_q, int H_kv, int d_h,
                                 int block_size, int k_blocks, void *ws, size_t ws_bytes,
                                 void *stream);

/* Workspace bytes msa_sparse_attn_bwd needs (0 for invalid sizes): per (group, block) bucket
 * counts and offsets, per selection an entry and a bf16 dQ partial of G*d_h values (the bulk:
 * 2*H_kv*N*k*G*d_h bytes, 17.2 GB at N = 131072, H_q = 32, H_kv = 4, k = 16, d_h = 128), per
 * (row, head) the delta dO . O, and one fp32 dK/dV partial of 2*64*d_h values per piece of at
 * most 64 work tiles of a bucket. */
size_t msa_sparse_attn_bwd_workspace(int64_t N, int H_q, int H_kv, int d_h, int k);

/* Backward of the sparse main branch (eq. O^(h)_i of section 主分支 differentiated; the
 * persistent, load-balanced backward of section Kernel).  With the forward's o and lse for the
 * same q, k, v, idx and the upstream gradient d_o, for every row i, head h (group r) and selected
 * visible token j (the forward's T_i):
 *   P_j = exp(q[i,h].k[j,r]/sqrt(d_h) - lse[h,i]),  D = d_o[i,h] . o[i,h],
 *   dS_j = P_j (d_o[i,h] . v[j,r] - D)
 *   dq[i,h,:] = sum_j dS_j k[j,r,:] / sqrt(d_h)
 *   dk[j,r,:] = sum_{(i,h): j in T_i} dS_j q[i,h,:] / sqrt(d_h),  dv[j,r,:] = sum_{(i,h)} P_j d_o[i,h,:]
 *   q, d_o, o  bf16 [N, H_q, d_h];  k, v bf16 [N, H_kv, d_h];  idx int32 [H_kv, N, k] (as the
 *              forward requires it);  lse fp32 [H_q, N] (the forward's, natural log)
 *   dq         fp32 [N, H_q, d_h];  dk, dv fp32 [N, H_kv, d_h] (written in full; tokens no query
 *              selected get 0)
 *   ws         device workspace of msa_sparse_attn_bwd_workspace() bytes, 16-byte aligned.
 * P and dS enter the tensor-core products as bf16, each selection's dQ contribution is kept in
 * bf16 until the merge, accumulation is fp32.  Every selection is
 * bucketed by (group, block) and each bucket cut into pieces of at most 64 work tiles; dq sums a
 * row's partials in slot order and dk/dv a bucket's pieces in piece order, with no atomic update
 * of any result, so the outputs are deterministic.  Errors as msa_sparse_attn_fwd; N > 2^21 or
 * H_kv * N * k >= 2^31: MSA_ERR_UNSUPPORTED. */
msa_status_t msa_sparse_attn_bwd(const void *q, const void *k, const void *v, const int32_t *idx,
                                 const void *o, const float *lse, const void *d_o, float *dq,
                                 float *dk, float *dv, int64_t N, int H_q, int H_kv, int d_h,
                                 int block_size, int k_blocks, void *ws, size_t ws_bytes,
                                 void *stream);

/* Workspace bytes msa_prefill_varlen needs (0 for invalid sizes); cu_seqlens is host memory
 * here.  The batch runs over Tv virtual rows, each sequence padded to a multiple of
 * max(128, 256 / H_kv) rows: the main-branch workspace of msa_sparse_attn_fwd for Tv rows, the
 * selections and LSEs over the virtual rows and, unless every length is such a multiple,
 * virtual copies of q, k, v, q_idx, k_idx and o (sized for d_idx = 64). */
size_t msa_prefill_varlen_workspace(const int64_t *cu_seqlens, int nseq, int H_q, int H_kv,
                                    int d_h, int k);

/* Batched / varlen prefill: the whole prefill path (msa_index_select, then msa_sparse_attn_fwd)
 * for each of nseq independent sequences packed along the token axis.  Sequence s is rows
 * cu_seqlens[s] .. cu_seqlens[s+1]-1 of every packed tensor, with causal attention inside the
 * sequence only (positions restart at 0 for each sequence).
 *   q      bf16 [T, H_q, d_h];  k, v bf16 [T, H_kv, d_h];  q_idx bf16 [T, H_kv, d_idx];
 *   k_idx  bf16 [T, d_idx];  T = cu_seqlens[nseq]
 *   o      bf16 [T, H_q, d_h]
 *   idx    int32: sequence s's selections [H_kv, N_s, k] at element offset cu_seqlens[s] * H_kv * k
 *   lse    fp32: sequence s's [H_q, N_s] at element offset cu_seqlens[s] * H_q
 *   cu_seqlens  int64 [nseq + 1], HOST memory, cu_seqlens[0] = 0, every sequence >= 1 token
 *   ws     device workspace of msa_prefill_varlen_workspace() bytes.
 * Each sequence's results equal those of the single-sequence calls on its rows, bit for bit.
 * The whole batch runs in one launch per stage: every sequence starts on an aligned row of a
 * virtual row space (see msa_prefill_varlen_workspace), where the index branch starts each
 * row's key range at its sequence's first block and the main branch runs unchanged; rows are
 * gathered into and scattered out of that space only when a length is not aligned.
 * k > MSA_INDEX_SELECT_MAX_K: MSA_ERR_UNSUPPORTED; other errors as the two calls. */
msa_status_t msa_prefill_varlen(const void *q, const void *k, const void *v, const void *q_idx,
                                const void *k_idx, const int64_t *cu_seqlens, int nseq, int H_q,
                                int H_kv, int d_h, int d_idx, int block_size, int k_blocks,
                                int32_t *idx, void *o, float *lse, void *ws, size_t ws_bytes,
                                void *stream);

/* Workspace bytes msa_sparse_decode needs (block scores, and the selections when idx_out is
 * NULL). */
size_t msa_sparse_decode_workspace(int S, int64_t max_len, int H_q, int H_kv, int d_h, int d_idx,
                                   int k);

/* Decode: the whole path (index scores, selection, main branch) for one new query per
 * sequence.  Sequence s occupies cache rows cu_seqlens[s] .. cu_seqlens[s+1]-1 (length
 * L_s >= 1, L_s <= max_len); its newest token, already appended, is the query at position
 * i = L_s - 1, so its local block is floor((L_s-1)/64).  Same formulas as the prefill calls
 * for that one row.
 *   q            bf16 [S, H_q, d_h]        q_idx  bf16 [S, H_kv, d_idx]
 *   k_cache      bf16 [sum L, H_kv, d_h]   v_cache bf16 [sum L, H_kv, d_h]
 *   k_idx_cache  bf16 [sum L, d_idx]       cu_seqlens int64 [S+1], cu_seqlens[0] = 0
 *   o            bf16 [S, H_q, d_h]        lse fp32 [S, H_q]
 *   idx_out      int32 [S, H_kv, k] or NULL (selected blocks, as msa_select_blocks)
 *   ws           device workspace of msa_sparse_decode_workspace() bytes.
 * cu_seqlens is read on the device only (the call never synchronises); lengths outside
 * [1, max_len] are a caller error that the kernels clamp rather than trust.  The offsets
 * themselves are trusted: every cu_seqlens[s] must be a row of the caches. */
msa_status_t msa_sparse_decode(const void *q, const void *q_idx, const void *k_cache,
                               const void *v_cache, const void *k_idx_cache,
                               const int64_t *cu_seqlens, int S, int64_t max_len, int H_q,
                               int H_kv, int d_h, int d_idx, int block_size, int k, void *o,
                               float *lse, int32_t *idx_out, void *ws, size_t ws_bytes,
                               void *stream);

/* Decode from a paged KV cache: the same computation as msa_sparse_decode, with each sequence's
 * cache held in 64-token pages -- one page per MSA block, so a selected block is one page.
 * Token j of sequence s is row j % 64 of page page_table[s * max_pages + j / 64]; the sequence
 * is seq_lens[s] tokens long and its newest token (position seq_lens[s] - 1) is the query.
 *   k_pages, v_pages   bf16 [num_pages, 64, H_kv, d_h]
 *   k_idx_pages        bf16 [num_pages, 64, d_idx]
 *   page_table         int32 [S, max_pages]  (entries past a sequence's last block are ignored)
 *   seq_lens           int64 [S], 1 <= seq_lens[s] <= max_len <= 64 * max_pages
 *   q, q_idx, o, lse, idx_out, ws: as msa_sparse_decode (ws of msa_sparse_decode_workspace()).
 * page_table and seq_lens are read on the device only; a length outside [1, max_len] or a page id
 * outside [0, num_pages) is a caller error that the kernels clamp rather than trust.  The results
 * equal those of msa_sparse_decode on the same tokens stored packed, bit for bit.
 * max_pages * 64 < max_len or num_pages < 1: MSA_ERR_INVALID_ARGUMENT; other errors as
 * msa_sparse_decode. */
msa_status_t msa_sparse_decode_paged(const void *q, const void *q_idx, const void *k_pages,
                                     const void *v_pages, const void *k_idx_pages,
                                     const int32_t *page_table, const int64_t *seq_lens, int S,
                                     int64_t max_pages, int64_t num_pages, int64_t max_len,
                                     int H_q, int H_kv, int d_h, int d_idx, int block_size, int k,
                                     void *o, float *lse, int32_t *idx_out, void *ws,
                                     size_t ws_bytes, void *stream);

/* Size of the fixed device scratch used by msa_sparse_decode_noalloc (8 MiB). */
#define MSA_DECODE_NOALLOC_SCRATCH_BYTES (8u << 20)

/* Decode exactly as msa_sparse_decode, for callers that cannot allocate device memory where they
 * decode (a runtime that reserved all device memory for its own pool, or a latency-critical loop
 * that must not call cudaMalloc/cudaFree, which can block or synchronise).  The paper has no
 * counterpart to this entry point; it changes where the scratch lives, not what is computed.
 *   - Arguments and results are those of msa_sparse_decode without ws/ws_bytes; the caller still
 *     owns and passes every input and output.  Nothing is allocated by the call.
 *   - The temporaries (block scores, selections) live in a fixed device array of
 *     MSA_DECODE_NOALLOC_SCRATCH_BYTES inside libmsa.so, held by every GPU that loads the library
 *     until the process exits.  Sizes whose msa_sparse_decode_workspace() exceeds it return
 *     MSA_ERR_WORKSPACE before any launch.
 *   - The first call on each device looks up the array's device address (cudaGetSymbolAddress)
 *     with that device current; make that first call before capturing any stream.  The address
 *     is kept for the life of the process: after a device reset (cudaDeviceReset, or anything
 *     else that destroys and re-creates the device's primary context) the library may load at
 *     another address, so do not call this entry point on that device again in that process.
 *   - All calls share the array and it keeps the last call's contents (nothing in it needs to
 *     start at zero).  Calls whose GPU work overlaps -- on different streams or from different
 *     host threads on one device -- race on it and must be serialised by the caller. */
msa_status_t msa_sparse_decode_noalloc(const void *q, const void *q_idx, const void *k_cache,
                                       const void *v_cache, const void *k_idx_cache,
                                       const int64_t *cu_seqlens, int S, int64_t max_len, int H_q,
                                       int H_kv, int d_h, int d_idx, int block_size, int k,
                                       void *o, float *lse, int32_t *idx_out, void *stream);

/* Workspace bytes msa_kl_loss_fwd needs (0 for invalid sizes): per (group, block) bucket counts
 * and offsets, and per selection an entry and a 16-byte partial -- 20 * H_kv * N * k bytes plus
 * 16 * H_kv * ceil(N/64) (168 MB at N = 131072, H_kv = 4, k = 16). */
size_t msa_kl_loss_fwd_workspace(int64_t N, int H_kv, int k);

/* Forward of the KL alignment loss that trains the index branch (section 训练：top-k 不可导怎么办
 * of the digest, eqs. P^idx, P and L_KL; the LSE it needs is the main branch's, section Kernel).
 * For every group r and row i, over the selected token set T = {j : floor(j/64) in idx[r,i,:],
 * j <= i} (the main branch's T):
 *   teacher  P_j     = (1/G) sum_{h = rG .. rG+G-1} exp(q[i,h,:] . k[j,r,:] / sqrt(d_h) - lse[h,i])
 *   student  P^idx_j = exp(S^idx_j) / sum_{u in T} exp(S^idx_u),  S^idx_j = q_idx[i,r,:] . k_idx[j,:] / sqrt(d_idx)
 *   kl[r, i] = sum_{j in T} P_j (ln P_j - ln P^idx_j)      (terms with P_j = 0 count 0)
 * No reduction over rows or groups is applied (the caller averages as its training step needs).
 *   q    bf16 [N, H_q, d_h];  k bf16 [N, H_kv, d_h];  q_idx bf16 [N, H_kv, d_idx];
 *   k_idx bf16 [N, d_idx];  idx int32 [H_kv, N, k] (as msa_sparse_attn_fwd requires it);
 *   lse  fp32 [H_q, N], the natural-log LSE msa_sparse_attn_fwd wrote for the same q, k, idx
 *        (with another lse the teacher rows do not sum to 1 and the result is not a KL);
 *   kl   fp32 [H_kv, N];
 *   lse_idx, p_sum  fp32 [H_kv, N] or NULL: the student's LSE over T (natural log) and the
 *        teacher's mass sum_j P_j, which msa_kl_loss_bwd takes;
 *   ws   device workspace of at least msa_kl_loss_fwd_workspace() bytes, 16-byte aligned
 *        (contents ignored on entry, unspecified on return; one call at a time per workspace).
 * fp32 arithmetic from bf16 inputs.  Each selection's contribution is computed independently
 * and a row's contributions are combined in slot order, with no atomic update of any result.
 * Errors as msa_sparse_attn_fwd; N > 2^21 or H_kv * N * k >= 2^31: MSA_ERR_UNSUPPORTED. */
msa_status_t msa_kl_loss_fwd(const void *q, const void *k, const void *q_idx, const void *k_idx,
                             const int32_t *idx, const float *lse, float *kl, float *lse_idx,
                             float *p_sum, int64_t N, int H_q, int H_kv, int d_h, int d_idx,
                             int block_size, int k_blocks, void *ws, size_t ws_bytes,
                             void *stream);

/* Workspace bytes msa_kl_loss_bwd needs: that of msa_kl_loss_fwd plus one d_idx-float partial of
 * dQ_idx per selection, 64 x d_idx floats of dK_idx partial per (bucket, CTA, epilogue group)
 * slot for 2 (H_kv * ceil(N/64) + 1024) slots, and the row-ordered bucketing's counters (one
 * int per bucket and range of 1024 rows): 2.62 GB at N = 131072, H_kv = 4, k = 16, d_idx = 64. */
size_t msa_kl_loss_bwd_workspace(int64_t N, int H_kv, int d_idx, int k);

/* Gradient of the KL alignment loss with respect to the index branch (part of the training
 * backward; the teacher is held fixed -- the gradient detach of section 训练).  For the scalar
 * L = sum_{r,i} grad_kl[r,i] * kl[r,i], with kl as msa_kl_loss_fwd defines it:
 *   dS_j = grad_kl[r,i] * (p_sum[r,i] * P^idx_j - P_j) / sqrt(d_idx)   for j in T (else 0)
 *   dq_idx[i,r,:] = sum_j dS_j k_idx[j,:],   dk_idx[j,:] = sum over (r,i) with j in T of dS_j q_idx[i,r,:]
 * where P^idx_j = exp(q_idx[i,r,:].k_idx[j,:]/sqrt(d_idx) - lse_idx[r,i]) and P_j the teacher.
 *   lse_idx, p_sum  fp32 [H_kv, N] as msa_kl_loss_fwd wrote them for the same inputs
 *   grad_kl         fp32 [H_kv, N]  the upstream gradient of each row's loss
 *   dq_idx          fp32 [N, H_kv, d_idx] (written);  dk_idx fp32 [N, d_idx] (written)
 *   other arguments as msa_kl_loss_fwd; ws of msa_kl_loss_bwd_workspace() bytes.
 * dq_idx sums its row's selections in slot order; dk_idx sums, per token, one partial per
 * (group, CTA of the block-major pass, epilogue group) in that order, with no atomic update of
 * any result, so repeated calls on one device give identical bits.  G = H_q/H_kv in
 * {1, 2, 4, 8} (otherwise MSA_ERR_UNSUPPORTED). */
msa_status_t msa_kl_loss_bwd(const void *q, const void *k, const void *q_idx, const void *k_idx,
                             const int32_t *idx, const float *lse, const float *lse_idx,
                             const float *p_sum, const float *grad_kl, float *dq_idx,
                             float *dk_idx, int64_t N, int H_q, int H_kv, int d_h, int d_idx,
                             int block_size, int k_blocks, void *ws, size_t ws_bytes,
                             void *stream);

/* Reads and clears the device status words of the current device (synchronising call).
 * Returns MSA_ERR_TIMEOUT if any kernel since the last call gave up a bounded wait,
 * MSA_ERR_CUDA if the read itself failed, MSA_OK otherwise.
 * The status words are per device and per library, not per call: several calls may share one
 * stream or workspace-free entry points (msa_index_block_scores, msa_select_blocks,
 * msa_index_select) have no workspace to hold a status word, so a timeout is reported for
 * the device since the last read; read it after synchronising the calls you want covered. */
msa_status_t msa_device_status(void);

/* Time limit, in nanoseconds, of the pipeline waits (ring slots and accumulator hand-offs)
 * inside the index-branch kernel -- the kernel of msa_index_block_scores and msa_index_select,
 * also run by msa_prefill_varlen -- on the current device; the default is 2e9 (2 s).  A wait
 * that reaches the limit gives up: the kernel stops its loops, waits for the copies and MMAs it
 * has in flight (those waits keep the fixed 2 s bound), frees its tensor memory and records
 * MSA_ERR_TIMEOUT for msa_device_status(); that call's outputs are unspecified.  ns = 0 makes
 * every pipeline wait that is not already satisfied give up at once, which exercises the
 * timeout path without any fault.  Every other kernel keeps the fixed 2 s bound.
 * Synchronising call (it writes a device variable); MSA_ERR_CUDA if that write failed. */
msa_status_t msa_set_wait_limit_ns(uint64_t ns);

#ifdef __cplusplus
}
#endif

#endif /* MSA_H_ */

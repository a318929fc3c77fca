// KL alignment loss, forward («MiniMax-M3：MSA 技术报告速读», section 训练：top-k 不可导怎么办,
// eqs. P^idx, P and L_KL; the kernel section's note that the LSE the sparse KL loss needs is
// produced by the forward).  For each group r and row i, over the selected token set T (the
// visible tokens of the blocks in idx[r, i, :], the main branch's own T):
//   teacher  P_j = (1/G) sum_{h in group r} exp(s^h_j - LSE[h, i]),  s^h_j = Q[i,h].K[j,r]/sqrt(d_h)
//   student  P^idx_j = exp(S^idx_j - LSE^idx),  S^idx_j = Q_idx[i,r].K_idx[j]/sqrt(d_idx)
//   KL[r, i] = sum_{j in T} P_j (ln P_j - S^idx_j) + LSE^idx * sum_{j in T} P_j
// The forward's LSE normalises each teacher head, so the teacher needs no second pass over T;
// the student's normaliser LSE^idx is merged like a split softmax.
//
// Organisation: the same KV-outer scheme as the main branch's block-major pass.  Every
// selection (row, slot) is bucketed by (group, block); a work tile stacks up to 128/G entries of
// one bucket, G rows each, into one 128-row UMMA tile, per TMEM stage:
//   S     = Q_stack [128 x d_h] . K_b^T [d_h x 64]              columns [0, 64)
//   S^i^T = K_idx_b [64 tokens on M] . Qi^T [d_idx x entries]    columns [64, 64 + 128/G)
// (the student scores transposed, one index-query row per entry, moved to (entry, token) order
// through shared memory).  The teacher's head mean is a reduce-scatter over the entry's G lanes
// by shuffles, after which each lane owns 64/G of the block's tokens; each entry leaves one
// partial (sum P (ln P - S^idx), sum P, and the student's max and sum of exponentials in the log2
// domain) at the fixed position of its (group, row, slot).  A merge kernel combines a row's
// partials in slot order: no atomic update of any result.
// One persistent, warp-specialized CTA per SM: producer warps (query rows by TMA, keys and index
// queries by cp.async), an MMA warp, and two epilogue groups taking alternate tiles.
//
// Gradient (the BWD instantiation, G = 8): the same pass recomputes teacher and student per
// tile and turns them into dS = g (W P^idx - P) / sqrt(d_idx); dQ_idx per selection (partials,
// merged in slot order) and dK_idx per block (fp32 atomics per run of tiles of one block).
#include <cmath>

#include "attn_tile.cuh"
#include "msa_device.cuh"
#include "msa_internal.h"

namespace msa {
namespace {

__device__ unsigned g_kl_status = 0;

constexpr int kKlRows = 128;                 // UMMA M
constexpr int kKlPlanWarps = 4;
constexpr float kLn2 = 0.693147180559945309f;
constexpr float kLog2e = 1.442695040888963407f;

// One persistent CTA per SM (its TMEM stages take all 512 columns).  Shared memory holds a ring
// of query stages -- the tile's stacked query rows and its entries' index queries, one row per
// entry -- a ring of two key stages (K_b and K_idx_b of one bucket) and, per epilogue group, the
// tile's student scores transposed to (entry, token).  TMEM holds kTStages accumulator stages:
// S (128 rows x 64 tokens) and the student scores (64 tokens on the lanes x the tile's entries).
constexpr int kSiStride = 68;
// TCG (gradient pass; d_idx = 64 and G = 4, 8, or 2 at d_h = 64): the gradient products run on
// the tensor core.  Per
// epilogue group: dS in bf16 split into hi + lo (so the products keep about fp32 accuracy) as
// [entry][64 tokens] rows of 128 bytes, and a copy of the bucket's K_idx block [64 tokens][64
// dims], both in the 128-byte swizzle; the tile's index queries are stored swizzled as well.
template <int D_H, int G, bool BWD = false, bool TCG = false>
struct KlSmem {
  static constexpr int kEpt = kKlRows / G;        // entries per work tile
  static constexpr int kHalves = D_H / 64;
  static constexpr int kQHalf = kKlRows * 128;    // 128 rows x 64 dims, bf16, SW128
  static constexpr int kKHalf = 64 * 128;         // 64 keys x 64 dims
  static constexpr int kQiBytes = kEpt * 128 < 1024 ? 1024 : kEpt * 128;
  // (the gradient pass at G = 1, d_h = 128 keeps one query stage: two do not fit with its
  // per-group index-query copies)
  static constexpr int kQStages =
      G == 8 ? 4 : (G == 4 ? 3 : (BWD && G == 1 && D_H == 128 ? 1 : 2));
  static constexpr int kKStages = 2;
  static constexpr int kTCols = 64 + kEpt <= 128 ? 128 : 256;
  // TCG: two score stages; the other half of TMEM holds each group's dQ_idx^T (kEpt columns)
  // and dK_idx (64 columns) accumulators at kColGrad + 128 grp
  static constexpr int kTStages = TCG ? 2 : 512 / kTCols;
  static constexpr uint32_t kColGrad = 2u * kTCols;
  static constexpr int kQStage = kHalves * kQHalf + kQiBytes;
  static constexpr int kKStage = kHalves * kKHalf + kKHalf;
  static constexpr int kOffQ = 0;
  static constexpr int kOffK = kOffQ + kQStages * kQStage;
  // the student MMA reads 128 rows of K_idx_b, the last 64 of them past the stage (ignored
  // lanes): the transposed-score buffers (>= 8 KB) follow the key stages
  static constexpr int kOffSi = kOffK + kKStages * kKStage;
  // per epilogue group: [entry][token] at a row stride of kSiStride floats (68: rows of different
  // entries fall in different banks, and each row stays 16-byte aligned)
  static constexpr int kSiBytes = kEpt * kSiStride * 4;
  // gradient pass, per epilogue group: the tile's index queries (one 128-byte row per entry)
  static constexpr int kOffQg =
      TCG ? (kOffSi + 2 * kSiBytes + 1023) / 1024 * 1024 : kOffSi + 2 * kSiBytes;
  static constexpr int kQgBytes = BWD ? kEpt * 128 : 0;
  static constexpr int kDsBytes = TCG ? kEpt * 128 : 0;      // per group and half (hi, lo)
  static constexpr int kKgBytes = TCG ? 64 * 128 : 0;        // per group
  static constexpr int kOffKg = kOffQg + 2 * kQgBytes;
  static constexpr int kOffDs = kOffKg + 2 * kKgBytes;
  // the MN-major operands of the gradient MMAs span M = 128 of which rows 64..127 are unused:
  // those reads land up to 1 KB past a tile, inside the next tile or this zeroed pad
  static constexpr int kPad = TCG ? 1024 : 0;
  static constexpr int kOffBar = kOffDs + 4 * kDsBytes + kPad;
  // + per group the completion of its gradient MMAs (TCG)
  static constexpr int kNumBars = 2 * kQStages + 2 * kKStages + 2 * kTStages + (TCG ? 2 : 0);
  static constexpr int kOffMisc = kOffBar + 8 * kNumBars;
  static constexpr int kOffPEnt = kOffMisc + 16;  // each producer warp's copy of a tile's entries
  static constexpr int kBytes = kOffPEnt + 2 * 4 * kKlRows;
  // more than half of the SM's shared memory: one CTA per SM
  static constexpr int kAlloc = kBytes + 1024 > 116 * 1024 ? kBytes + 1024 : 116 * 1024;
  static_assert(kQStage % 1024 == 0 && kKStage % 1024 == 0, "swizzle atoms");
  static_assert(2 * kSiBytes >= 8 * 1024, "rows 64..127 of the student A operand stay in bounds");
  static_assert(kAlloc <= 227 * 1024, "shared memory");
  static_assert(!TCG || (G >= 2 && kEpt <= 64 && kTCols == 128 && kColGrad + 256 <= 512),
                "TCG layout");
  static_assert(!TCG || (kOffQg % 1024 == 0 && kQgBytes % 1024 == 0 && kDsBytes % 1024 == 0),
                "swizzle atoms");
};

__device__ __forceinline__ void kl_cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void kl_zero16(uint32_t dst) {
  asm volatile("st.shared.v4.b32 [%0], {%1,%1,%1,%1};" ::"r"(dst), "r"(0u) : "memory");
}

// ----------------------------------------------------------------- planning --
// Per 16-query tile (one warp): the tile's selections as a union of blocks with query masks
// (tile_union).  Pass 0 counts each block's selections in its (group, block) bucket; pass 1
// reserves a contiguous range of the bucket per (tile, block) and writes each selection as
// (row << 6 | slot) at its place in that range.
template <int EPL>
__device__ __forceinline__ void kl_plan_tile(const int32_t* __restrict__ idx, int r, int64_t i0,
                                             int64_t N, int kk, int64_t nblk, int pass, int* s_U,
                                             unsigned* s_mask, int* count, const int* offset,
                                             int* cursor, int* entries) {
  const int lane = threadIdx.x & 31;
  int x[EPL], rank[EPL];
  const int nU = tile_union<EPL>(idx, r, i0, N, N, kk, x, rank, s_U, s_mask);
  for (int u = lane; u < nU; u += 32) {
    const int64_t bucket = (int64_t)r * nblk + s_U[u];
    const int n = __popc(s_mask[u]);
    if (pass == 0)
      atomicAdd(count + bucket, n);
    else
      s_U[u] = offset[bucket] + atomicAdd(cursor + bucket, n);   // start of this tile's range
  }
  if (pass == 0) return;
  __syncwarp();
#pragma unroll
  for (int j = 0; j < EPL; ++j) {
    const int key = x[j];
    if (key == INT_MAX) continue;
    const int w = TileKeys::query(key);
    const int pos = s_U[rank[j]] + __popc(s_mask[rank[j]] & ((1u << w) - 1u));
    entries[pos] = (int)(((i0 + w) << 6) | TileKeys::slot(key));
  }
}

// The planning kernels are instantiated per keys-per-lane EPL (32 EPL >= 16 k), so their
// registers and shared memory fit the k in use.
template <int EPL>
__global__ void __launch_bounds__(32 * kKlPlanWarps)
    k_kl_plan(const int32_t* __restrict__ idx, int64_t N, int kk, int64_t nblk, int pass,
              int* count, const int* offset, int* cursor, int* entries) {
  __shared__ int s_U[kKlPlanWarps][32 * EPL];
  __shared__ unsigned s_mask[kKlPlanWarps][32 * EPL];
  const int warp = threadIdx.x >> 5;
  const int r = blockIdx.y;
  const int64_t i0 = ((int64_t)blockIdx.x * kKlPlanWarps + warp) * kTileQ;
  if (i0 >= N) return;
  kl_plan_tile<EPL>(idx, r, i0, N, kk, nblk, pass, s_U[warp], s_mask[warp], count, offset,
                    cursor, entries);
}

// Launches kern<EPL> for the EPL that k needs.
template <template <int> class K, typename... A>
cudaError_t launch_epl(int kk, dim3 grid, dim3 block, cudaStream_t st, A... args) {
  if (kk <= 2) K<1>::launch(grid, block, st, args...);
  else if (kk <= 4) K<2>::launch(grid, block, st, args...);
  else if (kk <= 8) K<4>::launch(grid, block, st, args...);
  else if (kk <= 16) K<8>::launch(grid, block, st, args...);
  else if (kk <= 32) K<16>::launch(grid, block, st, args...);
  else K<32>::launch(grid, block, st, args...);
  return cudaGetLastError();
}
template <int EPL>
struct KlPlanK {
  template <typename... A>
  static void launch(dim3 g, dim3 b, cudaStream_t st, A... a) { k_kl_plan<EPL><<<g, b, 0, st>>>(a...); }
};

// ------------------------------------------------- row-ordered bucketing --
// The same buckets with every bucket's selections in row order, whatever order the hardware
// runs the warps in: counts per bucket and per (bucket, range of kRangeTiles tiles), bases from
// an exclusive scan over a bucket's ranges, then one warp per range that walks its tiles in order
// and alone advances that range's cursors.
constexpr int kRangeTiles = 64;

template <int EPL>
__device__ __forceinline__ void order_count_tile(const int32_t* __restrict__ idx, int r, int64_t i0,
                                                 int64_t N, int kk, int64_t nblk, int R, int range,
                                                 int* s_U, unsigned* s_mask, int* count,
                                                 int* cnt_mat) {
  const int lane = threadIdx.x & 31;
  int x[EPL], rank[EPL];
  const int nU = tile_union<EPL>(idx, r, i0, N, N, kk, x, rank, s_U, s_mask);
  for (int u = lane; u < nU; u += 32) {
    const int64_t bucket = (int64_t)r * nblk + s_U[u];
    const int n = __popc(s_mask[u]);
    atomicAdd(count + bucket, n);
    atomicAdd(cnt_mat + bucket * R + range, n);
  }
}

template <int EPL>
__global__ void __launch_bounds__(32 * kKlPlanWarps)
    k_order_count(const int32_t* __restrict__ idx, int64_t N, int kk, int64_t nblk, int R,
                  int* count, int* cnt_mat) {
  __shared__ int s_U[kKlPlanWarps][32 * EPL];
  __shared__ unsigned s_mask[kKlPlanWarps][32 * EPL];
  const int warp = threadIdx.x >> 5;
  const int r = blockIdx.y;
  const int64_t t = (int64_t)blockIdx.x * kKlPlanWarps + warp;
  const int64_t i0 = t * kTileQ;
  if (i0 >= N) return;
  order_count_tile<EPL>(idx, r, i0, N, kk, nblk, R, (int)(t / kRangeTiles), s_U[warp],
                        s_mask[warp], count, cnt_mat);
}
template <int EPL>
struct OrderCountK {
  template <typename... A>
  static void launch(dim3 g, dim3 b, cudaStream_t st, A... a) { k_order_count<EPL><<<g, b, 0, st>>>(a...); }
};

// cnt_mat[b][range] := offset[b] + sum of the bucket's counts in earlier ranges
__global__ void __launch_bounds__(256)
    k_order_bases(const int* __restrict__ offset, int* cnt_mat, int nb, int R) {
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= nb) return;
  int run = offset[b];
  int* row = cnt_mat + (int64_t)b * R;
  for (int g = 0; g < R; ++g) {
    const int c = row[g];
    row[g] = run;
    run += c;
  }
}

template <int EPL>
__device__ __forceinline__ void order_scatter_range(const int32_t* __restrict__ idx, int r,
                                                    int range, int64_t N, int kk, int64_t nblk,
                                                    int R, int* s_U, unsigned* s_mask,
                                                    int* cnt_mat, int* entries) {
  const int lane = threadIdx.x & 31;
  const int64_t t_end = (N + kTileQ - 1) / kTileQ;
  for (int64_t t = (int64_t)range * kRangeTiles; t < t_end && t < (int64_t)(range + 1) * kRangeTiles;
       ++t) {
    const int64_t i0 = t * kTileQ;
    int x[EPL], rank[EPL];
    const int nU = tile_union<EPL>(idx, r, i0, N, N, kk, x, rank, s_U, s_mask);
    // each union block is a different bucket: its lane alone moves that bucket's cursor
    for (int u = lane; u < nU; u += 32) {
      int* cur = cnt_mat + ((int64_t)r * nblk + s_U[u]) * R + range;
      const int pos = *cur;
      *cur = pos + __popc(s_mask[u]);
      s_U[u] = pos;
    }
    __syncwarp();
#pragma unroll
    for (int j = 0; j < EPL; ++j) {
      const int key = x[j];
      if (key == INT_MAX) continue;
      const int w = TileKeys::query(key);
      const int pos = s_U[rank[j]] + __popc(s_mask[rank[j]] & ((1u << w) - 1u));
      entries[pos] = (int)(((i0 + w) << 6) | TileKeys::slot(key));
    }
    __syncwarp();
  }
}

template <int EPL>
__global__ void __launch_bounds__(32 * kKlPlanWarps)
    k_order_scatter(const int32_t* __restrict__ idx, int64_t N, int kk, int64_t nblk, int R,
                    int* cnt_mat, int* entries) {
  __shared__ int s_U[kKlPlanWarps][32 * EPL];
  __shared__ unsigned s_mask[kKlPlanWarps][32 * EPL];
  const int warp = threadIdx.x >> 5;
  const int r = blockIdx.y;
  const int range = blockIdx.x * kKlPlanWarps + warp;
  if (range >= R) return;
  order_scatter_range<EPL>(idx, r, range, N, kk, nblk, R, s_U[warp], s_mask[warp], cnt_mat,
                           entries);
}
template <int EPL>
struct OrderScatterK {
  template <typename... A>
  static void launch(dim3 g, dim3 b, cudaStream_t st, A... a) { k_order_scatter<EPL><<<g, b, 0, st>>>(a...); }
};

// ------------------------------------------------------- block-major partials --
// Reduce-scatter over the G lanes of an entry (lanes e*G .. e*G+G-1 of one warp, h = lane's
// head): afterwards lane h holds, in a[0 .. 64/G), the sums over the G lanes of columns
// (64/G)*h .. (64/G)*h + 64/G - 1.  Each step halves the width: the lane whose step bit is set
// keeps the upper half and sends the lower one.
template <int G, bool ADD>
__device__ __forceinline__ void lane_split(float (&a)[64], int h) {
#pragma unroll
  for (int st = 0; (G >> (st + 1)) >= 1; ++st) {
    const int m = G >> (st + 1);
    const int half = 32 >> st;
    const bool hi = (h & m) != 0;
#pragma unroll
    for (int c = 0; c < half; ++c) {
      const float keep = hi ? a[c + half] : a[c];
      if (ADD) {
        const float send = hi ? a[c] : a[c + half];
        a[c] = keep + __shfl_xor_sync(0xffffffffu, send, m);
      } else {
        a[c] = keep;
      }
    }
  }
}

#define KL_TMEM_LD16(taddr, r)                                                                  \
  asm volatile(                                                                                 \
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "                                                 \
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"                         \
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),     \
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), \
        "=r"(r[14]), "=r"(r[15])                                                                \
      : "r"(taddr))

__device__ __forceinline__ void kl_group_sync(int id) {
  asm volatile("bar.sync %0, 128;" ::"r"(id) : "memory");
}
// Barrier of one epilogue group (four warps) that also ANDs a predicate over its 128 threads:
// the only place where a group may leave its loop, so all four warps leave together.
__device__ __forceinline__ bool kl_group_and(int id, bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\tbar.red.and.pred q, %2, 128, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)v), "r"(id)
      : "memory");
  return r != 0;
}

// Q as [N, H_q, d_h] with boxes of 64 dims x G heads x 2^m consecutive tokens (m = 0..4): a run
// of consecutive query rows among a tile's entries (the queries of one 16-query tile that chose
// the same block land next to each other in its bucket) loads with a few large boxes instead of
// one box per row.
struct KlQMaps {
  CUtensorMap m[5];
};

// Warp roles: warps 0 and 11.. load the query rows (their TMA boxes dealt round-robin: a warp
// issues one box at a time, so several warps keep more of them in flight), warp 10 loads the
// keys and index queries, warp 1 issues the MMAs, warps 2..9 are two epilogue groups of four
// (one warp per TMEM lane quarter) that take alternate work tiles.
// The gradient pass keeps per-thread key-gradient accumulators, so it runs one query-row warp
// (more registers per thread) where the loss pass runs four.
template <bool BWD>
struct KlWarps {
  static constexpr int kQ = BWD ? 1 : 4;            // query-row warps
  static constexpr int kAll = 10 + 1 + (kQ - 1);
  static constexpr int kThreads = 32 * kAll;
};

// Gradient inputs and outputs (the BWD instantiation only): per row the upstream gradient, the
// student's LSE over T and the teacher's mass, from the loss pass; per selection a partial of
// dQ_idx (d_idx floats at its (group, row, slot) position); dK_idx accumulated in fp32.
struct KlGrad {
  const float* grad_kl;     // [H_kv, N]
  const float* lse_idx;     // [H_kv, N], natural log
  const float* psum;        // [H_kv, N]
  float* part_dq;           // [H_kv, N, k, d_idx]
  float* part_dk;           // [(buckets + CTAs) * 2, 64, d_idx]: see kl_dk_slot
};

// Slot of the dK_idx partial that epilogue group `grp` of CTA `cta` writes for bucket `bkt`.
// The CTAs take contiguous ranges of the bucket-ordered work tiles, so a bucket's CTAs are
// consecutive and bkt + cta is unique over the (CTA, bucket) pairs that occur.
__host__ __device__ __forceinline__ int64_t kl_dk_slot(int bkt, int cta, int grp) {
  return ((int64_t)bkt + cta) * 2 + grp;
}
constexpr int kKlMaxGrid = 1024;          // CTAs of the block-major pass at most (workspace bound)

template <int D_H, int G, bool BWD, bool TCG = false>
__global__ void __launch_bounds__(KlWarps<BWD>::kThreads, 1)
    k_kl_kvouter(const __grid_constant__ KlQMaps tm_q, const __nv_bfloat16* __restrict__ q,
                 const __nv_bfloat16* __restrict__ k, const __nv_bfloat16* __restrict__ q_idx,
                 const __nv_bfloat16* __restrict__ k_idx, const float* __restrict__ lse,
                 const int* __restrict__ entries, const int* __restrict__ offset,
                 const int* __restrict__ tile_off, int nbuckets, int64_t nblk, int64_t N,
                 int H_kv, int d_idx, int kk, float4* __restrict__ part, float scale_log2,
                 float idx_scale, const KlGrad gr) {
  constexpr int kKlQWarps = KlWarps<BWD>::kQ;
  using L = KlSmem<D_H, G, BWD, TCG>;
  constexpr int kEpt = L::kEpt;
  constexpr int kQStages = L::kQStages, kKStages = L::kKStages, kTStages = L::kTStages;
  constexpr int kCpl = 64 / G;               // columns a lane owns after the reduce-scatter
  constexpr int kChunks = D_H / 8;           // 16-byte chunks per K / Q row
  constexpr int kEntPerLane = kEpt > 32 ? kEpt / 32 : 1;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t sb = smem_u32(smem);
  const uint32_t bar0 = sb + L::kOffBar;
  auto q_full = [&](int s) { return bar0 + 8u * s; };
  auto q_empty = [&](int s) { return bar0 + 8u * (kQStages + s); };
  auto k_full = [&](int s) { return bar0 + 8u * (2 * kQStages + s); };
  auto k_empty = [&](int s) { return bar0 + 8u * (2 * kQStages + kKStages + s); };
  auto t_full = [&](int s) { return bar0 + 8u * (2 * kQStages + 2 * kKStages + s); };
  auto t_empty = [&](int s) { return bar0 + 8u * (2 * kQStages + 2 * kKStages + kTStages + s); };
  auto g_done = [&](int g) { return bar0 + 8u * (2 * kQStages + 2 * kKStages + 2 * kTStages + g); };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kOffMisc);
  volatile int* s_abort = reinterpret_cast<volatile int*>(smem + L::kOffMisc + 4);
  int* s_pent = reinterpret_cast<int*>(smem + L::kOffPEnt);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int H_q = H_kv * G;
  const int ichunks = d_idx / 8;             // 16-byte chunks per index row

  if (threadIdx.x == 0) {
    for (int s = 0; s < kQStages; ++s) {
      // warp 0's arrive (with the TMA transaction bytes at G = 8), warp 10's 32 lanes' copies,
      // and at G = 8 one arrive of each other query-row warp (so that none of them can fall a
      // full phase behind when a tile gives it no box), else warp 0's 32 lanes' copies
      mbar_init(q_full(s), G == 8 ? 33 + (kKlQWarps - 1) : 65);
      mbar_init(q_empty(s), 1);              // MMA commit
    }
    for (int s = 0; s < kKStages; ++s) {
      mbar_init(k_full(s), 32);
      mbar_init(k_empty(s), 1);
    }
    for (int s = 0; s < kTStages; ++s) {
      mbar_init(t_full(s), 1);
      mbar_init(t_empty(s), 4 * 32);         // the 128 threads of one epilogue group
    }
    if (TCG) {
      mbar_init(g_done(0), 1);
      mbar_init(g_done(1), 1);
    }
    *s_abort = 0;
    fence_barrier_init();
  }
  if (TCG) {
    // index queries, dS and K_idx copies start as zeros: rows a tile leaves unwritten are
    // multiplied by zero dS, and must not hold NaN bit patterns
    for (int x = threadIdx.x; x < (L::kOffBar - L::kOffQg) / 16; x += blockDim.x)
      kl_zero16(sb + L::kOffQg + 16 * x);
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tc_fence_before();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  // a contiguous range of work tiles per CTA (consecutive tiles often share a bucket)
  const int total_tiles = tile_off[nbuckets];
  const int per = (total_tiles + gridDim.x - 1) / gridDim.x;
  const int t_beg = blockIdx.x * per;
  const int t_end = min(total_tiles, t_beg + per);
  const int ntiles = max(0, t_end - t_beg);
  int bucket0 = 0;
  if (ntiles > 0) {
    int lo = 0, hi = nbuckets;                             // tile_off[lo] <= t_beg < tile_off[hi]
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (__ldg(tile_off + mid) <= t_beg) lo = mid; else hi = mid;
    }
    bucket0 = lo;
  }
  const int next0 = ntiles > 0 ? __ldg(tile_off + bucket0 + 1) : 0;
  // tile -> (bucket, first entry, entries), advancing a cursor (bkt, nxt) over increasing tiles
  auto describe = [&](int tile, int& bkt, int& nxt, int& e0, int& n_e) {
    while (nxt <= tile) {
      ++bkt;
      nxt = __ldg(tile_off + bkt + 1);
    }
    e0 = __ldg(offset + bkt) + (tile - __ldg(tile_off + bkt)) * kEpt;
    n_e = min(kEpt, __ldg(offset + bkt + 1) - e0);
  };
  auto fail = [&]() { *s_abort = 1; };

  if (warp == 0 || warp == 10 || (warp >= 11 && G == 8)) {
    // ------------------------------------------------------------ producers
    const bool pq = warp != 10;                            // query rows; else keys, index queries
    const int qw = warp == 0 ? 0 : warp - 10;              // index among the query-row warps
    // each producer warp keeps its own copy of the tile's entries (in registers, or in shared
    // memory for the index-query warp)
    int* s_pw = s_pent + (pq ? 0 : kKlRows);
    int bkt = bucket0, nxt = next0;
    int last_bkt = -1, kfill = 0, issued = 0;
    // entries of the next tile, loaded one iteration ahead into registers
    int pb = bkt, pn = nxt, p_e0 = 0, p_ne = 0;
    int pre[kEntPerLane];
    auto load_ents = [&](int j) {
      describe(t_beg + j, pb, pn, p_e0, p_ne);
#pragma unroll
      for (int m = 0; m < kEntPerLane; ++m) {
        const int x = lane + 32 * m;
        pre[m] = x < p_ne ? __ldg(entries + p_e0 + x) : 0;
      }
    };
    if (ntiles > 0) load_ents(0);
    for (int j = 0; j < ntiles; ++j) {
      if (__any_sync(0xffffffffu, *s_abort != 0)) break;  // warp-uniform exits only
      int e0, n_e;
      describe(t_beg + j, bkt, nxt, e0, n_e);
      const int rb = (int)(bkt / nblk);
      const int64_t bb = bkt - (int64_t)rb * nblk;
      if (!pq && bkt != last_bkt) {                        // K_b and K_idx_b of a new bucket
        const int ks = kfill % kKStages;
        if (!__all_sync(0xffffffffu,
                        mbar_wait(k_empty(ks), ((kfill / kKStages) & 1) ^ 1, &g_kl_status))) {
          fail();
          break;
        }
        const uint32_t kbase = sb + L::kOffK + ks * L::kKStage;
        const __nv_bfloat16* kb = k + (bb * kBlock * H_kv + rb) * (int64_t)D_H;
        for (int x = lane; x < kBlock * kChunks; x += 32) {
          const int jj = x / kChunks, c = x - jj * kChunks;
          const uint32_t off = (c >> 3) * L::kKHalf + jj * 128 + (((c & 7) ^ (jj & 7)) << 4);
          if (bb * kBlock + jj < N)
            kl_cp_async16(kbase + off, kb + jj * (int64_t)H_kv * D_H + c * 8);
          else
            kl_zero16(kbase + off);
        }
        const __nv_bfloat16* kib = k_idx + bb * kBlock * (int64_t)d_idx;
        for (int x = lane; x < kBlock * ichunks; x += 32) {
          const int jj = x / ichunks, c = x - jj * ichunks;
          const uint32_t off = L::kHalves * L::kKHalf + jj * 128 + ((c ^ (jj & 7)) << 4);
          if (bb * kBlock + jj < N)
            kl_cp_async16(kbase + off, kib + (int64_t)jj * d_idx + c * 8);
          else
            kl_zero16(kbase + off);
        }
        asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        mbar_arrive(k_full(ks));
        last_bkt = bkt;
        ++kfill;
      }
      const int s = j % kQStages;
      if (!__all_sync(0xffffffffu,
                      mbar_wait(q_empty(s), ((j / kQStages) & 1) ^ 1, &g_kl_status))) {
        fail();
        break;
      }
      const uint32_t qbase = sb + L::kOffQ + s * L::kQStage;
      const int my_ent = pre[0];                           // entry `lane` (G = 8: <= 16 entries)
      if (!(pq && G == 8)) {                               // cp.async paths read them from smem
        __syncwarp();                                      // the previous tile's reads are done
#pragma unroll
        for (int m = 0; m < kEntPerLane; ++m)
          if (lane + 32 * m < kEpt) s_pw[lane + 32 * m] = pre[m];
        __syncwarp();
      }
      if (j + 1 < ntiles) load_ents(j + 1);                // lands while this tile is issued
      if (pq && G == 8) {
        // runs of consecutive query rows: the lane at the start of a run issues its boxes
        if (warp == 0 && lane == 0)
          mbar_expect_tx(q_full(s), (uint32_t)(n_e * 8 * 128 * L::kHalves));
        __syncwarp();
        const int row = lane < n_e ? (my_ent >> 6) : -2;
        const int prev = __shfl_up_sync(0xffffffffu, row, 1);
        const bool start = lane < n_e && (lane == 0 || prev != row - 1);
        const unsigned starts = __ballot_sync(0xffffffffu, start);
        if (start) {
          const unsigned later = starts & ~((2u << lane) - 1u);
          const int stop = later ? __ffs(later) - 1 : n_e;
          int off = 0;
          while (off < stop - lane) {
            const int rem = stop - lane - off;
            const int m = rem >= 16 ? 4 : rem >= 8 ? 3 : rem >= 4 ? 2 : rem >= 2 ? 1 : 0;
            // the boxes are dealt round-robin over the query-row warps by (first entry, half);
            // every such warp computes the same decomposition
#pragma unroll
            for (int bx = 0; bx < L::kHalves; ++bx)
              if (((lane + off) * L::kHalves + bx) % kKlQWarps == qw)
                tma_load_3d(qbase + bx * L::kQHalf + (lane + off) * 1024, &tm_q.m[m], q_full(s),
                            64 * bx, rb * 8, row + off);
            off += 1 << m;
          }
        }
        __syncwarp();
        if (warp != 0 && lane == 0) mbar_arrive(q_full(s));   // after this warp's boxes
      } else if (pq) {
        if (lane == 0) mbar_arrive(q_full(s));             // no transaction bytes
        for (int x = lane; x < n_e * G * kChunks; x += 32) {
          const int R = x / kChunks, c = x - R * kChunks;
          const int e = R / G, h = R - e * G;
          const int64_t i = s_pw[e] >> 6;
          const uint32_t off = (c >> 3) * L::kQHalf + R * 128 + (((c & 7) ^ (R & 7)) << 4);
          kl_cp_async16(qbase + off, q + (i * H_q + (int64_t)rb * G + h) * D_H + c * 8);
        }
      } else {
        for (int x = lane; x < n_e * ichunks; x += 32) {   // index queries, one row per entry
          const int e = x / ichunks, c = x - e * ichunks;
          const int64_t i = s_pw[e] >> 6;
          const uint32_t off = L::kHalves * L::kQHalf + e * 128 + ((c ^ (e & 7)) << 4);
          kl_cp_async16(qbase + off, q_idx + (i * H_kv + rb) * d_idx + c * 8);
        }
      }
      // each lane's copies arrive on the stage's barrier when they land (the MMA issuer then
      // makes them visible to the tensor core with a proxy fence)
      if (!pq || G != 8)
        asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(q_full(s))
                     : "memory");
      ++issued;
    }
    asm volatile("cp.async.wait_all;" ::: "memory");
    // every tile issued has its arrivals; wait until the copies of the last stages have landed
    for (int j = max(0, issued - kQStages); j < issued; ++j)
      mbar_wait(q_full(j % kQStages), (j / kQStages) & 1, &g_kl_status);
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer (one lane)
    if (lane == 0) {
      int bkt = bucket0, nxt = next0;
      int last_bkt = -1, kfill = -1, issued = 0;
      constexpr uint32_t idesc_s = umma_idesc_bf16(kKlRows, 64);
      constexpr uint32_t idesc_i = umma_idesc_bf16(kKlRows, kEpt);
      for (int j = 0; j < ntiles; ++j) {
        if (*s_abort) break;
        int e0, n_e;
        describe(t_beg + j, bkt, nxt, e0, n_e);
        if (bkt != last_bkt) {
          if (kfill >= 0) umma_commit(k_empty(kfill % kKStages));   // its MMAs are all issued
          ++kfill;
          if (!mbar_wait(k_full(kfill % kKStages), (kfill / kKStages) & 1, &g_kl_status)) {
            fail();
            break;
          }
          last_bkt = bkt;
        }
        const int s = j % kQStages, t = j % kTStages;
        if (!mbar_wait(q_full(s), (j / kQStages) & 1, &g_kl_status)) { fail(); break; }
        if (!mbar_wait(t_empty(t), ((j / kTStages) & 1) ^ 1, &g_kl_status)) { fail(); break; }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");   // cp.async data -> MMA
        tc_fence_after();
        const uint32_t qbase = sb + L::kOffQ + s * L::kQStage;
        const uint32_t kbase = sb + L::kOffK + (kfill % kKStages) * L::kKStage;
        const uint32_t d = tmem + (uint32_t)(L::kTCols * t);
        // teacher scores: S = Q_stack K_b^T, 128 rows x 64 tokens
#pragma unroll
        for (int ks = 0; ks < D_H / 16; ++ks) {
          const uint32_t a = qbase + (ks >> 2) * L::kQHalf + (ks & 3) * 32;
          const uint32_t bk = kbase + (ks >> 2) * L::kKHalf + (ks & 3) * 32;
          umma_bf16(d, umma_desc_kmajor(a, 1024, 128), umma_desc_kmajor(bk, 1024, 128), idesc_s,
                    ks > 0 ? 1u : 0u);
        }
        // student scores, transposed: K_idx_b [tokens on M] . Qi^T [the tile's entries on N]
        for (int ks = 0; ks < d_idx / 16; ++ks) {
          const uint32_t a = kbase + L::kHalves * L::kKHalf + ks * 32;
          const uint32_t bq = qbase + L::kHalves * L::kQHalf + ks * 32;
          umma_bf16(d + 64, umma_desc_kmajor(a, 1024, 128), umma_desc_kmajor(bq, 1024, 128),
                    idesc_i, ks > 0 ? 1u : 0u);
        }
        umma_commit(t_full(t));
        umma_commit(q_empty(s));
        issued = j + 1;
      }
      // the MMAs in flight complete before TMEM is released
      if (issued > 0)
        mbar_wait(t_full((issued - 1) % kTStages), ((issued - 1) / kTStages) & 1, &g_kl_status);
    }
  } else if (warp >= 2 && warp <= 9) {
    // ------------------------------------------------------------ epilogue groups
    const int grp = (warp - 2) >> 2;
    const int qd = warp & 3;                               // TMEM lane quarter of this warp
    const int R = 32 * qd + lane;                          // row (TMEM lane) of this thread
    const int e = R / G, h = R - e * G;
    float* s_si = reinterpret_cast<float*>(smem + L::kOffSi + grp * L::kSiBytes);
    const uint32_t s_qg = sb + L::kOffQg + grp * L::kQgBytes;   // gradient pass only
    const uint32_t s_ds = sb + L::kOffDs + grp * 2 * L::kDsBytes;   // TCG: dS hi, then lo
    const uint32_t s_kg = sb + L::kOffKg + grp * L::kKgBytes;       // TCG: K_idx block
    int kg_bkt = -1, gcount = 0;                                     // TCG state
    bool dk_fresh = true;
    int bkt = bucket0, nxt = next0;
    // this row's entry and forward LSE, fetched one group-tile ahead
    int c_e0 = 0, c_ne = 0, c_bkt = 0;
    int ent = 0;
    float lse_raw = 0.f;
    if (grp < ntiles) {
      describe(t_beg + grp, bkt, nxt, c_e0, c_ne);
      c_bkt = bkt;
      const int r0 = (int)(bkt / nblk);
      if (R < c_ne * G) {
        ent = __ldg(entries + c_e0 + e);
        lse_raw = __ldg(lse + (int64_t)(r0 * G + h) * N + (ent >> 6));
      }
    }
    // gradient pass: key-gradient accumulators of this thread's (token, dims) of the current
    // bucket's block, written to the group's partial slot of the bucket when the group moves
    // to another bucket (no atomics: k_kl_dk_merge sums the slots in a fixed order)
    float dkacc[BWD ? 32 : 1];
#pragma unroll
    for (int d = 0; d < (BWD ? 32 : 1); ++d) dkacc[d] = 0.f;
    for (int j = grp; j < ntiles; j += 2) {
      const int r = (int)(c_bkt / nblk);
      const int64_t b = c_bkt - (int64_t)r * nblk;
      const bool rv = R < c_ne * G;
      const int cur_ent = ent;
      const float cur_lse = lse_raw;
      // the group's next tile: its entry now, its LSE (which needs the entry) after this tile
      int n_e0 = 0, n_ne = 0, n_bkt = c_bkt;
      const bool has_next = j + 2 < ntiles;
      if (has_next) {
        describe(t_beg + j + 2, bkt, nxt, n_e0, n_ne);
        n_bkt = bkt;
        ent = R < n_ne * G ? __ldg(entries + n_e0 + e) : 0;
      }
      const int t = j % kTStages;
      if constexpr (BWD) {
        // this tile's index queries -> s_qg[entry], 16 bytes per (entry, chunk) item, landing
        // under the MMA wait and the loss part (at G = 8 item R is a chunk of this thread's own
        // entry R / 8)
        for (int item = R; item < kEpt * 8; item += kKlRows) {
          const int eq = item >> 3, qc = item & 7;
          if (eq < c_ne && qc < (d_idx >> 3)) {
            const int eg = G == 8 ? cur_ent : __ldg(entries + c_e0 + eq);
            kl_cp_async16(s_qg + eq * 128 + ((TCG ? qc ^ (eq & 7) : qc) << 4),
                          q_idx + ((int64_t)(eg >> 6) * H_kv + r) * d_idx + qc * 8);
          }
        }
        if (TCG && c_bkt != kg_bkt) {
          // the bucket's K_idx block for the gradient MMAs (the previous tile's have completed)
          const __nv_bfloat16* kib = k_idx + b * kBlock * (int64_t)d_idx;
          for (int x = R; x < kBlock * 8; x += kKlRows) {
            const int jj = x >> 3, c = x & 7;
            const uint32_t dst = s_kg + jj * 128 + ((c ^ (jj & 7)) << 4);
            if (b * kBlock + jj < N)
              kl_cp_async16(dst, kib + (int64_t)jj * d_idx + c * 8);
            else
              kl_zero16(dst);
          }
          kg_bkt = c_bkt;
        }
        asm volatile("cp.async.commit_group;" ::: "memory");
      }
      const bool okw = *s_abort == 0 && mbar_wait(t_full(t), (j / kTStages) & 1, &g_kl_status);
      if (!kl_group_and(1 + grp, okw)) { fail(); break; }
      tc_fence_after();
      const uint32_t tbase = tmem + ((uint32_t)(32 * qd) << 16) + (uint32_t)(L::kTCols * t);
      // student scores of tokens 32*qd .. 32*qd+31 (lanes 0..63 only) -> s_si[entry][token]
      if (qd < 2) {
#pragma unroll
        for (int cc = 0; cc < kEpt; cc += 16) {
          uint32_t v[16];
          KL_TMEM_LD16(tbase + 64 + cc, v);
          tmem_ld_wait();
#pragma unroll
          for (int c = 0; c < 16; ++c) s_si[(cc + c) * kSiStride + R] = __uint_as_float(v[c]);
        }
      }
      int cmax = -1;                                       // last visible column, -1: none
      if (rv) {
        const int64_t i = cur_ent >> 6;
        cmax = b == (i >> 6) ? (int)(i - b * kBlock) : kBlock - 1;
      }
      const float lse2 = cur_lse * kLog2e;
      float a[64];
      {
        uint32_t sv[64];
        MSA_TMEM_LD64(tbase, sv);
        tmem_ld_wait();
#pragma unroll
        for (int c = 0; c < 64; c += 2) {
          float x0, x1;
          ffma2(x0, x1, __uint_as_float(sv[c]), __uint_as_float(sv[c + 1]), scale_log2,
                scale_log2, -lse2, -lse2);
          a[c] = c <= cmax ? ex2(x0) : 0.f;
          a[c + 1] = c + 1 <= cmax ? ex2(x1) : 0.f;
        }
      }
      tc_fence_before();
      mbar_arrive(t_empty(t));                             // this TMEM stage may be reused
      lane_split<G, true>(a, h);                           // a[c]: G * P of column kCpl*h + c
      kl_group_sync(1 + grp);                              // s_si is complete
      const int cb = kCpl * h;
      float si[kCpl];
#pragma unroll
      for (int c = 0; c < kCpl; c += 4) {
        const float4 v = *reinterpret_cast<const float4*>(s_si + e * kSiStride + cb + c);
        si[c] = v.x;
        si[c + 1] = v.y;
        si[c + 2] = v.z;
        si[c + 3] = v.w;
      }
      kl_group_sync(1 + grp);                              // s_si may be overwritten
      if (has_next && R < n_ne * G)                        // the next tile's LSE, under this one
        lse_raw = __ldg(lse + (int64_t)((int)(n_bkt / nblk) * G + h) * N + (ent >> 6));

      // this lane's columns: sum P (ln P - S^idx), sum P, student max / sum (log2 domain)
      const float invG = 1.f / (float)G, log2G = __log2f((float)G);
      float C = 0.f, W = 0.f, mx = -1e30f, l = 0.f;
#pragma unroll
      for (int c = 0; c < kCpl; ++c)
        if (cb + c <= cmax) mx = fmaxf(mx, si[c] * idx_scale * kLog2e);
#pragma unroll
      for (int c = 0; c < kCpl; ++c) {
        if (cb + c <= cmax) {
          const float x2 = si[c] * idx_scale * kLog2e;
          l += ex2(x2 - mx);
          const float P = a[c] * invG;
          if (P > 0.f) C += P * ((__log2f(a[c]) - log2G) * kLn2 - si[c] * idx_scale);
          W += P;
        }
      }
      // combine the entry's G lanes; its first lane writes the partial
#pragma unroll
      for (int m = 1; m < G; m <<= 1) {
        C += __shfl_xor_sync(0xffffffffu, C, m);
        W += __shfl_xor_sync(0xffffffffu, W, m);
        const float mo = __shfl_xor_sync(0xffffffffu, mx, m);
        const float lo = __shfl_xor_sync(0xffffffffu, l, m);
        const float nm = fmaxf(mx, mo);
        l = l * ex2(mx - nm) + lo * ex2(mo - nm);
        mx = nm;
      }
      if (!BWD && rv && h == 0)
        part[((int64_t)r * N + (cur_ent >> 6)) * kk + (cur_ent & 63)] = make_float4(C, W, mx, l);
      if constexpr (BWD) {
        // dS of this lane's columns: g (W P^idx - P) / sqrt(d_idx), with the row's upstream
        // gradient g, teacher mass W and student LSE from the loss pass; 0 where not visible
        float g = 0.f, wsum = 0.f, lsei2 = 0.f;
        if (rv) {
          const int64_t row = (int64_t)r * N + (cur_ent >> 6);
          g = __ldg(gr.grad_kl + row);
          wsum = __ldg(gr.psum + row);
          lsei2 = __ldg(gr.lse_idx + row) * kLog2e;
        }
        if constexpr (TCG) {
          // dS of this lane's columns, split into bf16 hi + lo, into row e of the group's dS
          // tiles (column c of row e: 16-byte chunk c / 8 at position (c / 8) ^ (e & 7))
#pragma unroll
          for (int c8 = 0; c8 < kCpl; c8 += 8) {
            uint32_t hw[4], lw[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              float dv[2];
#pragma unroll
              for (int q2 = 0; q2 < 2; ++q2) {
                const int c = c8 + 2 * u + q2;
                const float pidx = ex2(si[c] * idx_scale * kLog2e - lsei2);
                dv[q2] = cb + c <= cmax ? g * (wsum * pidx - a[c] * invG) * idx_scale : 0.f;
              }
              hw[u] = pack_bf16x2(dv[0], dv[1]);
              lw[u] = pack_bf16x2(dv[0] - __uint_as_float(hw[u] << 16),
                                  dv[1] - __uint_as_float(hw[u] & 0xffff0000u));
            }
            const int chunk = (cb + c8) >> 3;
            const uint32_t off = (uint32_t)((e >> 3) * 1024 + (e & 7) * 128 + ((chunk ^ (e & 7)) << 4));
            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(s_ds + off), "r"(hw[0]),
                         "r"(hw[1]), "r"(hw[2]), "r"(hw[3]) : "memory");
            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(s_ds + L::kDsBytes + off),
                         "r"(lw[0]), "r"(lw[1]), "r"(lw[2]), "r"(lw[3]) : "memory");
          }
          asm volatile("cp.async.wait_all;" ::: "memory");   // index queries, K_idx block
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
          tc_fence_before();
          kl_group_sync(1 + grp);                            // dS, Q_idx, K_idx are complete
          const uint32_t col_dq = L::kColGrad + 128u * grp, col_dk = col_dq + 64u;
          if (R == 0) {
            tc_fence_after();
            constexpr uint32_t idesc_dq = umma_idesc_bf16(128, kEpt) | (1u << 15);
            constexpr uint32_t idesc_dk = umma_idesc_bf16(128, 64) | (1u << 15) | (1u << 16);
            // dQ_idx^T [dims][entries] = K_idx_b^T [dims][tokens] . dS^T [tokens][entries]
            // (A: K_idx rows read MN-major; rows 64..127 of M are unused lanes)
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
#pragma unroll
              for (int part = 0; part < 2; ++part)
                umma_bf16(tmem + col_dq, desc_mn_sw128(s_kg + ks * 2048, 1024, 1024),
                          umma_desc_kmajor(s_ds + part * L::kDsBytes + ks * 32, 1024, 128),
                          idesc_dq, (ks | part) ? 1u : 0u);
            // dK_idx [tokens][dims] += dS^T [tokens][entries] . Q_idx [entries][dims], over the
            // group's tiles of this bucket
#pragma unroll
            for (int ks = 0; ks < kEpt / 16; ++ks)
#pragma unroll
              for (int part = 0; part < 2; ++part)
                umma_bf16(tmem + col_dk,
                          desc_mn_sw128(s_ds + part * L::kDsBytes + ks * 2048, 1024, 1024),
                          desc_mn_sw128(s_qg + ks * 2048, 8192, 1024), idesc_dk,
                          (!dk_fresh || ks || part) ? 1u : 0u);
            umma_commit(g_done(grp));
          }
          const bool okg = mbar_wait(g_done(grp), gcount & 1, &g_kl_status);
          ++gcount;
          if (!kl_group_and(1 + grp, okg)) { fail(); break; }
          tc_fence_after();
          const bool flush = !has_next || n_bkt != c_bkt;
          if (qd < 2) {
            // lanes 0..63: this thread's dims row R of dQ_idx^T over the tile's entries
            const uint32_t lanes = (uint32_t)(32 * qd) << 16;
#pragma unroll
            for (int cc = 0; cc < kEpt; cc += 16) {
              uint32_t v[16];
              KL_TMEM_LD16(tmem + lanes + col_dq + cc, v);
              tmem_ld_wait();
#pragma unroll
              for (int c = 0; c < 16; ++c)
                if (cc + c < c_ne) {
                  const int ent_q = __ldg(entries + c_e0 + cc + c);
                  gr.part_dq[(((int64_t)r * N + (ent_q >> 6)) * kk + (ent_q & 63)) * d_idx + R] =
                      __uint_as_float(v[c]);
                }
            }
            if (flush) {
              // token row R of the bucket's dK_idx, to the group's slot
              uint32_t v[64];
              MSA_TMEM_LD64(tmem + lanes + col_dk, v);
              tmem_ld_wait();
              float4* dst = reinterpret_cast<float4*>(
                  gr.part_dk + (kl_dk_slot(c_bkt, blockIdx.x, grp) * kBlock + R) * d_idx);
#pragma unroll
              for (int d = 0; d < 64; d += 4)
                dst[d / 4] = make_float4(__uint_as_float(v[d]), __uint_as_float(v[d + 1]),
                                         __uint_as_float(v[d + 2]), __uint_as_float(v[d + 3]));
            }
          }
          dk_fresh = flush;
          tc_fence_before();
          kl_group_sync(1 + grp);                          // TMEM and dS may be overwritten
        } else {
#pragma unroll
          for (int c = 0; c < kCpl; ++c) {
            const float pidx = ex2(si[c] * idx_scale * kLog2e - lsei2);
            const float ds = g * (wsum * pidx - a[c] * invG) * idx_scale;
            s_si[e * kSiStride + cb + c] = cb + c <= cmax ? ds : 0.f;
          }
          asm volatile("cp.async.wait_all;" ::: "memory");   // this thread's index-query copy
          kl_group_sync(1 + grp);                            // dS and the index queries are complete
          const int64_t tok0 = b * kBlock;
          // dQ_idx of (entry, dims chunk) items: entry item / 8, dims (item % 8) * d_idx / 8 ..,
          // summed over the block's tokens
          for (int item = R; item < kEpt * 8; item += kKlRows) {
            const int eq = item >> 3, nd = d_idx >> 3, d0 = (item & 7) * nd;
            if (eq < c_ne) {
              float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
              // tokens past the sequence have dS = 0; their loads read the last row instead
  #pragma unroll 8
              for (int c = 0; c < kBlock; ++c) {
                const float ds = s_si[eq * kSiStride + c];
                const int64_t tok = tok0 + c < N ? tok0 + c : N - 1;
                const __nv_bfloat16* kr = k_idx + tok * d_idx + d0;
                if (nd == 8) {
                  const uint4 v = ldg_nc_v4(kr);
                  const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
  #pragma unroll
                  for (int u = 0; u < 4; ++u)   // bf16 pair -> fp32 pair is exact (a shift), then one packed FMA
                    ffma2(acc[2 * u], acc[2 * u + 1], ds, ds, __uint_as_float(w4[u] << 16),
                          __uint_as_float(w4[u] & 0xffff0000u), acc[2 * u], acc[2 * u + 1]);
                } else {
                  const uint2 v = *reinterpret_cast<const uint2*>(kr);
                  const float2 f0 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&v.x));
                  const float2 f1 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&v.y));
                  acc[0] += ds * f0.x;
                  acc[1] += ds * f0.y;
                  acc[2] += ds * f1.x;
                  acc[3] += ds * f1.y;
                }
              }
              const int ent_q = __ldg(entries + c_e0 + eq);
              float* dst = gr.part_dq +
                           (((int64_t)r * N + (ent_q >> 6)) * kk + (ent_q & 63)) * d_idx + d0;
              // 16-byte stores: a thread's nd floats are contiguous and 16-byte aligned
              reinterpret_cast<float4*>(dst)[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
              if (nd == 8)
                reinterpret_cast<float4*>(dst)[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
            }
          }
          // dK_idx of token R / 2, dims (R % 2) * d_idx / 2 ..: sum over the tile's entries
          {
            const int ck = R >> 1, nd = d_idx >> 1, d0 = (R & 1) * nd;
  #pragma unroll 4
            for (int eq = 0; eq < c_ne; ++eq) {
              const float ds = s_si[eq * kSiStride + ck];
              const uint8_t* qr = smem + L::kOffQg + grp * L::kQgBytes + eq * 128 + d0 * 2;
  #pragma unroll
              for (int u = 0; u < 4; ++u) {
                if (8 * u >= nd) break;
                const uint4 v = *reinterpret_cast<const uint4*>(qr + 16 * u);
                const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
  #pragma unroll
                for (int t = 0; t < 4; ++t)
                  ffma2(dkacc[8 * u + 2 * t], dkacc[8 * u + 2 * t + 1], ds, ds,
                        __uint_as_float(w4[t] << 16), __uint_as_float(w4[t] & 0xffff0000u),
                        dkacc[8 * u + 2 * t], dkacc[8 * u + 2 * t + 1]);
              }
            }
            kl_group_sync(1 + grp);                          // s_si may be overwritten
            const bool flush = !has_next || n_bkt != c_bkt;
            if (flush) {
              float4* dst = reinterpret_cast<float4*>(
                  gr.part_dk + (kl_dk_slot(c_bkt, blockIdx.x, grp) * kBlock + ck) * d_idx + d0);
  #pragma unroll
              for (int d = 0; d < 32; d += 4)
                if (d < nd) dst[d / 4] = make_float4(dkacc[d], dkacc[d + 1], dkacc[d + 2], dkacc[d + 3]);
  #pragma unroll
              for (int d = 0; d < 32; ++d) dkacc[d] = 0.f;
            }
          }
        }
        }
      c_bkt = n_bkt;
      c_e0 = n_e0;
      c_ne = n_ne;
    }
  }
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ---------------------------------------------------------------------- merge --
// One thread per (group, row): KL = sum_e C_e + (sum_e W_e) * LSE^idx, with LSE^idx merged from
// the entries' (max, sum) pairs in slot order.
__global__ void __launch_bounds__(256)
    k_kl_merge(const int32_t* __restrict__ idx, const float4* __restrict__ part, float* kl,
               float* lse_idx, float* psum, int64_t N, int H_kv, int kk) {
  const int64_t x = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (x >= (int64_t)H_kv * N) return;
  const int64_t i = x % N;
  const int32_t* sel = idx + x * kk;
  const float4* pp = part + x * kk;
  float C = 0.f, W = 0.f, mx = -1e30f, l = 0.f;
  for (int t = 0; t < kk; ++t) {
    const int b = __ldg(sel + t);
    if (b < 0 || (int64_t)b > (i >> 6)) continue;
    const float4 v = pp[t];
    C += v.x;
    W += v.y;
    const float nm = fmaxf(mx, v.z);
    l = l * ex2(mx - nm) + v.w * ex2(v.z - nm);
    mx = nm;
  }
  const float lsei = (mx + __log2f(l)) * kLn2;
  kl[x] = C + W * lsei;
  if (lse_idx) lse_idx[x] = lsei;                 // by-products for the gradient pass
  if (psum) psum[x] = W;
}

// dQ_idx[i, r, :] = sum over the row's selections (slot order) of their partials.
__global__ void __launch_bounds__(256)
    k_kl_dq_merge(const int32_t* __restrict__ idx, const float* __restrict__ part_dq,
                  float* __restrict__ dq_idx, int64_t N, int H_kv, int kk, int d_idx) {
  const int64_t x = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;   // ((r * N + i) * d_idx + d)
  if (x >= (int64_t)H_kv * N * d_idx) return;
  const int64_t ri = x / d_idx;
  const int d = (int)(x - ri * d_idx);
  const int64_t r = ri / N, i = ri - r * N;
  const int32_t* sel = idx + ri * kk;
  float acc = 0.f;
  for (int t = 0; t < kk; ++t) {
    const int b = __ldg(sel + t);
    if (b < 0 || (int64_t)b > (i >> 6)) continue;
    acc += __ldg(part_dq + (ri * kk + t) * d_idx + d);
  }
  dq_idx[(i * H_kv + r) * d_idx + d] = acc;
}

// dK_idx[j, d] = sum over the groups r, then the CTAs that processed bucket (r, floor(j/64)) in
// CTA order, then their two epilogue groups, of the slots' partials: a fixed order, so the
// result does not depend on the hardware's schedule.  `grid` and the tile ranges are those of
// the block-major pass.
__global__ void __launch_bounds__(256)
    k_kl_dk_merge(const int* __restrict__ tile_off, const float* __restrict__ part_dk,
                  float* dk_idx, int64_t N, int64_t nblk, int H_kv, int d_idx, int grid) {
  const int64_t x = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (x >= N * d_idx) return;
  const int64_t j = x / d_idx;
  const int d = (int)(x - j * d_idx);
  const int64_t b = j >> 6;
  const int c = (int)(j & 63);
  const int total = __ldg(tile_off + H_kv * nblk);
  const int per = (total + grid - 1) / grid;
  float acc = 0.f;
  for (int r = 0; r < H_kv; ++r) {
    const int bkt = (int)(r * nblk + b);
    const int t0 = __ldg(tile_off + bkt), t1 = __ldg(tile_off + bkt + 1);
    if (t0 == t1) continue;
    for (int cta = t0 / per; cta <= (t1 - 1) / per; ++cta) {
      const int tb = cta * per;
      const int lo = max(t0, tb) - tb, hi = min(t1, tb + per) - tb;   // local tiles [lo, hi)
#pragma unroll
      for (int g = 0; g < 2; ++g)
        if (hi - lo >= 2 || (lo & 1) == g)
          acc += __ldg(part_dk + (kl_dk_slot(bkt, cta, g) * kBlock + c) * d_idx + d);
    }
  }
  dk_idx[x] = acc;
}

}  // namespace

// Every selection of idx bucketed by (group, block): count -> scan -> scatter, with each bucket's
// selections in (16-query tile, query) order and ept entries per work tile.
cudaError_t launch_bucket_selections(const int32_t* idx, int64_t N, int H_kv, int kk, int ept,
                                     int* count, int* offset, int* tile_off, int* cursor,
                                     int* entries, cudaStream_t st) {
  const int64_t nblk = (N + kBlock - 1) / kBlock;
  const int nb = (int)(H_kv * nblk);
  cudaError_t e = cudaMemsetAsync(count, 0, sizeof(int) * (size_t)nb, st);
  if (e != cudaSuccess) return e;
  const int64_t tiles = (N + kTileQ - 1) / kTileQ;
  const dim3 pgrid((unsigned)((tiles + kKlPlanWarps - 1) / kKlPlanWarps), (unsigned)H_kv);
  if ((e = launch_epl<KlPlanK>(kk, pgrid, dim3(32 * kKlPlanWarps), st, idx, N, kk, nblk, 0, count,
                               (const int*)offset, cursor, entries)) != cudaSuccess)
    return e;
  if ((e = launch_attn_scan(count, offset, tile_off, nb, ept, st)) != cudaSuccess) return e;
  if ((e = cudaMemsetAsync(cursor, 0, sizeof(int) * (size_t)nb, st)) != cudaSuccess) return e;
  return launch_epl<KlPlanK>(kk, pgrid, dim3(32 * kKlPlanWarps), st, idx, N, kk, nblk, 1, count,
                             (const int*)offset, cursor, entries);
}

int ordered_bucket_ranges(int64_t N) {
  return (int)(((N + kTileQ - 1) / kTileQ + kRangeTiles - 1) / kRangeTiles);
}

cudaError_t launch_bucket_selections_ordered(const int32_t* idx, int64_t N, int H_kv, int kk,
                                             int ept, int* count, int* offset, int* tile_off,
                                             int* cursor, int* cnt_mat, int* entries,
                                             cudaStream_t st) {
  const int64_t nblk = (N + kBlock - 1) / kBlock;
  const int nb = (int)(H_kv * nblk);
  const int R = ordered_bucket_ranges(N);
  cudaError_t e = cudaMemsetAsync(count, 0, sizeof(int) * (size_t)nb, st);
  if (e != cudaSuccess) return e;
  if ((e = cudaMemsetAsync(cnt_mat, 0, sizeof(int) * (size_t)nb * R, st)) != cudaSuccess) return e;
  const int64_t tiles = (N + kTileQ - 1) / kTileQ;
  const dim3 cgrid((unsigned)((tiles + kKlPlanWarps - 1) / kKlPlanWarps), (unsigned)H_kv);
  if ((e = launch_epl<OrderCountK>(kk, cgrid, dim3(32 * kKlPlanWarps), st, idx, N, kk, nblk, R,
                                   count, cnt_mat)) != cudaSuccess)
    return e;
  if ((e = launch_attn_scan(count, offset, tile_off, nb, ept, st)) != cudaSuccess) return e;
  k_order_bases<<<(nb + 255) / 256, 256, 0, st>>>(offset, cnt_mat, nb, R);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  const dim3 sgrid((unsigned)((R + kKlPlanWarps - 1) / kKlPlanWarps), (unsigned)H_kv);
  return launch_epl<OrderScatterK>(kk, sgrid, dim3(32 * kKlPlanWarps), st, idx, N, kk, nblk, R,
                                   cnt_mat, entries);
}

size_t kl_ws_bytes(int64_t N, int H_kv, int kk) {
  const int64_t nb = (int64_t)H_kv * ((N + kBlock - 1) / kBlock);
  auto a256 = [](size_t x) { return (x + 255) & ~size_t(255); };
  const size_t sel = (size_t)H_kv * N * kk;
  return 4 * a256(4 * (size_t)(nb + 1)) + a256(4 * sel) + a256(16 * sel);
}

size_t kl_bwd_ws_bytes(int64_t N, int H_kv, int d_idx, int kk) {
  auto a256 = [](size_t x) { return (x + 255) & ~size_t(255); };
  const int64_t nb = (int64_t)H_kv * ((N + kBlock - 1) / kBlock);
  return kl_ws_bytes(N, H_kv, kk) + a256(4 * (size_t)H_kv * N * kk * d_idx) +
         a256(4 * (size_t)kl_dk_slot((int)nb, kKlMaxGrid, 0) * kBlock * d_idx) +
         a256(4 * (size_t)nb * ordered_bucket_ranges(N));
}

namespace {

// Plan (bucket every selection by (group, block)), then the block-major pass, forward or gradient.
cudaError_t kl_pass(bool bwd, const void* q, const void* k, const void* q_idx, const void* k_idx,
                    const int32_t* idx, const float* lse, int64_t N, int H_q, int H_kv, int d_h,
                    int d_idx, int kk, void* ws, const KlGrad& gr, int* cnt_mat,
                    float4** part_out, int* grid_out, cudaStream_t st) {
  const int G = H_q / H_kv;
  const int64_t nblk = (N + kBlock - 1) / kBlock;
  const int nb = (int)(H_kv * nblk);
  const size_t sel = (size_t)H_kv * N * kk;
  auto a256 = [](size_t x) { return (x + 255) & ~size_t(255); };
  char* base = static_cast<char*>(ws);
  int* count = reinterpret_cast<int*>(base);
  int* offset = reinterpret_cast<int*>(base + a256(4 * (size_t)(nb + 1)));
  int* tile_off = reinterpret_cast<int*>(base + 2 * a256(4 * (size_t)(nb + 1)));
  int* cursor = reinterpret_cast<int*>(base + 3 * a256(4 * (size_t)(nb + 1)));
  int* entries = reinterpret_cast<int*>(base + 4 * a256(4 * (size_t)(nb + 1)));
  float4* part = reinterpret_cast<float4*>(base + 4 * a256(4 * (size_t)(nb + 1)) + a256(4 * sel));
  *part_out = part;

  // the gradient pass sums dK_idx over a bucket's work tiles: it takes the buckets in row order,
  // so that the tiles, and with them the sums, are the same on every call
  cudaError_t e =
      bwd ? launch_bucket_selections_ordered(idx, N, H_kv, kk, kKlRows / G, count, offset,
                                             tile_off, cursor, cnt_mat, entries, st)
          : launch_bucket_selections(idx, N, H_kv, kk, kKlRows / G, count, offset, tile_off,
                                     cursor, entries, st);
  if (e != cudaSuccess) return e;

  KlQMaps tq;
  for (int m = 0; m < 5; ++m) {
    e = make_tma_3d_bf16(&tq.m[m], q, (uint64_t)d_h, (uint64_t)H_q, (uint64_t)N, 64, G, 1 << m,
                         128);
    if (e != cudaSuccess) return e;
  }
  int dev = 0, sms = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
    return e;
  const float scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)d_h));
  const float idx_scale = (float)(1.0 / std::sqrt((double)d_idx));
  const auto* qq = static_cast<const __nv_bfloat16*>(q);
  const auto* kp = static_cast<const __nv_bfloat16*>(k);
  const auto* qi = static_cast<const __nv_bfloat16*>(q_idx);
  const auto* ki = static_cast<const __nv_bfloat16*>(k_idx);
  const int grid = sms < kKlMaxGrid ? sms : kKlMaxGrid;    // persistent: one CTA per SM
  if (grid_out) *grid_out = grid;
  auto run = [&](auto kern, int smem, int threads) -> cudaError_t {
    cudaError_t x = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (x != cudaSuccess) return x;
    kern<<<grid, threads, smem, st>>>(tq, qq, kp, qi, ki, lse, entries, offset, tile_off, nb,
                                      nblk, N, H_kv, d_idx, kk, part, scale_log2, idx_scale, gr);
    return cudaGetLastError();
  };
  auto dispatch = [&](auto dh) -> cudaError_t {
    constexpr int D = decltype(dh)::value;
    if (bwd) {
      constexpr int TB = KlWarps<true>::kThreads;
      // the gradient products on the tensor core where the layout allows (d_idx = 64, G = 4 or 8,
      // or G = 2 at d_h = 64: at d_h = 128 its buffers do not fit), on the CUDA cores otherwise
      if (d_idx == 64) {
        if (G == 8) return run(k_kl_kvouter<D, 8, true, true>, KlSmem<D, 8, true, true>::kAlloc, TB);
        if (G == 4) return run(k_kl_kvouter<D, 4, true, true>, KlSmem<D, 4, true, true>::kAlloc, TB);
        if constexpr (D == 64)
          if (G == 2) return run(k_kl_kvouter<D, 2, true, true>, KlSmem<D, 2, true, true>::kAlloc, TB);
      }
      switch (G) {
        case 1: return run(k_kl_kvouter<D, 1, true>, KlSmem<D, 1, true>::kAlloc, TB);
        case 2: return run(k_kl_kvouter<D, 2, true>, KlSmem<D, 2, true>::kAlloc, TB);
        case 4: return run(k_kl_kvouter<D, 4, true>, KlSmem<D, 4, true>::kAlloc, TB);
        default: return run(k_kl_kvouter<D, 8, true>, KlSmem<D, 8, true>::kAlloc, TB);
      }
    }
    constexpr int T = KlWarps<false>::kThreads;
    switch (G) {
      case 1: return run(k_kl_kvouter<D, 1, false>, KlSmem<D, 1>::kAlloc, T);
      case 2: return run(k_kl_kvouter<D, 2, false>, KlSmem<D, 2>::kAlloc, T);
      case 4: return run(k_kl_kvouter<D, 4, false>, KlSmem<D, 4>::kAlloc, T);
      default: return run(k_kl_kvouter<D, 8, false>, KlSmem<D, 8>::kAlloc, T);
    }
  };
  return d_h == 128 ? dispatch(std::integral_constant<int, 128>())
                    : dispatch(std::integral_constant<int, 64>());
}

}  // namespace

cudaError_t launch_kl_loss_fwd(const void* q, const void* k, const void* q_idx, const void* k_idx,
                               const int32_t* idx, const float* lse, float* kl, float* lse_idx,
                               float* psum, int64_t N, int H_q, int H_kv, int d_h, int d_idx,
                               int kk, void* ws, cudaStream_t st) {
  float4* part = nullptr;
  cudaError_t e = kl_pass(false, q, k, q_idx, k_idx, idx, lse, N, H_q, H_kv, d_h, d_idx, kk, ws,
                          KlGrad{}, nullptr, &part, nullptr, st);
  if (e != cudaSuccess) return e;
  const int64_t n = (int64_t)H_kv * N;
  k_kl_merge<<<(unsigned)((n + 255) / 256), 256, 0, st>>>(idx, part, kl, lse_idx, psum, N, H_kv,
                                                          kk);
  return cudaGetLastError();
}

cudaError_t launch_kl_loss_bwd(const void* q, const void* k, const void* q_idx, const void* k_idx,
                               const int32_t* idx, const float* lse, const float* lse_idx,
                               const float* psum, const float* grad_kl, float* dq_idx,
                               float* dk_idx, int64_t N, int H_q, int H_kv, int d_h, int d_idx,
                               int kk, void* ws, cudaStream_t st) {
  auto a256 = [](size_t x) { return (x + 255) & ~size_t(255); };
  char* base = static_cast<char*>(ws) + kl_ws_bytes(N, H_kv, kk);
  float* part_dq = reinterpret_cast<float*>(base);
  const size_t dq_bytes = a256(4 * (size_t)H_kv * N * kk * d_idx);
  float* part_dk = reinterpret_cast<float*>(base + dq_bytes);
  const int64_t nb = (int64_t)H_kv * ((N + kBlock - 1) / kBlock);
  int* cnt_mat = reinterpret_cast<int*>(
      base + dq_bytes + a256(4 * (size_t)kl_dk_slot((int)nb, kKlMaxGrid, 0) * kBlock * d_idx));
  const KlGrad gr{grad_kl, lse_idx, psum, part_dq, part_dk};
  float4* part = nullptr;
  int grid = 0;
  cudaError_t e = kl_pass(true, q, k, q_idx, k_idx, idx, lse, N, H_q, H_kv, d_h, d_idx, kk, ws, gr,
                          cnt_mat, &part, &grid, st);
  if (e != cudaSuccess) return e;
  const int64_t n = (int64_t)H_kv * N * d_idx;
  k_kl_dq_merge<<<(unsigned)((n + 255) / 256), 256, 0, st>>>(idx, part_dq, dq_idx, N, H_kv, kk,
                                                             d_idx);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  const int64_t nblk = (N + kBlock - 1) / kBlock;
  const int* tile_off = reinterpret_cast<const int*>(static_cast<char*>(ws) +
                                                     2 * a256(4 * (size_t)(H_kv * nblk + 1)));
  const int64_t nk = N * d_idx;
  k_kl_dk_merge<<<(unsigned)((nk + 255) / 256), 256, 0, st>>>(tile_off, part_dk, dk_idx, N, nblk,
                                                              H_kv, d_idx, grid);
  return cudaGetLastError();
}

cudaError_t read_reset_kl_status(unsigned* out) {
  unsigned zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(out, g_kl_status, sizeof(unsigned));
  if (e != cudaSuccess) return e;
  return cudaMemcpyToSymbol(g_kl_status, &zero, sizeof(unsigned));
}

}  // namespace msa

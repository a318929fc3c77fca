// Index branch of MSA on sm_103a: causal token scores Q_idx . K_idx^T / sqrt(d_idx) with the
// per-block max-pool fused into the epilogue («MiniMax-M3：MSA 技术报告速读», section 索引分支,
// eqs. S^idx and M^idx).
//
// One dense GEMM  [N*H_kv x d_idx] . [d_idx x N]  restricted to the causal triangle:
//   * rows are (query i, group r) pairs, i.e. Q_idx viewed as [N*H_kv, d_idx]; 128 consecutive
//     rows (128/H_kv queries x H_kv groups) form one UMMA M=128 sub-tile, and SUB sub-tiles
//     share every K_idx tile, so the shared index key is read once for all groups.  Every
//     variant dispatched runs one sub-tile per CTA and two CTAs per SM, so one CTA's MMAs run
//     while the other's epilogue drains its accumulators.
//   * K_idx tiles of 128 keys (two 64-token blocks) stream through a TMA ring (3 to 6 stages).
//   * one thread issues tcgen05.mma (bf16 x bf16 -> fp32) into a double-buffered TMEM
//     accumulator; the next tile's MMA overlaps the epilogue of the previous one.
//   * epilogue warps read 64 columns (= one block) per row with tcgen05.ld.red, which also
//     returns the row's maximum over them (the diagonal block masks j > i and reduces in
//     registers), scale once, and stage 32 blocks per row in shared memory before one
//     coalesced 128-byte store per row.
//   * blocks after a row's own block are written as -inf.
// Warp roles: warp 0 = TMA producer, warp 1 = TMEM allocator + MMA issuer,
// warps 2.. = 4*SUB epilogue warps (warp w reads TMEM lanes 32*(w%4) .. +31); with the select
// epilogue at k <= 16, 4*SUB more warps, one selection warp per epilogue warp (below).
//
// The SELECT variant fuses the per-group top-k of the same section (eq. I^(r)_i) into the
// epilogue and never writes M: the thread that owns a (query, group) row sees the row's block
// maxima in ascending block order, and keeps every block b < l(i) whose score is strictly
// above tau, the (k-1)-th best score among the blocks kept so far, in a per-row buffer in
// shared memory.  When a buffer is about to overflow, the warp compacts (all lanes at once) to
// each row's best k-1 under (score desc, block asc) and raises tau.  A block with a score equal
// to tau ranks below the k-1 earlier (lower-indexed) blocks that hold tau or more, so the
// strict test loses nothing.  Compaction is stable, so the buffer stays in ascending block
// order; at the end each row writes its kept blocks, then l(i), then -1 padding: exactly what
// msa_select_blocks writes from the same fp32 block scores.  At k <= 16 the epilogue warps only
// reduce each key tile to its two block maxima per row and pass them through a shared-memory
// ring to a selection warp that owns the same rows and does the bookkeeping: a compaction then
// delays nothing but its own warp, where it used to hold a TMEM accumulator (and with it the
// MMA pipeline, two accumulators deep) until it finished.
#include <cudaTypedefs.h>

#include <algorithm>
#include <climits>
#include <cmath>
#include <mutex>

#include "msa_device.cuh"
#include "msa_internal.h"

namespace msa {
namespace {

__device__ unsigned g_score_status = 0;
// Bound on the pipeline waits of this kernel (ring slots, accumulators); the waits that drain
// copies and MMAs still in flight before the CTA exits keep the fixed kWaitNs bound.  Set from
// the host by set_score_wait_limit (msa_set_wait_limit_ns).
__device__ unsigned long long g_score_wait_ns = kWaitNs;

constexpr int kRows = 128;     // UMMA M: rows per sub-tile
constexpr int kKeys = 128;     // UMMA N: keys per tile
constexpr int kGroupBlocks = 32;   // blocks staged per row before a store
constexpr int kTilesPerGroup = kGroupBlocks / (kKeys / kBlock);
// SELECT: candidate slots per row, CAP = 24 for k <= 16 and 56 for k <= 32 (k - 1 kept after
// each compaction); the row stride CAP + 1 is odd, so the 32 lanes' rows fall in distinct banks.
template <int D_IDX, int SUB, int CAP = 0>
struct ScoreSmem {
  static constexpr bool SELECT = CAP > 0;
  static constexpr int kCapStride = CAP + 1;
  static constexpr int kABytes = kRows * D_IDX * 2;
  static constexpr int kBBytes = kKeys * D_IDX * 2;
  // K_idx ring depth: six stages keep about two microseconds of key tiles in flight with two
  // sub-tiles per CTA (four beside the k <= 32 candidate buffers).  One sub-tile (SUB = 1: 128
  // rows, 256 TMEM columns, about 110 KB) runs two CTAs per SM: one CTA's MMAs run while the
  // other's epilogue drains its accumulators.  There the ring has four stages beside the k <= 16
  // buffers of 24 candidates and a 4-tile maxima ring (3.108 -> 3.088 ms at 128K against three
  // stages with 32 candidates), three beside the plain block scores' staging, two beside the
  // k <= 32 buffers.
  static constexpr int kStages =
      SUB == 1 ? (CAP > 32 ? 2 : (CAP > 24 ? 3 : 4)) : (SELECT && CAP > 32 ? 4 : 6);
  static constexpr int kCtasPerSm = SUB == 1 ? 2 : 1;
  static constexpr int kEpiWarps = 4 * SUB;
  static constexpr int kStageFloats = 32 * 33;        // 32 rows x 32 blocks, padded
  static constexpr int kOffA = 0;
  static constexpr int kOffB = kOffA + SUB * kABytes;
  static constexpr int kOffStage = kOffB + kStages * kBBytes;
  // SELECT: candidate scores of every epilogue row (row stride kCapStride), then their blocks
  static constexpr int kStageBytes =
      SELECT ? kEpiWarps * 32 * kCapStride * 8 : kEpiWarps * kStageFloats * 4;
  // SELECT with CAP <= 32: each epilogue warp hands its rows' block maxima to a selection warp of
  // its own through a ring of kRing key tiles (32 rows x 2 blocks, 8 bytes per row), so the
  // candidate bookkeeping never holds a TMEM accumulator.  CAP = 56 keeps the bookkeeping in the
  // epilogue warps (its compaction needs more registers than twice the threads leave).
  static constexpr int kRing = SELECT && CAP <= 32 ? (CAP <= 24 ? 4 : 8) : 0;
  static constexpr int kSelWarps = kRing > 0 ? kEpiWarps : 0;
  static constexpr int kOffRing = kOffStage + kStageBytes;
  static constexpr int kOffBar = kOffRing + kSelWarps * kRing * 32 * 8;
  // barriers: full_a, full_b[kStages], empty_b[kStages], tfull[2], tempty[2], done,
  // ring_full[kSelWarps][kRing], ring_empty[kSelWarps][kRing]
  static constexpr int kNumBars = 1 + 2 * kStages + 4 + 1 + 2 * kSelWarps * kRing;
  static constexpr int kOffTmem = kOffBar + kNumBars * 8;
  static constexpr int kBytes = kOffTmem + 16;
  static constexpr int kAlloc = kBytes + 1024;
  static constexpr int kThreads = 64 + 32 * (kEpiWarps + kSelWarps);
  static constexpr uint32_t kTmemCols = 2 * SUB * kKeys;
  static_assert(kTmemCols <= 512, "TMEM has 512 columns");
  static_assert(kAlloc <= 227 * 1024, "shared memory per CTA");
  static_assert(kOffB % 1024 == 0 && kOffStage % 1024 == 0, "1024-B aligned swizzle atoms");
};

__device__ __forceinline__ float max64(const uint32_t* v) {
  float m0 = fmax3(__uint_as_float(v[0]), __uint_as_float(v[1]), __uint_as_float(v[2]));
  float m1 = fmax3(__uint_as_float(v[3]), __uint_as_float(v[4]), __uint_as_float(v[5]));
  float m2 = fmax3(__uint_as_float(v[6]), __uint_as_float(v[7]), __uint_as_float(v[8]));
  float m3 = fmax3(__uint_as_float(v[9]), __uint_as_float(v[10]), __uint_as_float(v[11]));
#pragma unroll
  for (int c = 12; c < 60; c += 8) {
    m0 = fmax3(m0, __uint_as_float(v[c + 0]), __uint_as_float(v[c + 1]));
    m1 = fmax3(m1, __uint_as_float(v[c + 2]), __uint_as_float(v[c + 3]));
    m2 = fmax3(m2, __uint_as_float(v[c + 4]), __uint_as_float(v[c + 5]));
    m3 = fmax3(m3, __uint_as_float(v[c + 6]), __uint_as_float(v[c + 7]));
  }
  m0 = fmax3(m0, __uint_as_float(v[60]), __uint_as_float(v[61]));
  m1 = fmax3(m1, __uint_as_float(v[62]), __uint_as_float(v[63]));
  return fmax3(m0, m1, fmaxf(m2, m3));
}

// Bitonic sorting network over P2 registers, every index a compile-time constant: merge stage
// (K2, J) compares t with t ^ J, descending where bit K2 of t is clear.
template <int P2, int K2, int J>
__device__ __forceinline__ void bitonic_stage(float (&v)[P2]) {
#pragma unroll
  for (int t = 0; t < P2; ++t) {
    constexpr int kJ = J;
    const int u = t ^ kJ;
    if (u > t) {
      const float hi = fmaxf(v[t], v[u]), lo = fminf(v[t], v[u]);
      const bool desc = (t & K2) == 0;
      v[t] = desc ? hi : lo;
      v[u] = desc ? lo : hi;
    }
  }
  if constexpr (J > 1) bitonic_stage<P2, K2, J / 2>(v);
}
template <int P2, int K2>
__device__ __forceinline__ void bitonic_pass(float (&v)[P2]) {
  bitonic_stage<P2, K2, K2 / 2>(v);
  if constexpr (K2 < P2) bitonic_pass<P2, K2 * 2>(v);
}

// SELECT: a row's buffer always holds its candidates in ascending block order (blocks are
// appended in increasing order and compaction is stable), which is also the order that breaks
// score ties.  Compaction keeps the row's best min(cnt, km1) candidates: it finds the km1-th best
// score t (a bitonic sort of the scores, unrolled in registers), then keeps, in buffer order,
// every entry above t and the first entries equal to t until km1 are kept.  Returns the new tau:
// t once km1 entries are held, -inf while fewer, +inf for k = 1 (only the local block).
template <int CAP>
__device__ __forceinline__ float compact_row(float* sc, int* bl, int& cnt, int km1) {
  if (km1 == 0) {
    cnt = 0;
    return INFINITY;
  }
  constexpr int P2 = CAP <= 32 ? 32 : 64;
  float v[P2];
#pragma unroll
  for (int t = 0; t < P2; ++t) v[t] = t < cnt && t < CAP ? sc[t] : -INFINITY;
  bitonic_pass<P2, 2>(v);                        // descending overall
  // the km1-th best is the least of the first km1 sorted scores (a running min keeps every
  // index a constant, so v stays in registers)
  float th = INFINITY;
  int above = 0;
#pragma unroll
  for (int j = 0; j < P2; ++j)
    if (j < km1) th = fminf(th, v[j]);
#pragma unroll
  for (int j = 0; j < P2; ++j) above += v[j] > th;
  int eq_left = km1 - above, kept = 0;
  float sv[CAP];
  int bv[CAP];
#pragma unroll
  for (int t = 0; t < CAP; ++t) {
    sv[t] = sc[t];
    bv[t] = bl[t];
  }
#pragma unroll
  for (int t = 0; t < CAP; ++t) {
    if (t < cnt) {
      const bool eq = sv[t] == th;
      if (sv[t] > th || (eq && eq_left > 0)) {
        eq_left -= eq;
        sc[kept] = sv[t];
        bl[kept] = bv[t];
        ++kept;
      }
    }
  }
  cnt = kept;
  return kept == km1 ? th : -INFINITY;
}

// SELECT: offer block b's score m to a row's candidate buffer (blocks before the row's local
// block l only, strictly above the running threshold tau).
template <int CAP>
__device__ __forceinline__ void offer_block(float* sc, int* bl, int& cnt, float tau, int64_t b,
                                            int64_t l, float m) {
  if (b < l && m > tau) {
    sc[cnt] = m;
    bl[cnt] = (int)b;
    ++cnt;
  }
}

// SELECT: the row's final selection -- its best k-1 kept blocks (already ascending), then l,
// then -1 padding.  The whole warp calls it (the compaction is unrolled).
template <int CAP>
__device__ __forceinline__ void write_selection(float* sc, int* bl, int cnt, int km1, int kk,
                                                int64_t R, int log2_hkv, int64_t N, int64_t i,
                                                int64_t i_end, int64_t l, int32_t* idx) {
  compact_row<CAP>(sc, bl, cnt, km1);
  if (i < i_end) {
    const int rr = (int)(R & ((1 << log2_hkv) - 1));
    int32_t* out = idx + ((int64_t)rr * N + i) * kk;
    for (int j = 0; j < cnt; ++j) out[j] = bl[j];
    out[cnt] = (int32_t)l;
    for (int j = cnt + 1; j < kk; ++j) out[j] = -1;
  }
}

template <int D_IDX, int SUB, int CAP>
__global__ void __launch_bounds__(ScoreSmem<D_IDX, SUB, CAP>::kThreads,
                                  ScoreSmem<D_IDX, SUB, CAP>::kCtasPerSm)
    k_index_block_scores(const __grid_constant__ CUtensorMap tm_q,
                         const __grid_constant__ CUtensorMap tm_k, float* __restrict__ M,
                         int32_t* __restrict__ idx, int kk, int64_t N, int log2_hkv,
                         int64_t q_start, int64_t q_count, int64_t nblk, float scale,
                         const int* __restrict__ ktab) {
  using L = ScoreSmem<D_IDX, SUB, CAP>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
  const uint32_t sbase = smem_u32(smem);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int H_kv = 1 << log2_hkv;
  const int QT = kRows >> log2_hkv;                      // queries per sub-tile
  const int64_t per_cta = (int64_t)SUB * QT;
  const int64_t n_super = (q_count + per_cta - 1) / per_cta;
  const int64_t st = n_super - 1 - blockIdx.x;           // heaviest (latest) tiles first
  const int64_t i0 = q_start + st * per_cta;
  const int64_t i_end = min(i0 + per_cta, q_start + q_count);
  const int nkt = (int)((i_end - 1) / kKeys) + 1;         // key tiles covering [0, i_end)
  // first key tile: 0, or (packed variable-length batches) the first tile of the sequence that
  // holds this CTA's rows -- sequences start on 128-row boundaries and no CTA spans two of them
  const int kt0 = ktab != nullptr ? __ldg(ktab + (i0 >> 7)) : 0;
  const int64_t R0 = i0 << log2_hkv;                      // first (query, group) row

  const uint32_t bar0 = sbase + L::kOffBar;
  const uint32_t full_a = bar0;
  auto full_b = [&](int s) { return bar0 + 8u * (1 + s); };
  auto empty_b = [&](int s) { return bar0 + 8u * (1 + L::kStages + s); };
  auto tfull = [&](int a) { return bar0 + 8u * (1 + 2 * L::kStages + a); };
  auto tempty = [&](int a) { return bar0 + 8u * (3 + 2 * L::kStages + a); };
  const uint32_t done_bar = bar0 + 8u * (5 + 2 * L::kStages);
  auto ring_full = [&](int e, int slot) {
    return bar0 + 8u * (6 + 2 * L::kStages + e * L::kRing + slot);
  };
  auto ring_empty = [&](int e, int slot) {
    return bar0 + 8u * (6 + 2 * L::kStages + (L::kSelWarps + e) * L::kRing + slot);
  };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kOffTmem);

  if (threadIdx.x == 0) {
    mbar_init(full_a, 1);
    for (int s = 0; s < L::kStages; ++s) {
      mbar_init(full_b(s), 1);
      mbar_init(empty_b(s), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(tfull(a), 1);
      mbar_init(tempty(a), L::kEpiWarps);
    }
    mbar_init(done_bar, 1);
    for (int x = 0; x < L::kSelWarps * L::kRing; ++x) {
      mbar_init(bar0 + 8u * (6 + 2 * L::kStages + x), 32);
      mbar_init(bar0 + 8u * (6 + 2 * L::kStages + L::kSelWarps * L::kRing + x), 32);
    }
    fence_barrier_init();
  }
  if (warp == 1) tmem_alloc(smem_u32(tmem_slot), L::kTmemCols);
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const unsigned long long lim = g_score_wait_ns;          // pipeline waits only

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      prefetch_tensormap(&tm_q);
      prefetch_tensormap(&tm_k);
      mbar_expect_tx(full_a, SUB * L::kABytes);
      for (int s = 0; s < SUB; ++s)
        tma_load_2d(sbase + L::kOffA + s * L::kABytes, &tm_q, full_a, 0, (int)(R0 + s * kRows));
      int last_round[L::kStages];
      for (int s = 0; s < L::kStages; ++s) last_round[s] = -1;
      for (int kt = kt0; kt < nkt; ++kt) {
        const int u = kt - kt0;
        const int stg = u % L::kStages, round = u / L::kStages;
        if (!mbar_wait(empty_b(stg), (round & 1) ^ 1, &g_score_status, lim)) break;
        mbar_expect_tx(full_b(stg), L::kBBytes);
        tma_load_2d(sbase + L::kOffB + stg * L::kBBytes, &tm_k, full_b(stg), 0, kt * kKeys);
        last_round[stg] = round;
      }
      // never leave the CTA with a copy in flight
      mbar_wait(full_a, 0, &g_score_status);
      for (int s = 0; s < L::kStages; ++s)
        if (last_round[s] >= 0) mbar_wait(full_b(s), last_round[s] & 1, &g_score_status);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = umma_idesc_bf16(kRows, kKeys);
      constexpr uint32_t sbo = 8 * D_IDX * 2;            // 8 rows of one swizzle atom
      constexpr int swz = D_IDX * 2;                     // 128-B or 64-B swizzle rows
      if (mbar_wait(full_a, 0, &g_score_status, lim)) {
        tc_fence_after();
        for (int kt = kt0; kt < nkt; ++kt) {
          const int u = kt - kt0;
          const int stg = u % L::kStages, round = u / L::kStages;
          const int acc = u & 1, use = u >> 1;
          if (!mbar_wait(tempty(acc), (use & 1) ^ 1, &g_score_status, lim)) break;
          if (!mbar_wait(full_b(stg), round & 1, &g_score_status, lim)) break;
          tc_fence_after();
          const uint32_t b_addr = sbase + L::kOffB + stg * L::kBBytes;
#pragma unroll
          for (int s = 0; s < SUB; ++s) {
            const uint32_t d = tmem_base + (uint32_t)((acc * SUB + s) * kKeys);
            const uint32_t a_addr = sbase + L::kOffA + s * L::kABytes;
#pragma unroll
            for (int ks = 0; ks < D_IDX / 16; ++ks)
              umma_bf16(d, umma_desc_kmajor(a_addr + ks * 32, sbo, swz),
                        umma_desc_kmajor(b_addr + ks * 32, sbo, swz), idesc, ks > 0 ? 1u : 0u);
          }
          umma_commit(empty_b(stg));
          umma_commit(tfull(acc));
        }
      }
      umma_commit(done_bar);                           // every MMA issued has completed
      mbar_wait(done_bar, 0, &g_score_status);
    }
  } else if (warp >= 2 + L::kEpiWarps) {
    // ----------------------------------------------- selection (SELECT, CAP <= 32)
    // selection warp e takes the rows of epilogue warp e (warp 2 + e) from the ring
    if constexpr (L::kRing > 0) {
      const int e = warp - 2 - L::kEpiWarps;
      const int s = e >> 2, q = (e + 2) & 3;
      const int64_t R = R0 + (int64_t)s * kRows + 32 * q + lane;
      const int64_t i = R >> log2_hkv;
      const int64_t l = i >> 6;
      float* sc = reinterpret_cast<float*>(smem + L::kOffStage) + (e * 32 + lane) * L::kCapStride;
      int* bl = reinterpret_cast<int*>(smem + L::kOffStage) +
                (L::kEpiWarps + e) * 32 * L::kCapStride + lane * L::kCapStride;
      const float2* ring = reinterpret_cast<const float2*>(smem + L::kOffRing) + e * L::kRing * 32;
      const int km1 = kk - 1;
      int cnt = 0;
      float tau = km1 > 0 ? -INFINITY : INFINITY;
      bool ok = true;
      for (int kt = kt0; kt < nkt; ++kt) {
        const int u = kt - kt0, slot = u % L::kRing, round = u / L::kRing;
        if (!__all_sync(0xffffffffu,
                        mbar_wait(ring_full(e, slot), round & 1, &g_score_status, lim))) {
          ok = false;
          break;
        }
        const float2 m = ring[slot * 32 + lane];
        mbar_arrive(ring_empty(e, slot));
        offer_block<CAP>(sc, bl, cnt, tau, 2 * (int64_t)kt, l, m.x);
        offer_block<CAP>(sc, bl, cnt, tau, 2 * (int64_t)kt + 1, l, m.y);
        if (__any_sync(0xffffffffu, cnt > CAP - 2)) tau = compact_row<CAP>(sc, bl, cnt, km1);
      }
      if (ok) write_selection<CAP>(sc, bl, cnt, km1, kk, R, log2_hkv, N, i, i_end, l, idx);
    }
  } else {
    // --------------------------------------------------------------- epilogue
    const int e = warp - 2;
    const int s = e >> 2;                                 // sub-tile
    const int q = warp & 3;                               // TMEM lane quarter
    if constexpr (L::kRing > 0) {
      // block maxima of each key tile into the ring of this warp's selection warp
      const int64_t R = R0 + (int64_t)s * kRows + 32 * q + lane;
      const int64_t l = (R >> log2_hkv) >> 6;             // local block of this row
      float2* ring = reinterpret_cast<float2*>(smem + L::kOffRing) + e * L::kRing * 32;
      for (int kt = kt0; kt < nkt; ++kt) {
        const int u = kt - kt0, acc = u & 1, use = u >> 1;
        const int slot = u % L::kRing, round = u / L::kRing;
        if (!__all_sync(0xffffffffu, mbar_wait(tfull(acc), use & 1, &g_score_status, lim))) break;
        tc_fence_after();
        float m[2] = {-INFINITY, -INFINITY};
        {
          // both blocks' loads in flight at once; only their maxima are used, so the two share
          // one (dead) destination vector
          const int64_t b0 = 2 * (int64_t)kt;
          const bool need0 = __any_sync(0xffffffffu, b0 < l);
          const bool need1 = __any_sync(0xffffffffu, b0 + 1 < l);
          uint32_t v[64];
          float mx0 = -INFINITY, mx1 = -INFINITY;
          const uint32_t taddr = tmem_base + ((uint32_t)(32 * q) << 16) +
                                 (uint32_t)((acc * SUB + s) * kKeys);
          if (need0) MSA_TMEM_LDMAX64(taddr, v, mx0);
          if (need1) MSA_TMEM_LDMAX64(taddr + 64, v, mx1);
          tmem_ld_wait();
          if (b0 < l) m[0] = mx0 * scale;
          if (b0 + 1 < l) m[1] = mx1 * scale;
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(tempty(acc));
        if (!__all_sync(0xffffffffu,
                        mbar_wait(ring_empty(e, slot), (round & 1) ^ 1, &g_score_status, lim)))
          break;
        ring[slot * 32 + lane] = make_float2(m[0], m[1]);
        mbar_arrive(ring_full(e, slot));
      }
    } else if constexpr (L::SELECT) {
      const int64_t R = R0 + (int64_t)s * kRows + 32 * q + lane;
      const int64_t i = R >> log2_hkv;
      const int64_t l = i >> 6;                           // local block of this row
      float* sc = reinterpret_cast<float*>(smem + L::kOffStage) + (e * 32 + lane) * L::kCapStride;
      int* bl = reinterpret_cast<int*>(smem + L::kOffStage) +
                (L::kEpiWarps + e) * 32 * L::kCapStride + lane * L::kCapStride;
      const int km1 = kk - 1;
      int cnt = 0;
      float tau = km1 > 0 ? -INFINITY : INFINITY;
      bool ok = true;
      for (int kt = kt0; kt < nkt; ++kt) {
        const int acc = (kt - kt0) & 1, use = (kt - kt0) >> 1;
        // every lane waits; the warp leaves together if any lane gave up (the loop body has
        // warp-wide operations)
        if (!__all_sync(0xffffffffu, mbar_wait(tfull(acc), use & 1, &g_score_status, lim))) {
          ok = false;
          break;
        }
        tc_fence_after();
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int64_t b = 2 * (int64_t)kt + h;
          if (!__any_sync(0xffffffffu, b < l)) continue;   // no row of the warp needs it
          uint32_t v[64];
          float mx;
          const uint32_t taddr = tmem_base + ((uint32_t)(32 * q) << 16) +
                                 (uint32_t)((acc * SUB + s) * kKeys + 64 * h);
          MSA_TMEM_LDMAX64(taddr, v, mx);
          tmem_ld_wait();
          if (b < l) offer_block<CAP>(sc, bl, cnt, tau, b, l, mx * scale);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(tempty(acc));
        if (__any_sync(0xffffffffu, cnt > CAP - 2)) tau = compact_row<CAP>(sc, bl, cnt, km1);
      }
      if (ok) write_selection<CAP>(sc, bl, cnt, km1, kk, R, log2_hkv, N, i, i_end, l, idx);
    } else {
      float* stage = reinterpret_cast<float*>(smem + L::kOffStage) + e * L::kStageFloats;
      const int64_t Rw = R0 + (int64_t)s * kRows + 32 * q;  // first row of this warp
      const int64_t R = Rw + lane;
      const int64_t i = R >> log2_hkv;
      const int64_t l = i >> 6;                             // local block of this row
      const float ninf = -INFINITY;

      auto flush = [&](int g, int ncols) {
        __syncwarp();
        for (int rho = 0; rho < 32; ++rho) {
          const int64_t Rr = Rw + rho;
          const int64_t ir = Rr >> log2_hkv;
          if (ir >= i_end) break;
          const int rr = (int)(Rr & (H_kv - 1));
          const int64_t b = (int64_t)g * kGroupBlocks + lane;
          if (b < nblk) {
            const float val = lane < ncols ? stage[rho * 33 + lane] : ninf;
            M[((int64_t)rr * q_count + (ir - q_start)) * nblk + b] = val;
          }
        }
        __syncwarp();
      };

      bool ok = true;
      for (int kt = 0; kt < nkt; ++kt) {
        const int acc = kt & 1, use = kt >> 1;
        // every lane waits; the warp leaves together if any lane gave up (the loop body has
        // warp-wide operations)
        if (!__all_sync(0xffffffffu, mbar_wait(tfull(acc), use & 1, &g_score_status, lim))) {
          ok = false;
          break;
        }
        tc_fence_after();
  #pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int64_t b = 2 * (int64_t)kt + h;
          uint32_t v[64];
          float mx;
          const uint32_t taddr = tmem_base + ((uint32_t)(32 * q) << 16) +
                                 (uint32_t)((acc * SUB + s) * kKeys + 64 * h);
          MSA_TMEM_LDMAX64(taddr, v, mx);
          tmem_ld_wait();
          float m = ninf;
          if (b < l) {
            m = mx * scale;
          } else if (b == l) {                              // diagonal block: keys j <= i only
            const int lim = (int)(i - 64 * b);
  #pragma unroll
            for (int c = 0; c < 64; ++c)
              if (c > lim) v[c] = __float_as_uint(ninf);
            m = max64(v) * scale;
          }
          stage[lane * 33 + (int)(b & (kGroupBlocks - 1))] = m;
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(tempty(acc));
        const int kt_in_group = kt % kTilesPerGroup;
        if (kt_in_group == kTilesPerGroup - 1 || kt == nkt - 1)
          flush(kt / kTilesPerGroup, 2 * (kt_in_group + 1));
      }
      if (ok) {
        // blocks after the last key tile are in every row's future
        const int64_t b_first = ((int64_t)(nkt - 1) / kTilesPerGroup + 1) * kGroupBlocks;
        for (int rho = 0; rho < 32; ++rho) {
          const int64_t Rr = Rw + rho;
          const int64_t ir = Rr >> log2_hkv;
          if (ir >= i_end) break;
          const int rr = (int)(Rr & (H_kv - 1));
          float* row = M + ((int64_t)rr * q_count + (ir - q_start)) * nblk;
          for (int64_t b = b_first + lane; b < nblk; b += 32) row[b] = ninf;
        }
      }
    }
  }

  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, L::kTmemCols);
  }
}

template <int D_IDX, int SUB, int CAP>
cudaError_t launch_scores(const CUtensorMap& tq, const CUtensorMap& tk, float* M, int32_t* idx,
                          int kk, int64_t N, int H_kv, int64_t q_start, int64_t q_count,
                          int64_t nblk, const int* ktab, cudaStream_t stream) {
  using L = ScoreSmem<D_IDX, SUB, CAP>;
  auto kern = k_index_block_scores<D_IDX, SUB, CAP>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kAlloc);
  if (e != cudaSuccess) return e;
  int log2_hkv = 0;
  while ((1 << log2_hkv) < H_kv) ++log2_hkv;
  const int64_t per_cta = (int64_t)SUB * (kRows / H_kv);
  const int64_t grid = (q_count + per_cta - 1) / per_cta;
  const float scale = (float)(1.0 / std::sqrt((double)D_IDX));
  kern<<<(unsigned)grid, L::kThreads, L::kAlloc, stream>>>(tq, tk, M, idx, kk, N, log2_hkv,
                                                           q_start, q_count, nblk, scale, ktab);
  return cudaGetLastError();
}

}  // namespace

static cudaError_t launch_index(const void* q_idx, const void* k_idx, float* M, int32_t* idx,
                               int kk, int64_t N, int H_kv, int d_idx, int64_t q_start,
                               int64_t q_count, const int* ktab, cudaStream_t stream) {
  CUtensorMap tq, tk;
  const int swz = d_idx * 2;   // one swizzle row per index vector
  cudaError_t e = make_tma_2d_bf16(&tq, q_idx, (uint64_t)d_idx, (uint64_t)N * H_kv, d_idx, kRows, swz);
  if (e != cudaSuccess) return e;
  e = make_tma_2d_bf16(&tk, k_idx, (uint64_t)d_idx, (uint64_t)N, d_idx, kKeys, swz);
  if (e != cudaSuccess) return e;
  const int64_t nblk = (N + kBlock - 1) / kBlock;
#define MSA_SCORES(D, SUB, CAP) \
  launch_scores<D, SUB, CAP>(tq, tk, M, idx, kk, N, H_kv, q_start, q_count, nblk, ktab, stream)
  // one sub-tile per CTA, two CTAs per SM (fused branch at 128K: 3.53 -> 3.11 ms at k = 16,
  // 4.51 -> 3.63 ms at k = 32, whose 168-register compaction fits two 192-thread CTAs with a
  // two-stage key ring)
  if (idx != nullptr && kk <= 16) return d_idx == 64 ? MSA_SCORES(64, 1, 24) : MSA_SCORES(32, 1, 24);
  if (idx != nullptr) return d_idx == 64 ? MSA_SCORES(64, 1, 56) : MSA_SCORES(32, 1, 56);
  return d_idx == 64 ? MSA_SCORES(64, 1, 0) : MSA_SCORES(32, 1, 0);
#undef MSA_SCORES
}

cudaError_t launch_index_block_scores(const void* q_idx, const void* k_idx, float* M, int64_t N,
                                      int H_kv, int d_idx, int64_t q_start, int64_t q_count,
                                      cudaStream_t stream) {
  return launch_index(q_idx, k_idx, M, nullptr, 0, N, H_kv, d_idx, q_start, q_count, nullptr,
                      stream);
}

cudaError_t launch_index_select(const void* q_idx, const void* k_idx, int32_t* idx, int64_t N,
                                int H_kv, int d_idx, int k, int64_t q_start, int64_t q_count,
                                cudaStream_t stream, const int* ktab) {
  return launch_index(q_idx, k_idx, nullptr, idx, k, N, H_kv, d_idx, q_start, q_count, ktab,
                      stream);
}

// a bound on the query rows one CTA covers (two sub-tiles' worth; every variant dispatched
// above runs one), used to align variable-length sequences
int index_rows_per_cta(int H_kv) { return 2 * (kRows / H_kv); }

cudaError_t set_score_wait_limit(unsigned long long ns) {
  return cudaMemcpyToSymbol(g_score_wait_ns, &ns, sizeof(ns));
}

cudaError_t read_reset_score_status(unsigned* out) {
  unsigned zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(out, g_score_status, sizeof(unsigned));
  if (e != cudaSuccess) return e;
  return cudaMemcpyToSymbol(g_score_status, &zero, sizeof(unsigned));
}

}  // namespace msa

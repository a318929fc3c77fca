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
// one bucket, G rows each, into one 128-row UMMA tile:
//   S   = Q_stack  [128 x d_h]   . K_b^T     [d_h x 64]     tcgen05 -> TMEM columns [0, 64)
//   S^i = Qi_stack [128 x d_idx] . K_idx_b^T [d_idx x 64]   tcgen05 -> TMEM columns [64, 128)
// (an entry's index query is repeated on its G rows, so every TMEM lane holds the student
// scores of its own entry).  The teacher's head mean is a reduce-scatter over the entry's G
// lanes by shuffles, after which each lane owns 64/G of the block's tokens; each entry leaves
// one partial (sum P (ln P - S^idx), sum P, and the student's max and sum of exponentials in the
// log2 domain) at the fixed position of its (group, row, slot).  A merge kernel combines a row's
// partials in slot order: no atomic update of any result.
#include <cmath>

#include "attn_tile.cuh"
#include "msa_device.cuh"
#include "msa_internal.h"

namespace msa {
namespace {

__device__ unsigned g_kl_status = 0;

constexpr int kKlRows = 128;                 // UMMA M
constexpr int kKlThreads = 128;              // 4 warps: TMEM lane quarters
constexpr int kKlPlanWarps = 4;
constexpr float kLn2 = 0.693147180559945309f;
constexpr float kLog2e = 1.442695040888963407f;

template <int D_H>
struct KlSmem {
  static constexpr int kHalves = D_H / 64;
  static constexpr int kQHalf = kKlRows * 128;    // 128 rows x 64 dims, bf16, SW128
  static constexpr int kKHalf = 64 * 128;         // 64 keys x 64 dims
  static constexpr int kOffQ = 0;
  static constexpr int kOffQi = kOffQ + kHalves * kQHalf;   // stacked index queries (<= 64 dims)
  static constexpr int kOffK = kOffQi + kQHalf;
  static constexpr int kOffKi = kOffK + kHalves * kKHalf;   // the block's index keys
  static constexpr int kOffBar = kOffKi + kKHalf;
  static constexpr int kOffMisc = kOffBar + 16;
  static constexpr int kOffEnt = kOffMisc + 16;   // entries of this tile and the next
  static constexpr int kBytes = kOffEnt + 2 * kKlRows * 4;
  static constexpr int kAlloc = kBytes + 1024;
  static constexpr uint32_t kTmemCols = 128;      // S, then S^idx
};
constexpr int kKlCtasPerSm = 3;
static_assert(kKlCtasPerSm * (KlSmem<128>::kAlloc + 1024) <= 228 * 1024, "3 CTAs per SM");

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

__global__ void __launch_bounds__(32 * kKlPlanWarps)
    k_kl_plan(const int32_t* __restrict__ idx, int64_t N, int kk, int64_t nblk, int pass,
              int* count, const int* offset, int* cursor, int* entries) {
  __shared__ int s_U[kKlPlanWarps][kMaxKeys];
  __shared__ unsigned s_mask[kKlPlanWarps][kMaxKeys];
  const int warp = threadIdx.x >> 5;
  const int r = blockIdx.y;
  const int64_t i0 = ((int64_t)blockIdx.x * kKlPlanWarps + warp) * kTileQ;
  if (i0 >= N) return;
  with_epl(kk, [&](auto e) {
    kl_plan_tile<decltype(e)::value>(idx, r, i0, N, kk, nblk, pass, s_U[warp], s_mask[warp],
                                     count, offset, cursor, entries);
    return 0;
  });
}

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

template <int D_H, int G>
__global__ void __launch_bounds__(kKlThreads, kKlCtasPerSm)
    k_kl_kvouter(const __grid_constant__ CUtensorMap tm_q, const __nv_bfloat16* __restrict__ q,
                 const __nv_bfloat16* __restrict__ k, const __nv_bfloat16* __restrict__ q_idx,
                 const __nv_bfloat16* __restrict__ k_idx, const float* __restrict__ lse,
                 const int* __restrict__ entries, const int* __restrict__ offset,
                 const int* __restrict__ tile_off, int nbuckets, int64_t nblk, int64_t N,
                 int H_kv, int d_idx, int kk, float4* __restrict__ part, float scale_log2,
                 float idx_scale) {
  using L = KlSmem<D_H>;
  constexpr int kEpt = kKlRows / G;          // entries per work tile
  constexpr int kCpl = 64 / G;               // columns a lane owns after the reduce-scatter
  constexpr int kChunks = D_H / 8;           // 16-byte chunks per K / Q row
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t sb = smem_u32(smem);
  const uint32_t mma_bar = sb + L::kOffBar, q_bar = sb + L::kOffBar + 8;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kOffMisc);
  int* s_ent = reinterpret_cast<int*>(smem + L::kOffEnt);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tid = threadIdx.x;
  const int H_q = H_kv * G;
  const int ichunks = d_idx / 8;             // 16-byte chunks per index row

  if (tid == 0) {
    mbar_init(mma_bar, 1);
    mbar_init(q_bar, 1);
    fence_barrier_init();
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(tmem_slot), L::kTmemCols);
    tc_fence_before();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  const int total_tiles = tile_off[nbuckets];
  const int64_t kv_stride = (int64_t)H_kv * D_H;
  uint32_t phase = 0, qphase = 0;
  bool ok = true;

  // a contiguous range of work tiles per CTA (consecutive tiles often share a bucket)
  const int per = (total_tiles + gridDim.x - 1) / gridDim.x;
  const int t_beg = blockIdx.x * per;
  const int t_end = min(total_tiles, t_beg + per);
  int bucket = 0;
  if (t_beg < t_end) {
    int lo = 0, hi = nbuckets;                             // tile_off[lo] <= t_beg < tile_off[hi]
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (__ldg(tile_off + mid) <= t_beg) lo = mid; else hi = mid;
    }
    bucket = lo;
  }
  int next_off = t_beg < t_end ? __ldg(tile_off + bucket + 1) : 0;
  auto describe = [&](int tile, int& bkt, int& nxt, int& e0, int& n_e) {
    while (nxt <= tile) {
      ++bkt;
      nxt = __ldg(tile_off + bkt + 1);
    }
    e0 = __ldg(offset + bkt) + (tile - __ldg(tile_off + bkt)) * kEpt;
    n_e = min(kEpt, __ldg(offset + bkt + 1) - e0);
  };
  // K_b and K_idx_b of a bucket (rows past the sequence: zeros; they are masked anyway)
  auto load_k = [&](int bkt) {
    const int rb = (int)(bkt / nblk);
    const int64_t bb = bkt - (int64_t)rb * nblk;
    const __nv_bfloat16* kb = k + (bb * kBlock * H_kv + rb) * (int64_t)D_H;
    for (int x = tid; x < kBlock * kChunks; x += kKlThreads) {
      const int j = x / kChunks, c = x - j * kChunks;
      const uint32_t off = (c >> 3) * L::kKHalf + j * 128 + (((c & 7) ^ (j & 7)) << 4);
      if (bb * kBlock + j < N) kl_cp_async16(sb + L::kOffK + off, kb + j * kv_stride + c * 8);
      else kl_zero16(sb + L::kOffK + off);
    }
    const __nv_bfloat16* kib = k_idx + bb * kBlock * (int64_t)d_idx;
    for (int x = tid; x < kBlock * ichunks; x += kKlThreads) {
      const int j = x / ichunks, c = x - j * ichunks;
      const uint32_t off = j * 128 + ((c ^ (j & 7)) << 4);
      if (bb * kBlock + j < N) kl_cp_async16(sb + L::kOffKi + off, kib + (int64_t)j * d_idx + c * 8);
      else kl_zero16(sb + L::kOffKi + off);
    }
  };
  // the stacked query rows (entry e's heads are rows e*G .. e*G+G-1) and the stacked index
  // queries (entry e's index query on each of its G rows); ent: the tile's entries in smem
  auto gather_q = [&](int bkt, const int* ent, int n_ent) {
    const int rb = (int)(bkt / nblk);
    if (G == 8) {
      // one lane of warp 0 per entry: the boxes are issued in parallel, not one after another
      if (warp == 0) {
        if (lane == 0) mbar_expect_tx(q_bar, (uint32_t)(n_ent * 8 * 128 * L::kHalves));
        __syncwarp();
        if (lane < n_ent) {
          const int i = ent[lane] >> 6;
#pragma unroll
          for (int bx = 0; bx < L::kHalves; ++bx)
            tma_load_3d(sb + L::kOffQ + bx * L::kQHalf + lane * 1024, &tm_q, q_bar, 64 * bx,
                        rb * 8, i);
        }
      }
    } else {
      for (int x = tid; x < n_ent * G * kChunks; x += kKlThreads) {
        const int R = x / kChunks, c = x - R * kChunks;
        const int e = R / G, h = R - e * G;
        const int64_t i = ent[e] >> 6;
        const uint32_t off = (c >> 3) * L::kQHalf + R * 128 + (((c & 7) ^ (R & 7)) << 4);
        kl_cp_async16(sb + L::kOffQ + off, q + (i * H_q + (int64_t)rb * G + h) * D_H + c * 8);
      }
    }
    for (int x = tid; x < n_ent * G * ichunks; x += kKlThreads) {
      const int R = x / ichunks, c = x - R * ichunks;
      const int64_t i = ent[R / G] >> 6;
      const uint32_t off = R * 128 + ((c ^ (R & 7)) << 4);
      kl_cp_async16(sb + L::kOffQi + off, q_idx + (i * H_kv + rb) * d_idx + c * 8);
    }
  };

  int e0 = 0, n_e = 0;
  if (t_beg < t_end) {
    describe(t_beg, bucket, next_off, e0, n_e);
    load_k(bucket);
    if (tid < n_e) s_ent[tid] = __ldg(entries + e0 + tid);
    __syncthreads();
    gather_q(bucket, s_ent, n_e);
  }
  const int R = 32 * warp + lane;                          // this thread's row (TMEM lane)
  for (int tile = t_beg; tile < t_end && ok; ++tile) {
    const int cur = (tile - t_beg) & 1;
    const int* ent_cur = s_ent + cur * kKlRows;
    const int r = (int)(bucket / nblk);
    const int64_t b = bucket - (int64_t)r * nblk;
    const int rows = n_e * G;
    asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    bool qok = true;
    if (G == 8 && tid == 0) qok = mbar_wait(q_bar, qphase, &g_kl_status);
    qphase ^= 1u;
    ok = __syncthreads_and(qok);
    if (!ok) break;
    // this row's entry and its head's forward LSE, loaded under the MMAs
    const bool rv = R < rows;
    const int e = R / G, h = R - e * G;
    const int ent = rv ? ent_cur[e] : 0;
    const float lse_raw = rv ? __ldg(lse + (int64_t)(r * G + h) * N + (ent >> 6)) : 0.f;

    // ---- S = Q_stack K_b^T (columns 0..63) and S^idx = Qi_stack K_idx_b^T (columns 64..127)
    if (tid == 0) {
      tc_fence_after();
      constexpr uint32_t idesc = umma_idesc_bf16(kKlRows, 64);
#pragma unroll
      for (int ks = 0; ks < D_H / 16; ++ks) {
        const uint32_t a = sb + L::kOffQ + (ks >> 2) * L::kQHalf + (ks & 3) * 32;
        const uint32_t bk = sb + L::kOffK + (ks >> 2) * L::kKHalf + (ks & 3) * 32;
        umma_bf16(tmem, umma_desc_kmajor(a, 1024, 128), umma_desc_kmajor(bk, 1024, 128), idesc,
                  ks > 0 ? 1u : 0u);
      }
      for (int ks = 0; ks < d_idx / 16; ++ks) {
        const uint32_t a = sb + L::kOffQi + ks * 32;
        const uint32_t bk = sb + L::kOffKi + ks * 32;
        umma_bf16(tmem + 64, umma_desc_kmajor(a, 1024, 128), umma_desc_kmajor(bk, 1024, 128),
                  idesc, ks > 0 ? 1u : 0u);
      }
      umma_commit(mma_bar);
    }
    // the next tile's entries, also under the MMAs
    const bool has_next = tile + 1 < t_end;
    int n_bucket = bucket, n_next = next_off, n_e0 = 0, n_ne = 0;
    if (has_next) {
      describe(tile + 1, n_bucket, n_next, n_e0, n_ne);
      if (tid < n_ne) s_ent[(cur ^ 1) * kKlRows + tid] = __ldg(entries + n_e0 + tid);
    }
    ok = __syncthreads_and(mbar_wait(mma_bar, phase, &g_kl_status));
    if (!ok) break;
    phase ^= 1u;
    tc_fence_after();

    // ---- shared memory is free: the next tile's rows (and its keys for a new bucket)
    if (has_next) {
      if (n_bucket != bucket) load_k(n_bucket);
      gather_q(n_bucket, s_ent + (cur ^ 1) * kKlRows, n_ne);
    }
    asm volatile("cp.async.commit_group;" ::: "memory");

    // ---- row R = (entry e, head h): teacher probabilities of the block's tokens
    int cmax = -1;                                         // last visible column, -1: none
    if (rv) {
      const int64_t i = ent >> 6;
      cmax = b == (i >> 6) ? (int)(i - b * kBlock) : kBlock - 1;
    }
    const float lse2 = lse_raw * kLog2e;
    float a[64];
    {
      uint32_t s[64];
      MSA_TMEM_LD64(tmem + ((uint32_t)(32 * warp) << 16), s);
      tmem_ld_wait();
#pragma unroll
      for (int c = 0; c < 64; c += 2) {
        float x0, x1;
        ffma2(x0, x1, __uint_as_float(s[c]), __uint_as_float(s[c + 1]), scale_log2, scale_log2,
              -lse2, -lse2);
        a[c] = c <= cmax ? ex2(x0) : 0.f;
        a[c + 1] = c + 1 <= cmax ? ex2(x1) : 0.f;
      }
    }
    lane_split<G, true>(a, h);                             // a[c]: G * P of column kCpl*h + c
    float si[64];
    {
      uint32_t s[64];
      MSA_TMEM_LD64(tmem + ((uint32_t)(32 * warp) << 16) + 64, s);
      tmem_ld_wait();
#pragma unroll
      for (int c = 0; c < 64; ++c) si[c] = __uint_as_float(s[c]);
    }
    lane_split<G, false>(si, h);                           // si[c]: raw S^idx of the same column
    tc_fence_before();

    // ---- this lane's columns: sum P (ln P - S^idx), sum P, student max / sum (log2 domain)
    const int cb = kCpl * h;
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
    // ---- combine the entry's G lanes; its first lane writes the partial
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
    if (rv && h == 0) {
      const int64_t i = ent >> 6;
      part[((int64_t)r * N + i) * kk + (ent & 63)] = make_float4(C, W, mx, l);
    }
    __syncthreads();                                       // TMEM read before the next MMA
    bucket = n_bucket;
    next_off = n_next;
    e0 = n_e0;
    n_e = n_ne;
  }
  asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
  if (G == 8 && !ok && tid == 0) {
    // a wait gave up: let this tile's Q copies land before the CTA exits (the phase of the
    // last wait on q_bar; it returns at once if that wait had succeeded)
    mbar_wait(q_bar, qphase ^ 1u, &g_kl_status);
  }
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, L::kTmemCols);
  }
}

// ---------------------------------------------------------------------- merge --
// One thread per (group, row): KL = sum_e C_e + (sum_e W_e) * LSE^idx, with LSE^idx merged from
// the entries' (max, sum) pairs in slot order.
__global__ void __launch_bounds__(256)
    k_kl_merge(const int32_t* __restrict__ idx, const float4* __restrict__ part, float* kl,
               int64_t N, int H_kv, int kk) {
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
  kl[x] = C + W * (mx + __log2f(l)) * kLn2;
}

}  // namespace

size_t kl_ws_bytes(int64_t N, int H_kv, int kk) {
  const int64_t nb = (int64_t)H_kv * ((N + kBlock - 1) / kBlock);
  auto a256 = [](size_t x) { return (x + 255) & ~size_t(255); };
  const size_t sel = (size_t)H_kv * N * kk;
  return 4 * a256(4 * (size_t)(nb + 1)) + a256(4 * sel) + a256(16 * sel);
}

cudaError_t launch_kl_loss_fwd(const void* q, const void* k, const void* q_idx, const void* k_idx,
                               const int32_t* idx, const float* lse, float* kl, int64_t N, int H_q,
                               int H_kv, int d_h, int d_idx, int kk, void* ws,
                               cudaStream_t st) {
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

  cudaError_t e = cudaMemsetAsync(count, 0, sizeof(int) * (size_t)nb, st);
  if (e != cudaSuccess) return e;
  const int64_t tiles = (N + kTileQ - 1) / kTileQ;
  const dim3 pgrid((unsigned)((tiles + kKlPlanWarps - 1) / kKlPlanWarps), (unsigned)H_kv);
  k_kl_plan<<<pgrid, 32 * kKlPlanWarps, 0, st>>>(idx, N, kk, nblk, 0, count, offset, cursor,
                                                 entries);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if ((e = launch_attn_scan(count, offset, tile_off, cursor, nb, kKlRows / G, st)) != cudaSuccess)
    return e;
  k_kl_plan<<<pgrid, 32 * kKlPlanWarps, 0, st>>>(idx, N, kk, nblk, 1, count, offset, cursor,
                                                 entries);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;

  CUtensorMap tq;
  e = make_tma_3d_bf16(&tq, q, (uint64_t)d_h, (uint64_t)H_q, (uint64_t)N, 64, G, 1, 128);
  if (e != cudaSuccess) return e;
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
  auto run = [&](auto kern, int smem) -> cudaError_t {
    cudaError_t x = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (x != cudaSuccess) return x;
    const int grid = kKlCtasPerSm * sms;                   // persistent: 3 CTAs per SM
    kern<<<grid, kKlThreads, smem, st>>>(tq, qq, kp, qi, ki, lse, entries, offset, tile_off, nb,
                                         nblk, N, H_kv, d_idx, kk, part, scale_log2, idx_scale);
    return cudaGetLastError();
  };
  auto dispatch_g = [&](auto dh) -> cudaError_t {
    constexpr int D = decltype(dh)::value;
    const int smem = KlSmem<D>::kAlloc;
    switch (G) {
      case 1: return run(k_kl_kvouter<D, 1>, smem);
      case 2: return run(k_kl_kvouter<D, 2>, smem);
      case 4: return run(k_kl_kvouter<D, 4>, smem);
      default: return run(k_kl_kvouter<D, 8>, smem);
    }
  };
  e = d_h == 128 ? dispatch_g(std::integral_constant<int, 128>())
                 : dispatch_g(std::integral_constant<int, 64>());
  if (e != cudaSuccess) return e;
  const int64_t n = (int64_t)H_kv * N;
  k_kl_merge<<<(unsigned)((n + 255) / 256), 256, 0, st>>>(idx, part, kl, N, H_kv, kk);
  return cudaGetLastError();
}

cudaError_t read_reset_kl_status(unsigned* out) {
  unsigned zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(out, g_kl_status, sizeof(unsigned));
  if (e != cudaSuccess) return e;
  return cudaMemcpyToSymbol(g_kl_status, &zero, sizeof(unsigned));
}

}  // namespace msa

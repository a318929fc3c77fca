// Block-major ("KV-outer") pass of the sparse main branch («MiniMax-M3：MSA 技术报告速读»,
// section 主分支 eq. O^(h)_i; the kernel section's organisation in which a selected KV block
// gathers the queries that chose it and stacks them to fill tensor-core MMAs).
//
// Input: the private selections of a query chunk -- (query, slot) pairs whose block fewer than
// kSharedMin queries of the same 16-query tile selected -- bucketed by (group r, block b).  A work
// tile is up to 128/G entries of one bucket; their G heads stack into the 128 rows of one UMMA
// tile:
//   S = Q_stack [128 x d_h] . K_b^T [d_h x 64]       tcgen05, bf16 -> fp32 in TMEM
//   row-wise softmax over the block's visible keys   one thread per row (TMEM lane)
//   O = P [128 x 64] . V_b [64 x d_h]                tcgen05, P read from TMEM, V MN-major
// and every row writes a partial: O normalised by its own sum (bf16) and its log2-domain LSE, at
// the fixed position of its (group, query, slot) -- a query's partials are contiguous, so the
// merge in the shared-block pass (k_attn_shared.cu) reads them in slot order without an index.
//
// One persistent, warp-specialised CTA per SM:
//   warp 0      query rows of each tile into a ring of Q stages (TMA at G = 8: one 4-D box per
//               entry, its 8 head rows of every 64-dim half; cp.async otherwise)
//   warp 10     K_b and V_b of each new bucket into one of two K/V stages (TMA, 64-token boxes;
//               rows past the sequence read as zeros)
//   warp 1      the MMA issuer: S of tile j, then O of tile j-1, so the tensor pipe computes the
//               next tile's scores while the softmax of the current one runs
//   warps 2-9   two epilogue groups of four warps (one per TMEM lane quarter) taking alternate
//               tiles: softmax -> P into TMEM -> O -> the partial stores
// TMEM holds two score buffers (S, then P written over its first columns once S is read) and two
// O buffers.  A score buffer is free again as soon as the O MMA that read its P has completed,
// an O buffer once its group has stored the partial: the next tile's S never waits for a store.
// The tiles of each KV group are split into one contiguous range per CTA, group after group, so
// the CTAs gather query rows of one group at a time (a chunk's rows of one group fit in L2) and a
// CTA's consecutive tiles mostly share their bucket's K_b and V_b.
// Every wait is bounded; a wait that gives up sets the device status word and an abort flag that
// every role checks, and each role drains its copies / MMAs in flight before the CTA exits.
#include <cmath>

#include "msa_device.cuh"
#include "msa_internal.h"

namespace msa {
namespace {

__device__ unsigned g_kvo_status = 0;

constexpr int kRowsT = 128;                // UMMA M
constexpr int kWarpsKvo = 11;              // 0 query rows, 1 MMA, 2..9 epilogue, 10 K/V
constexpr int kThreadsKvo = 32 * kWarpsKvo;
// TMEM columns: score buffer t (S fp32, then P bf16 pairs over its first 32 columns) at 64 t;
// O buffer t at 128 + 128 t
constexpr int kColS = 64, kColO0 = 128, kColOStride = 128;

template <int D_H>
struct KvoSmem {
  static constexpr int kHalves = D_H / 64;
  static constexpr int kQHalf = kRowsT * 128;     // 128 rows x 64 dims, SW128
  static constexpr int kKHalf = 64 * 128;         // 64 keys x 64 dims, SW128
  static constexpr int kQStage = kHalves * kQHalf;
  static constexpr int kQStages = D_H == 128 ? 3 : 6;
  static constexpr int kKVStage = 2 * kHalves * kKHalf;   // K halves, then V halves
  static constexpr int kKVStages = 2;
  static constexpr int kOffQ = 0;
  static constexpr int kOffKV = kOffQ + kQStages * kQStage;
  // per epilogue group: the tile's partials in the layout of a Q stage (entry e's G = 8 rows of
  // a 64-dim half are one 1-KB swizzle atom), stored to global memory by TMA
  static constexpr int kOffOut = kOffKV + kKVStages * kKVStage;
  static constexpr int kOutBytes = kQStage;
  static constexpr int kOffBar = kOffOut + 2 * kOutBytes;
  // q_full, q_empty [kQStages]; kv_full, kv_empty [2]; s_full, p_full, sp_free, o_full,
  // o_empty [2]; done
  static constexpr int kNumBars = 2 * kQStages + 2 * kKVStages + 10 + 1;
  static constexpr int kOffMisc = kOffBar + 8 * kNumBars;
  static constexpr int kOffPEnt = kOffMisc + 16;  // the cp.async query warp's copy of the entries
  static constexpr int kBytes = kOffPEnt + 4 * kRowsT;
  // more than half of the SM's shared memory: one CTA per SM (it holds all 512 TMEM columns)
  static constexpr int kAlloc = kBytes + 1024 > 116 * 1024 ? kBytes + 1024 : 116 * 1024;
  static_assert(kQStage % 1024 == 0 && kKVStage % 1024 == 0, "swizzle atoms");
  static_assert(kAlloc <= 227 * 1024, "shared memory");
};

__device__ __forceinline__ void kvo_cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}

// Byte offset of row R's 128-byte line of 64-dim half `half` in a Q stage (and in the partials'
// staging, which has the same layout).  At G = 8 an entry's 8 head rows of both halves are two
// adjacent 1-KB swizzle atoms, so one TMA box moves the entry; otherwise each half is a
// [128 rows x 64 dims] block.  q_line(8, 0) is the stride between 8-row atoms (the UMMA SBO).
template <int G, int D_H>
__device__ __forceinline__ constexpr uint32_t q_line(int R, int half) {
  return G == 8 ? (uint32_t)((R >> 3) * 1024 * (D_H / 64) + half * 1024 + (R & 7) * 128)
                : (uint32_t)(half * kRowsT * 128 + R * 128);
}

__device__ __forceinline__ float rowmax64(const uint32_t* v) {
  float m0 = fmax3(__uint_as_float(v[0]), __uint_as_float(v[1]), __uint_as_float(v[2]));
  float m1 = fmax3(__uint_as_float(v[3]), __uint_as_float(v[4]), __uint_as_float(v[5]));
#pragma unroll
  for (int c = 6; c < 62; c += 4) {
    m0 = fmax3(m0, __uint_as_float(v[c]), __uint_as_float(v[c + 1]));
    m1 = fmax3(m1, __uint_as_float(v[c + 2]), __uint_as_float(v[c + 3]));
  }
  return fmax3(m0, m1, fmaxf(__uint_as_float(v[62]), __uint_as_float(v[63])));
}

// Barrier of one epilogue group (four warps, 128 threads) that ANDs a flag over the group: the
// only place where a group leaves its loop, so its four warps leave together.
__device__ __forceinline__ bool kvo_group_and(int id, bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\tbar.red.and.pred q, %2, 128, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)v), "r"(id)
      : "memory");
  return r != 0;
}

// The work tiles of this CTA in order: for each KV group r, the group's tiles (tile_off[r*nblk]
// .. tile_off[(r+1)*nblk]) split into gridDim.x contiguous ranges, this CTA taking range
// blockIdx.x.  next() also tracks each tile's bucket: binary search at the start of a range,
// then a cursor that only moves forward.
struct TileWalk {
  const int* __restrict__ tile_off;
  int nblk, H_kv, r, t, t_end, bkt, nxt;

  __device__ __forceinline__ void init(const int* to, int nb, int hkv) {
    tile_off = to;
    nblk = nb;
    H_kv = hkv;
    r = -1;
    t = t_end = bkt = nxt = 0;
  }
  __device__ __forceinline__ bool next(int& tile, int& bucket) {
    while (t >= t_end) {
      if (++r >= H_kv) return false;
      const int gs = __ldg(tile_off + r * nblk), ge = __ldg(tile_off + (r + 1) * nblk);
      const int per = (ge - gs + (int)gridDim.x - 1) / (int)gridDim.x;
      t = gs + (int)blockIdx.x * per;
      t_end = min(ge, t + per);
      if (t < t_end) {
        int lo = r * nblk, hi = (r + 1) * nblk;           // tile_off[lo] <= t < tile_off[hi]
        while (hi - lo > 1) {
          const int mid = (lo + hi) >> 1;
          if (__ldg(tile_off + mid) <= t) lo = mid; else hi = mid;
        }
        bkt = lo;
        nxt = __ldg(tile_off + bkt + 1);
      }
    }
    while (nxt <= t) {
      ++bkt;
      nxt = __ldg(tile_off + bkt + 1);
    }
    tile = t++;
    bucket = bkt;
    return true;
  }
};

template <int D_H, int G>
__global__ void __launch_bounds__(kThreadsKvo, 1)
    k_attn_kvouter(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_p,
                   const __nv_bfloat16* __restrict__ q,
                   const int* __restrict__ entries, const int* __restrict__ offset,
                   const int* __restrict__ tile_off, int nblk, int64_t N, int64_t q0, int64_t nq,
                   int H_kv, int kk, __nv_bfloat16* __restrict__ part_o,
                   float* __restrict__ part_lse, float scale_log2) {
  using L = KvoSmem<D_H>;
  constexpr int kEpt = kRowsT / G;                 // entries per work tile
  constexpr int kQStages = L::kQStages;
  constexpr int kChunks = D_H / 8;                 // 16-byte chunks per query row
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t sb = smem_u32(smem);
  const uint32_t bar0 = sb + L::kOffBar;
  auto q_full = [&](int s) { return bar0 + 8u * s; };
  auto q_empty = [&](int s) { return bar0 + 8u * (kQStages + s); };
  auto kv_full = [&](int s) { return bar0 + 8u * (2 * kQStages + s); };
  auto kv_empty = [&](int s) { return bar0 + 8u * (2 * kQStages + 2 + s); };
  auto s_full = [&](int t) { return bar0 + 8u * (2 * kQStages + 4 + t); };
  auto p_full = [&](int t) { return bar0 + 8u * (2 * kQStages + 6 + t); };
  auto sp_free = [&](int t) { return bar0 + 8u * (2 * kQStages + 8 + t); };
  auto o_full = [&](int t) { return bar0 + 8u * (2 * kQStages + 10 + t); };
  auto o_empty = [&](int t) { return bar0 + 8u * (2 * kQStages + 12 + t); };
  const uint32_t done = bar0 + 8u * (2 * kQStages + 14);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kOffMisc);
  volatile int* s_abort = reinterpret_cast<volatile int*>(smem + L::kOffMisc + 4);
  int* s_pent = reinterpret_cast<int*>(smem + L::kOffPEnt);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int H_q = H_kv * G;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kQStages; ++s) {
      // G = 8: lane 0's arrive with the TMA transaction bytes; otherwise the 32 lanes' cp.async
      // arrivals
      mbar_init(q_full(s), G == 8 ? 1 : 32);
      mbar_init(q_empty(s), 1);                  // MMA commit after S
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(kv_full(s), 1);                  // expect_tx + TMA
      mbar_init(kv_empty(s), 1);                 // MMA commit after the bucket's last O
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(s_full(t), 1);                   // MMA commit after S
      mbar_init(p_full(t), 4);                   // one arrive per epilogue warp
      mbar_init(sp_free(t), 1);                  // MMA commit after the O that read P
      mbar_init(o_full(t), 1);                   // MMA commit after O
      mbar_init(o_empty(t), 4);                  // one arrive per epilogue warp
    }
    mbar_init(done, 1);
    *s_abort = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tc_fence_before();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  auto fail = [&]() { *s_abort = 1; };

  if (warp == 0) {
    // ------------------------------------------------------------- query rows
    // The next tile's bucket, entry range and (lane e) entry are fetched while the current one's
    // copies are issued, so the dependent index loads stay off the issue path.
    TileWalk w;
    w.init(tile_off, nblk, H_kv);
    int j = 0, tile, b;
    int nb_ = 0, ne0 = 0, nne = 0, nent = 0;
    bool have = w.next(tile, b);
    auto fetch = [&](int t_, int b_) {
      nb_ = b_;
      ne0 = __ldg(offset + b_) + (t_ - __ldg(tile_off + b_)) * kEpt;
      nne = min(kEpt, __ldg(offset + b_ + 1) - ne0);
      nent = lane < nne ? __ldg(entries + ne0 + lane) : 0;
    };
    if (have) fetch(tile, b);
    while (have) {
      if (__any_sync(0xffffffffu, *s_abort != 0)) break;   // warp-uniform exits only
      const int cb = nb_, e0 = ne0, n_e = nne, my_ent = nent;
      have = w.next(tile, b);
      if (have) fetch(tile, b);                             // lands while this tile is issued
      const int rb = cb / nblk;
      const int s = j % kQStages;
      if (!__all_sync(0xffffffffu,
                      mbar_wait(q_empty(s), ((j / kQStages) & 1) ^ 1, &g_kvo_status))) {
        fail();
        break;
      }
      const uint32_t qbase = sb + L::kOffQ + s * L::kQStage;
      if (G == 8) {
        // entry e's G = 8 head rows are one 1-KB swizzle atom per 64-dim half: lane e issues
        // its entry's boxes
        if (lane == 0) mbar_expect_tx(q_full(s), (uint32_t)(n_e * 8 * 128 * L::kHalves));
        __syncwarp();
        if (lane < n_e) {
          const int i = (int)(q0 + (my_ent >> 6));
          // one box: the entry's 8 head rows of both 64-dim halves, as two adjacent atoms
          tma_load_4d(qbase + lane * 1024 * L::kHalves, &tm_q, q_full(s), 0, rb * 8, 0, i);
        }
      } else {
        __syncwarp();                                       // the previous tile's reads are done
        for (int x = lane; x < n_e; x += 32) s_pent[x] = __ldg(entries + e0 + x);
        __syncwarp();
        for (int x = lane; x < n_e * G * kChunks; x += 32) {
          const int R = x / kChunks, c = x - R * kChunks;
          const int e = R / G, h = R - e * G;
          const int64_t i = q0 + (s_pent[e] >> 6);
          const uint32_t off = q_line<G, D_H>(R, c >> 3) + (((c & 7) ^ (R & 7)) << 4);
          kvo_cp_async16(qbase + off, q + (i * H_q + (int64_t)rb * G + h) * D_H + c * 8);
        }
        asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(q_full(s))
                     : "memory");
      }
      ++j;
    }
    if (G != 8) asm volatile("cp.async.wait_all;" ::: "memory");
    // never leave with a copy in flight: the last stages' copies have landed
    for (int x = max(0, j - kQStages); x < j; ++x)
      mbar_wait(q_full(x % kQStages), (x / kQStages) & 1, &g_kvo_status);
  } else if (warp == 10) {
    // -------------------------------------------------------------- K_b and V_b
    if (lane == 0) {
      TileWalk w;
      w.init(tile_off, nblk, H_kv);
      int last = -1, kfill = 0, tile, b;
      prefetch_tensormap(&tm_k);
      prefetch_tensormap(&tm_v);
      while (w.next(tile, b)) {
        if (*s_abort) break;
        if (b == last) continue;
        const int ks = kfill & 1;
        if (!mbar_wait(kv_empty(ks), ((kfill >> 1) & 1) ^ 1, &g_kvo_status)) {
          fail();
          break;
        }
        const int rb = b / nblk;
        const int tok = (b - rb * nblk) * kBlock;
        const uint32_t dst = sb + L::kOffKV + ks * L::kKVStage;
        mbar_expect_tx(kv_full(ks), (uint32_t)L::kKVStage);
#pragma unroll
        for (int bx = 0; bx < L::kHalves; ++bx) {
          tma_load_3d(dst + bx * L::kKHalf, &tm_k, kv_full(ks), 64 * bx, rb, tok);
          tma_load_3d(dst + (L::kHalves + bx) * L::kKHalf, &tm_v, kv_full(ks), 64 * bx, rb, tok);
        }
        last = b;
        ++kfill;
      }
      for (int f = max(0, kfill - 2); f < kfill; ++f)
        mbar_wait(kv_full(f & 1), (f >> 1) & 1, &g_kvo_status);
    }
  } else if (warp == 1) {
    // --------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_s = umma_idesc_bf16(kRowsT, 64);
      constexpr uint32_t idesc_o = umma_idesc_bf16(kRowsT, D_H) | (1u << 16);   // B MN-major
      TileWalk w;
      w.init(tile_off, nblk, H_kv);
      // O of tile jj into O buffer jj & 1, from its P (score buffer jj & 1) and V_b of K/V stage
      // kvs; the score buffer is free once this MMA completes
      auto issue_o = [&](int jj, int kvs) -> bool {
        const int t = jj & 1;
        if (!mbar_wait(p_full(t), (jj >> 1) & 1, &g_kvo_status)) return false;
        if (!mbar_wait(o_empty(t), ((jj >> 1) & 1) ^ 1, &g_kvo_status)) return false;
        tc_fence_after();
        const uint32_t vb = sb + L::kOffKV + kvs * L::kKVStage + L::kHalves * L::kKHalf;
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)                     // 64 keys, 16 per step
          umma_bf16_ta(tmem + kColO0 + kColOStride * t, tmem + kColS * t + 8 * ks,
                       desc_mn_sw128(vb + ks * 2048, L::kKHalf, 1024), idesc_o, ks > 0 ? 1u : 0u);
        umma_commit(o_full(t));
        umma_commit(sp_free(t));
        return true;
      };
      int j = 0, kfill = -1, last = -1, prev_kvs = 0, tile, b;
      bool ok = true;
      while (w.next(tile, b)) {
        if (*s_abort) { ok = false; break; }
        if (b != last) {
          ++kfill;
          if (!mbar_wait(kv_full(kfill & 1), (kfill >> 1) & 1, &g_kvo_status)) { ok = false; break; }
          last = b;
        }
        const int kvs = kfill & 1;
        const int s = j % kQStages, t = j & 1;
        if (!mbar_wait(q_full(s), (j / kQStages) & 1, &g_kvo_status)) { ok = false; break; }
        if (!mbar_wait(sp_free(t), ((j >> 1) & 1) ^ 1, &g_kvo_status)) { ok = false; break; }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");   // cp.async rows -> MMA
        tc_fence_after();
        const uint32_t qbase = sb + L::kOffQ + s * L::kQStage;
        const uint32_t kbase = sb + L::kOffKV + kvs * L::kKVStage;
        const uint32_t d = tmem + (uint32_t)(kColS * t);
#pragma unroll
        for (int ks = 0; ks < D_H / 16; ++ks) {
          const uint32_t a = qbase + q_line<G, D_H>(0, ks >> 2) + (ks & 3) * 32;
          const uint32_t bk = kbase + (ks >> 2) * L::kKHalf + (ks & 3) * 32;
          umma_bf16(d, umma_desc_kmajor(a, q_line<G, D_H>(8, 0), 128),
                    umma_desc_kmajor(bk, 1024, 128), idesc_s, ks > 0 ? 1u : 0u);
        }
        umma_commit(s_full(t));
        umma_commit(q_empty(s));                 // P goes to TMEM: the Q stage is free after S
        if (j > 0) {
          if (!issue_o(j - 1, prev_kvs)) { ok = false; break; }
          if (prev_kvs != kvs) umma_commit(kv_empty(prev_kvs));   // the old bucket's last MMA
        }
        prev_kvs = kvs;
        ++j;
      }
      if (ok && j > 0 && !issue_o(j - 1, prev_kvs)) ok = false;
      if (!ok) fail();
      umma_commit(done);                         // every MMA issued has completed
      mbar_wait(done, 0, &g_kvo_status);
    }
  } else {
    // ------------------------------------------------------------ epilogue groups
    const int grp = (warp - 2) >> 2;             // 0: even tiles, 1: odd tiles
    const int qd = warp & 3;                     // TMEM lane quarter of this warp
    const int R = 32 * qd + lane;                // row (TMEM lane) of this thread
    const int e = R / G, h = R - e * G;
    const uint32_t lanes = (uint32_t)(32 * qd) << 16;
    const uint32_t ts = tmem + lanes + (uint32_t)(kColS * grp);                 // S, then P
    const uint32_t to = tmem + lanes + (uint32_t)(kColO0 + kColOStride * grp);  // O
    TileWalk w;
    w.init(tile_off, nblk, H_kv);
    // this group's next tile (sequence index jn), with its bucket, entry count and this row's
    // entry fetched one tile ahead
    int jn = -1, nb_ = 0, ne0 = 0, nne = 0, nent = 0;
    auto advance = [&]() -> bool {
      int tile, b;
      do {
        if (!w.next(tile, b)) return false;
        ++jn;
      } while ((jn & 1) != grp);
      nb_ = b;
      ne0 = __ldg(offset + b) + (tile - __ldg(tile_off + b)) * kEpt;
      nne = min(kEpt, __ldg(offset + b + 1) - ne0);
      nent = R < nne * G ? __ldg(entries + ne0 + e) : 0;
      return true;
    };
    bool have = advance();
    while (have) {
      const int use = jn >> 1;
      const int b = nb_, ent = nent, e0_cur = ne0, n_cur = nne;
      const bool rv = R < nne * G;
      have = advance();                          // the next tile's indices, under this one
      const int r = b / nblk;
      const int64_t blk = b - (int64_t)r * nblk;
      const bool okw = *s_abort == 0 && mbar_wait(s_full(grp), use & 1, &g_kvo_status);
      if (!kvo_group_and(1 + grp, okw)) { fail(); break; }
      tc_fence_after();
      // ---- softmax of this row over the block's visible keys; P (bf16) over S's first columns
      const int64_t i = q0 + (ent >> 6);
      float mx = 0.f, l = 0.f;
      {
        uint32_t sv[64];
        float lmx;                               // the load's maximum over the 64 keys
        MSA_TMEM_LDMAX64(ts, sv, lmx);
        tmem_ld_wait();
        if (rv) {
          if (blk == (i >> 6)) {                 // local block: keys j <= i only
            const int lim = (int)(i - blk * kBlock);
#pragma unroll
            for (int c = 0; c < 64; ++c)
              if (c > lim) sv[c] = __float_as_uint(-INFINITY);
            lmx = rowmax64(sv);
          }
          mx = lmx * scale_log2;
        }
        uint32_t pk[32];
        float l0 = 0.f, l1 = 0.f;
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          float x0, x1;
          ffma2(x0, x1, __uint_as_float(sv[2 * c]), __uint_as_float(sv[2 * c + 1]), scale_log2,
                scale_log2, -mx, -mx);
          const float p0 = rv ? ex2(x0) : 0.f;
          const float p1 = rv ? ex2(x1) : 0.f;
          fadd2(l0, l1, l0, l1, p0, p1);
          pk[c] = pack_bf16x2(p0, p1);
        }
        l = l0 + l1;
        MSA_TMEM_ST32(ts, pk);
        tmem_st_wait();
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(p_full(grp));
      // ---- O of this row, normalised by its own sum: the partial (bf16) and its log2 LSE
      const bool oko = mbar_wait(o_full(grp), use & 1, &g_kvo_status);
      if (!kvo_group_and(1 + grp, oko)) { fail(); break; }
      tc_fence_after();
      const int64_t slot_pos = ((int64_t)r * nq + (ent >> 6)) * kk + (ent & 63);
      const float inv = l > 0.f ? 1.f / l : 0.f;
      const uint32_t out = sb + L::kOffOut + grp * L::kOutBytes;
#pragma unroll
      for (int half = 0; half < D_H / 64; ++half) {
        uint32_t o[64];
        MSA_TMEM_LD64(to + 64 * half, o);
        tmem_ld_wait();
        if (half == D_H / 64 - 1) {              // O is in registers: the buffer may be reused
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(o_empty(grp));
        }
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          uint4 v;
          v.x = pack_bf16x2(__uint_as_float(o[8 * c + 0]) * inv, __uint_as_float(o[8 * c + 1]) * inv);
          v.y = pack_bf16x2(__uint_as_float(o[8 * c + 2]) * inv, __uint_as_float(o[8 * c + 3]) * inv);
          v.z = pack_bf16x2(__uint_as_float(o[8 * c + 4]) * inv, __uint_as_float(o[8 * c + 5]) * inv);
          v.w = pack_bf16x2(__uint_as_float(o[8 * c + 6]) * inv, __uint_as_float(o[8 * c + 7]) * inv);
          if (G == 8) {
            // row R's 16-byte chunk c of this half, at its place in the 128-byte swizzle
            asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(
                             out + q_line<G, D_H>(R, half) + ((c ^ (R & 7)) << 4)),
                         "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                         : "memory");
          } else if (rv) {
            reinterpret_cast<uint4*>(part_o + (slot_pos * G + h) * D_H + 64 * half)[c] = v;
          }
        }
      }
      if (rv) part_lse[slot_pos * G + h] = mx + __log2f(l);
      if (G == 8) {
        // the group's rows are staged: one thread stores each entry (all its halves) by TMA
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        asm volatile("bar.sync %0, 128;" ::"r"(3 + grp) : "memory");
        if (qd == 2 && lane == 0) {
          for (int x = 0; x < n_cur; ++x) {
            const int ex = __ldg(entries + e0_cur + x);
            const int zs = (int)(((int64_t)r * nq + (ex >> 6)) * kk + (ex & 63));
            tma_store_4d(&tm_p, out + x * 1024 * L::kHalves, 0, 0, 0, zs);
          }
          bulk_commit();
          bulk_wait_read_all();                  // the staging buffer is free for the next tile
        }
      }
    }
    if (G == 8 && qd == 2 && lane == 0) bulk_wait_all();   // stores complete before exit
  }

  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace

cudaError_t launch_attn_kvouter(const void* q, const void* k, const void* v, const int* entries,
                                const int* offset, const int* tile_off, int nbuckets, int64_t nblk,
                                int64_t N, int64_t q0, int64_t q1, int H_q, int H_kv, int d_h,
                                int kk, int grid, void* part_o, float* part_lse,
                                cudaStream_t stream) {
  (void)nbuckets;
  const int G = H_q / H_kv;
  const float scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)d_h));
  // Q as [N, H_q, d_h]: one box = one query's G heads x 64 dims; K, V as [N, H_kv, d_h]: one box
  // = one group's 64 tokens x 64 dims; 128-byte swizzle
  // At G = 8 the query box is 4-D, [64 dims, 8 heads, d_h/64 halves, 1 token]: its two halves
  // land as two adjacent 1-KB atoms (the heads' stride is d_h elements, the halves' 64).
  CUtensorMap tq, tk, tv;
  const uint64_t qdims[4] = {64, (uint64_t)H_q, (uint64_t)d_h / 64, (uint64_t)N};
  const uint64_t qstr[3] = {(uint64_t)d_h * 2, 128, (uint64_t)H_q * d_h * 2};
  const int qbox[4] = {64, 8, d_h / 64, 1};
  cudaError_t e = G == 8 ? make_tma_4d_bf16(&tq, q, qdims, qstr, qbox, 128)
                         : make_tma_3d_bf16(&tq, q, (uint64_t)d_h, (uint64_t)H_q, (uint64_t)N, 64,
                                            G, 1, 128);
  if (e != cudaSuccess) return e;
  e = make_tma_3d_bf16(&tk, k, (uint64_t)d_h, (uint64_t)H_kv, (uint64_t)N, 64, 1, 64, 128);
  if (e != cudaSuccess) return e;
  e = make_tma_3d_bf16(&tv, v, (uint64_t)d_h, (uint64_t)H_kv, (uint64_t)N, 64, 1, 64, 128);
  if (e != cudaSuccess) return e;
  // the partials as [H_kv * chunk rows * k slots, G, d_h]: one box = one entry's G heads x 64 dims
  // (at G = 8 a 4-D box over [64 dims, 8 heads, d_h/64 halves, rows], one store per entry)
  CUtensorMap tp;
  const uint64_t prows = (uint64_t)H_kv * (uint64_t)(q1 - q0) * (uint64_t)kk;
  const uint64_t pdims[4] = {64, 8, (uint64_t)d_h / 64, prows};
  const uint64_t pstr[3] = {(uint64_t)d_h * 2, 128, (uint64_t)8 * d_h * 2};
  const int pbox[4] = {64, 8, d_h / 64, 1};
  e = G == 8 ? make_tma_4d_bf16(&tp, part_o, pdims, pstr, pbox, 128)
             : make_tma_3d_bf16(&tp, part_o, (uint64_t)d_h, (uint64_t)G, prows, 64, G, 1, 128);
  if (e != cudaSuccess) return e;
  const auto* qq = static_cast<const __nv_bfloat16*>(q);
  auto* po = static_cast<__nv_bfloat16*>(part_o);
  auto run = [&](auto kern, int smem) -> cudaError_t {
    cudaError_t x = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (x != cudaSuccess) return x;
    kern<<<grid, kThreadsKvo, smem, stream>>>(tq, tk, tv, tp, qq, entries, offset, tile_off, (int)nblk,
                                               N, q0, q1 - q0, H_kv, kk, po, part_lse, scale_log2);
    return cudaGetLastError();
  };
  auto dispatch = [&](auto dh) -> cudaError_t {
    constexpr int D = decltype(dh)::value;
    constexpr int S = KvoSmem<D>::kAlloc;
    switch (G) {
      case 1: return run(k_attn_kvouter<D, 1>, S);
      case 2: return run(k_attn_kvouter<D, 2>, S);
      case 4: return run(k_attn_kvouter<D, 4>, S);
      default: return run(k_attn_kvouter<D, 8>, S);
    }
  };
  return d_h == 128 ? dispatch(std::integral_constant<int, 128>())
                    : dispatch(std::integral_constant<int, 64>());
}

cudaError_t read_reset_kvo_status(unsigned* out) {
  unsigned zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(out, g_kvo_status, sizeof(unsigned));
  if (e != cudaSuccess) return e;
  return cudaMemcpyToSymbol(g_kvo_status, &zero, sizeof(unsigned));
}

}  // namespace msa

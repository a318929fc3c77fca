// Shared-block pass of the sparse main branch («MiniMax-M3：MSA 技术报告速读», section 主分支,
// eq. O^(h)_i; LSE from section Kernel): the KV blocks that at least kSharedMin (4) queries of a
// 16-query tile selected, processed once for the tile on the 5th-generation tensor cores.
//
// One CTA = one tile (16 consecutive queries of KV group r).  Its 16*G <= 128 (query, head)
// rows are the M side of every UMMA; they arrive by TMA (a 3-D map over [N, H_q, d_h]):
//   warp 0   loads the tile's shared blocks (recorded by the plan pass), then streams them
//            as 32-token half blocks (K and V, 3-D tensor maps over [N, H_kv, d_h], 128-byte
//            swizzle) through a 4-stage TMA ring;
//   warp 1   allocates TMEM and issues  S[b] = Q K^T  (M=128, N=32) and  O += P V  (M=128,
//            N=d_h, P read from TMEM, V as an MN-major operand); S is triple- and P
//            double-buffered, so QK^T runs two half blocks ahead of the softmax;
//   warps 2-9 two per TMEM lane quarter, one row per thread: warp half ch takes keys
//            [16 ch, 16 ch + 16) of every half block and columns [ch d_h/2, (ch+1) d_h/2) of O;
//            they read S (each warp its own 16 keys and the other half's maximum, so the pair
//            needs no exchange), mask queries that did not select the block and keys after the
//            query, and write P (bf16) back to TMEM; then all ten warps run the epilogue.
// Online softmax with a lazily moved reference max: a row's reference m moves only when a block
// max exceeds it by more than 2^8, so P <= 2^8 and O (in TMEM) is rescaled only then.  The
// result is exact either way -- O/l and m + log2 l use the same reference.
// The epilogue finishes each row: it combines the row's shared-block state (O in TMEM, fp32)
// with the row's private-block partials written by the block-major pass (k_attn_kvouter.cu, run
// before this kernel) at the row's own slot positions, in slot order, and writes O (bf16) and
// the natural-log LSE.
// Every wait is bounded; a timeout sets the device status word and the roles stop.
#include <climits>
#include <cmath>

#include "attn_tile.cuh"
#include "msa_internal.h"

namespace msa {
namespace {

__device__ unsigned g_shared_status = 0;

constexpr int kRing = 4;                 // half-block stages
constexpr int kSBufs = 3;                // S buffers in TMEM: QK^T runs two half blocks ahead
constexpr int kHalfTok = 32;             // tokens per stage
constexpr int kShThreads = 320;          // producer, MMA, 8 softmax/epilogue warps (2 per quarter)

template <int D_H>
struct ShSmem {
  static constexpr int kHalves = D_H / 64;
  static constexpr int kQHalf = 128 * 128;          // 128 rows x 64 dims
  static constexpr int kBox = kHalfTok * 128;       // 32 tokens x 64 dims
  static constexpr int kKBytes = kHalves * kBox;
  static constexpr int kStage = 2 * kKBytes;        // K boxes, then V boxes
  static constexpr int kOffQ = 0;
  static constexpr int kOffRing = kOffQ + kHalves * kQHalf;
  static constexpr int kOffList = kOffRing + kRing * kStage;
  static constexpr int kOffBar = kOffList + kMaxShared * 4;
  // kv_full[kRing], kv_empty[kRing], s_full[kSBufs], s_free[kSBufs], p_full[2], p_free[2],
  // q_ready, done
  static constexpr int kNumBars = 2 * kRing + 2 * kSBufs + 6;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;
  static constexpr int kOffPriv = kOffMisc + 16;    // per query: its private slots (bit t)
  // the two softmax warps of a lane quarter exchange per-row values: the halves of the row
  // sum, the O weight
  static constexpr int kOffLh = kOffPriv + kTileQ * 8;
  static constexpr int kOffCo = kOffLh + 2 * 128 * 4;
  static constexpr int kBytes = kOffCo + 128 * 4;
  static constexpr int kAlloc = kBytes + 1024;
  // TMEM columns: S[b] 32b..32b+31 for b < 3 (fp32); P[0] 96..111, P[1] 112..127 (bf16
  // pairs); O 128..128+d_h (fp32)
  static constexpr uint32_t kTmemCols = 256;
  static constexpr uint32_t kColP = 32 * kSBufs, kColO = 128;
  static_assert(kColP + 32 <= kColO, "S and P buffers below O");
  // epilogue, over Q / ring once every MMA has completed: the rows' shared-block O (fp32,
  // already weighted), per-row max and 1/sum of the merge, per query its private partials
  static constexpr int kOsStride = D_H + 4;          // floats; 16-byte pad against conflicts
  static constexpr int kOffOs = 0;
  static constexpr int kOffMx = kOffOs + 128 * kOsStride * 4;
  static constexpr int kOffInv = kOffMx + 128 * 4;
  static constexpr int kOffPos = kOffInv + 128 * 4;
  static constexpr int kOffNp = kOffPos + kTileQ * kMaxSel * 4;
  static_assert(kOffNp + kTileQ * 4 <= kOffList, "epilogue staging fits below the block list");
};

// Named barrier of the two softmax warps of one TMEM lane quarter (64 threads); the reducing
// form returns the AND of every thread's flag, so both warps take the same branch after it.
__device__ __forceinline__ bool pair_and(int id, bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\t"
      "bar.red.and.pred q, %2, 64, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)v), "r"(id)
      : "memory");
  return r != 0;
}
__device__ __forceinline__ void pair_sync(int id) {
  asm volatile("bar.sync %0, 64;" ::"r"(id) : "memory");
}

__device__ __forceinline__ void prefetch_l2_bulk(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}
__device__ __forceinline__ void prefetch_l2(const void* p) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(p) : "memory");
}
__device__ __forceinline__ float ldg_nc_f32(const float* p) {
  float v;
  asm volatile("ld.global.nc.f32 %0, [%1];" : "=f"(v) : "l"(p));
  return v;
}

template <int D_H>
__global__ void __launch_bounds__(kShThreads, 2)
    k_attn_shared(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v,
                  const __nv_bfloat16* __restrict__ q, const int* __restrict__ tile_list,
                  const unsigned long long* __restrict__ tile_priv,
                  const __nv_bfloat16* __restrict__ part_o,
                  const float* __restrict__ part_lse, __nv_bfloat16* __restrict__ o,
                  float* __restrict__ lse, int64_t N, int64_t q0, int64_t q1, int H_q, int G,
                  int kk, int64_t ntiles, float scale_log2) {
  using L = ShSmem<D_H>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t sb = smem_u32(smem);
  int* s_list = reinterpret_cast<int*>(smem + L::kOffList);
  int* s_nS = reinterpret_cast<int*>(smem + L::kOffMisc);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kOffMisc + 4);
  unsigned long long* s_priv = reinterpret_cast<unsigned long long*>(smem + L::kOffPriv);
  const uint32_t bar = sb + L::kOffBar;
  auto kv_full = [&](int s) { return bar + 8u * s; };
  auto kv_empty = [&](int s) { return bar + 8u * (kRing + s); };
  auto s_full = [&](int b) { return bar + 8u * (2 * kRing + b); };
  auto s_free = [&](int b) { return bar + 8u * (2 * kRing + kSBufs + b); };
  auto p_full = [&](int b) { return bar + 8u * (2 * kRing + 2 * kSBufs + b); };
  auto p_free = [&](int b) { return bar + 8u * (2 * kRing + 2 * kSBufs + 2 + b); };
  const uint32_t q_ready = bar + 8u * (2 * kRing + 2 * kSBufs + 4);
  const uint32_t done = bar + 8u * (2 * kRing + 2 * kSBufs + 5);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t bid = blockIdx.x;
  const int r = (int)(bid / ntiles);
  const int64_t i0 = q0 + (bid - (int64_t)r * ntiles) * kTileQ;
  const int rows = kTileQ * G;                       // 16 G <= 128 rows in use

  if (warp == 0) {
    // the tile's shared blocks (block << 16 | query mask) and its queries' private slots
    const int* lst = tile_list + bid * (kMaxShared + 1);
    const int nS = __ldg(lst);
    for (int x = lane; x < nS; x += 32) s_list[x] = __ldg(lst + 1 + x);
    if (lane < kTileQ) s_priv[lane] = __ldg(tile_priv + bid * kTileQ + lane);
    if (lane == 0) {
      *s_nS = nS;
      for (int s = 0; s < kRing; ++s) {
        mbar_init(kv_full(s), 1);
        mbar_init(kv_empty(s), 1);
      }
      for (int b = 0; b < kSBufs; ++b) {
        mbar_init(s_full(b), 1);
        mbar_init(s_free(b), 8);
      }
      for (int b = 0; b < 2; ++b) {
        mbar_init(p_full(b), 8);
        mbar_init(p_free(b), 1);
      }
      mbar_init(q_ready, 1);
      mbar_init(done, 1);
      fence_barrier_init();
    }
  } else if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), L::kTmemCols);
    tc_fence_before();
  }
  __syncthreads();
  tc_fence_after();
  const int nS = *s_nS;
  const int nH = 2 * nS;                              // half blocks
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------------ producer
    if (lane == 0) {
      // the tile's Q rows (row R = query w * G + head h): one box of G heads x 16 queries per
      // 64-dim half, 128-byte swizzle
      prefetch_tensormap(&tm_q);
      mbar_expect_tx(q_ready, (uint32_t)(L::kHalves * rows * 128));
#pragma unroll
      for (int bx = 0; bx < L::kHalves; ++bx)
        tma_load_3d(sb + L::kOffQ + bx * L::kQHalf, &tm_q, q_ready, 64 * bx, r * G, (int)i0);
      prefetch_tensormap(&tm_k);
      prefetch_tensormap(&tm_v);
      int last[kRing];
      for (int s = 0; s < kRing; ++s) last[s] = -1;
      for (int hb = 0; hb < nH; ++hb) {
        const int s = hb % kRing, round = hb / kRing;
        if (!mbar_wait(kv_empty(s), (round & 1) ^ 1, &g_shared_status)) break;
        const int tok = (s_list[hb >> 1] >> 16) * kBlock + (hb & 1) * kHalfTok;
        const uint32_t dst = sb + L::kOffRing + s * L::kStage;
        mbar_expect_tx(kv_full(s), L::kStage);
#pragma unroll
        for (int bx = 0; bx < L::kHalves; ++bx) {
          tma_load_3d(dst + bx * L::kBox, &tm_k, kv_full(s), 64 * bx, r, tok);
          tma_load_3d(dst + L::kKBytes + bx * L::kBox, &tm_v, kv_full(s), 64 * bx, r, tok);
        }
        last[s] = round;
      }
      for (int s = 0; s < kRing; ++s)
        if (last[s] >= 0) mbar_wait(kv_full(s), last[s] & 1, &g_shared_status);
      mbar_wait(q_ready, 0, &g_shared_status);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_s = umma_idesc_bf16(128, kHalfTok);
      constexpr uint32_t idesc_o = umma_idesc_bf16(128, D_H) | (1u << 16);   // B MN-major
      bool ok = mbar_wait(q_ready, 0, &g_shared_status);
      auto issue_s = [&](int hb) -> bool {
        const int s = hb % kRing, b = hb % kSBufs;
        if (!mbar_wait(kv_full(s), (hb / kRing) & 1, &g_shared_status)) return false;
        if (!mbar_wait(s_free(b), ((hb / kSBufs) & 1) ^ 1, &g_shared_status)) return false;
        tc_fence_after();
        const uint32_t kbase = sb + L::kOffRing + s * L::kStage;
#pragma unroll
        for (int ks = 0; ks < D_H / 16; ++ks)
          umma_bf16(tmem + 32 * b,
                    umma_desc_kmajor(sb + L::kOffQ + (ks >> 2) * L::kQHalf + (ks & 3) * 32, 1024, 128),
                    umma_desc_kmajor(kbase + (ks >> 2) * L::kBox + (ks & 3) * 32, 1024, 128),
                    idesc_s, ks > 0 ? 1u : 0u);
        umma_commit(s_full(b));
        return true;
      };
      if (ok && nH > 0) ok = issue_s(0);
      if (ok && nH > 1) ok = issue_s(1);
      for (int hb = 0; hb < nH && ok; ++hb) {
        if (hb + 2 < nH && !(ok = issue_s(hb + 2))) break;
        const int pb = hb & 1;
        if (!(ok = mbar_wait(p_full(pb), (hb >> 1) & 1, &g_shared_status))) break;
        tc_fence_after();
        const uint32_t vbase = sb + L::kOffRing + (hb % kRing) * L::kStage + L::kKBytes;
#pragma unroll
        for (int ks = 0; ks < kHalfTok / 16; ++ks)
          umma_bf16_ta(tmem + L::kColO, tmem + L::kColP + 16 * pb + 8 * ks,
                       desc_mn_sw128(vbase + ks * 2048, L::kBox, 1024), idesc_o,
                       (hb > 0 || ks > 0) ? 1u : 0u);
        umma_commit(p_free(pb));
        umma_commit(kv_empty(hb % kRing));
      }
      umma_commit(done);
      mbar_wait(done, 0, &g_shared_status);
    }
  } else {
    // ------------------------------------------------------ softmax and epilogue
    // warps 2..9, two per TMEM lane quarter: half ch takes keys [16 ch, 16 ch + 16) of every
    // half block and columns [ch d_h / 2, (ch + 1) d_h / 2) of O.  Both warps of a pair read
    // all 32 keys' maximum from TMEM (tcgen05.ld.red on each half), so they take the same
    // reference-max decisions without exchanging anything; they add their halves of the row sum
    // through shared memory at the end
    const int qd = warp & 3;                          // TMEM lane quarter
    const int ch = (warp - 2) >> 2;
    const int pair = 1 + qd;                          // named barrier id of the quarter's pair
    const int R = 32 * qd + lane;
    const int w = R / G, h = R - (R / G) * G;
    const int64_t i = i0 + w;
    const bool valid = R < rows && i < q1;
    const uint32_t lanes = (uint32_t)(32 * qd) << 16;
    float* s_lh = reinterpret_cast<float*>(smem + L::kOffLh);
    float* s_co = reinterpret_cast<float*>(smem + L::kOffCo);
    float m_ref = -INFINITY, l = 0.f;                 // l: this half's share of the row sum
    bool ok = true;
    // A warp leaves the loop at its own failed (bounded) wait; its partner then fails at one of
    // its next waits, and the pair agrees again at the epilogue's reducing barrier.
    for (int hb = 0; hb < nH; ++hb) {
      const int ent = s_list[hb >> 1];
      const int64_t b = ent >> 16;
      const bool sel = valid && ((ent >> w) & 1);
      const int buf = hb & 1, sbuf = hb % kSBufs;          // P buffer, S buffer
      const bool okw =
          ok && __all_sync(kAllLanes, mbar_wait(s_full(sbuf), (hb / kSBufs) & 1, &g_shared_status));
      uint32_t sv[16], so[16];                        // this half's keys; the other half's
      float pmx = -INFINITY, lmx, omx;                // pmx: the row max over all 32 keys
      if (okw) {
        tc_fence_after();
        MSA_TMEM_LDMAX16(tmem + lanes + 32 * sbuf + 16 * ch, sv, lmx);
        MSA_TMEM_LDMAX16(tmem + lanes + 32 * sbuf + 16 * (ch ^ 1), so, omx);
        tmem_ld_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(s_free(sbuf));
        if (sel) {
          if (b == (i >> 6)) {                        // local block: keys j <= i only
            const int lim = (int)(i - (b * kBlock + (hb & 1) * kHalfTok));
#pragma unroll
            for (int c = 0; c < 16; ++c) {
              if (16 * ch + c > lim) sv[c] = __float_as_uint(-INFINITY);
              if (16 * (ch ^ 1) + c > lim) so[c] = __float_as_uint(-INFINITY);
            }
            pmx = fmax3(__uint_as_float(sv[0]), __uint_as_float(so[0]), __uint_as_float(sv[1]));
#pragma unroll
            for (int c = 1; c < 15; ++c)
              pmx = fmax3(pmx, __uint_as_float(so[c]), __uint_as_float(sv[c + 1]));
            pmx = fmaxf(pmx, __uint_as_float(so[15]));
          } else {
            pmx = fmaxf(lmx, omx);                    // every key visible: the loads' maxima
          }
        }
      }
      ok = okw;
      if (!ok) break;
      float alpha = 1.f;
      uint32_t pk[8];
      if (sel) {
        const float bm = pmx * scale_log2;
        if (m_ref == -INFINITY) {
          m_ref = bm;                                 // this row's O and l are still zero
        } else if (bm > m_ref + 8.f) {
          alpha = ex2(m_ref - bm);
          m_ref = bm;
        }
        float ps0 = 0.f, ps1 = 0.f;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          float x0, x1;
          ffma2(x0, x1, __uint_as_float(sv[2 * c]), __uint_as_float(sv[2 * c + 1]), scale_log2,
                scale_log2, -m_ref, -m_ref);
          const float p0 = ex2(x0), p1 = ex2(x1);
          fadd2(ps0, ps1, ps0, ps1, p0, p1);
          pk[c] = pack_bf16x2(p0, p1);
        }
        l = l * alpha + (ps0 + ps1);
      } else {
#pragma unroll
        for (int c = 0; c < 8; ++c) pk[c] = 0u;
      }
      // P buffer hb&1 is free once O += P V of half block hb-2 has completed
      bool okp = true;
      if (hb > 1)
        okp = __all_sync(kAllLanes, mbar_wait(p_free(buf), ((hb >> 1) & 1) ^ 1, &g_shared_status));
      tc_fence_after();
      if (okp && __any_sync(kAllLanes, alpha != 1.f)) {
        // O itself may be rescaled only once O += P V of half block hb-1 (and so of every
        // earlier one) has completed: the (hb-1)/2-th phase of P buffer (hb-1)&1's "free"
        // barrier.  S of this half block was issued after O += P V of hb-3, so no later phase
        // of that barrier can be pending and the parity is unambiguous.  Both warps of the
        // pair decide alike (same rows, same maxima) and each rescales its half of O.
        if (hb > 0)
          okp = __all_sync(kAllLanes, mbar_wait(p_free((hb - 1) & 1), ((hb - 1) >> 1) & 1,
                                                &g_shared_status));
        tc_fence_after();
        if (okp) {
          uint32_t ov[D_H / 2];
          if constexpr (D_H == 128) {
            MSA_TMEM_LD64(tmem + lanes + L::kColO + 64 * ch, ov);
          } else {
            MSA_TMEM_LD32(tmem + lanes + L::kColO + 32 * ch, ov);
          }
          tmem_ld_wait();
#pragma unroll
          for (int c = 0; c < D_H / 2; ++c) ov[c] = __float_as_uint(__uint_as_float(ov[c]) * alpha);
          if constexpr (D_H == 128) {
            MSA_TMEM_ST64(tmem + lanes + L::kColO + 64 * ch, ov);
          } else {
            MSA_TMEM_ST32(tmem + lanes + L::kColO + 32 * ch, ov);
          }
        }
      }
      if (okp) {
        MSA_TMEM_ST8(tmem + lanes + L::kColP + 16 * buf + 8 * ch, pk);
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(p_full(buf));
      }
      ok = okp;
    }
    // ---- epilogue: shared-block state + private partials of each row, in slot order
    // the query's private partials start toward L2 now, while the last MMAs drain
    if (ch == 0 && valid && h == 0) {
      const unsigned long long pv = s_priv[w];
      const int64_t rp = ((int64_t)r * (q1 - q0) + (i - q0)) * kk;
      for (int t = 0; t < kk; ++t)
        if ((pv >> t) & 1ull) prefetch_l2_bulk(part_o + (rp + t) * G * D_H, (uint32_t)(G * D_H * 2));
      const float* lp = part_lse + rp * G;
      for (int x = 0; x < kk * G; x += 32) prefetch_l2(lp + x);
    }
    const bool okd = pair_and(
        pair, ok && __all_sync(kAllLanes, mbar_wait(done, 0, &g_shared_status)));
    tc_fence_after();
    const bool have_o = nH > 0 && okd;               // the same in both warps of the pair
    float* s_os = reinterpret_cast<float*>(smem + L::kOffOs);
    float* s_mx = reinterpret_cast<float*>(smem + L::kOffMx);
    float* s_inv = reinterpret_cast<float*>(smem + L::kOffInv);
    int* s_pos = reinterpret_cast<int*>(smem + L::kOffPos);
    int* s_np = reinterpret_cast<int*>(smem + L::kOffNp);
    s_lh[ch * 128 + R] = l;
    pair_sync(pair);
    const float lrow = s_lh[R] + s_lh[128 + R];      // the row sum over both halves
    if (ch == 0) {
      // (a) one thread per row: merge max and sum over the shared state and the private LSEs
      //     (online, 16 slots at a time); the query's head-0 row lists its private partials, which
      //     the block-major pass wrote at the row's own slot positions
      const unsigned long long priv = valid ? s_priv[w] : 0ull;
      const int64_t row_pos = ((int64_t)r * (q1 - q0) + (i - q0)) * kk;
      const float lse_s = lrow > 0.f ? m_ref + __log2f(lrow) : -INFINITY;
      float mx = lse_s, wsum = lse_s == -INFINITY ? 0.f : 1.f;
      int np = 0;
      for (int t0 = 0; t0 < kk; t0 += 16) {
        int pos[16];
        float lv[16];
#pragma unroll
        for (int d = 0; d < 16; ++d)
          pos[d] = (valid && t0 + d < kk && ((priv >> (t0 + d)) & 1ull)) ? (int)(row_pos + t0 + d) : -1;
#pragma unroll
        for (int d = 0; d < 16; ++d)
          lv[d] = pos[d] >= 0 ? __ldg(part_lse + (int64_t)pos[d] * G + h) : -INFINITY;
        float cm = mx;
#pragma unroll
        for (int d = 0; d < 16; ++d) cm = fmaxf(cm, lv[d]);
        if (cm != -INFINITY) {
          if (mx != -INFINITY) wsum *= ex2(mx - cm);
          mx = cm;
#pragma unroll
          for (int d = 0; d < 16; ++d)
            if (pos[d] >= 0) wsum += ex2(lv[d] - mx);
        }
        if (valid && h == 0) {
#pragma unroll
          for (int d = 0; d < 16; ++d)
            if (pos[d] >= 0) s_pos[w * kk + np++] = pos[d];
        }
      }
      const float inv_w = wsum > 0.f ? 1.f / wsum : 0.f;
      const float c_o = lrow > 0.f ? ex2(lse_s - mx) * inv_w / lrow : 0.f;
      if (valid) lse[((int64_t)r * G + h) * N + i] = (mx + __log2f(wsum)) * 0.69314718055994531f;
      s_mx[R] = mx;
      s_inv[R] = inv_w;
      if (valid && h == 0) s_np[w] = np;
      s_co[R] = c_o;
    }
    pair_sync(pair);
    // (b) this half of the row's shared-block O, weighted, into shared memory
    {
      const float c_o = s_co[R];
      uint32_t ov[D_H / 2];
      if (have_o) {
        if constexpr (D_H == 128) {
          MSA_TMEM_LD64(tmem + lanes + L::kColO + 64 * ch, ov);
        } else {
          MSA_TMEM_LD32(tmem + lanes + L::kColO + 32 * ch, ov);
        }
        tmem_ld_wait();
      }
      float4* dst = reinterpret_cast<float4*>(s_os + R * L::kOsStride + ch * (D_H / 2));
#pragma unroll
      for (int c = 0; c < D_H / 8; ++c)
        dst[c] = have_o ? make_float4(__uint_as_float(ov[4 * c]) * c_o,
                                      __uint_as_float(ov[4 * c + 1]) * c_o,
                                      __uint_as_float(ov[4 * c + 2]) * c_o,
                                      __uint_as_float(ov[4 * c + 3]) * c_o)
                        : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    tc_fence_before();
  }

  __syncthreads();                                    // (b) of every row is in shared memory
  // (c) every warp (the producer and MMA warps are idle by now) takes units of a query: a
  //     query's partial for all G heads is G*d_h contiguous bf16, as is its output row, split in
  //     16-byte pieces (coalesced) and in units of at most 64 pieces; lanes add the private
  //     partials to the staged shared-block O in slot order
  {
    const float* s_os = reinterpret_cast<const float*>(smem + L::kOffOs);
    const float* s_mx = reinterpret_cast<const float*>(smem + L::kOffMx);
    const float* s_inv = reinterpret_cast<const float*>(smem + L::kOffInv);
    const int* s_pos = reinterpret_cast<const int*>(smem + L::kOffPos);
    const int* s_np = reinterpret_cast<const int*>(smem + L::kOffNp);
    {
      const int U = G * D_H / 8;                      // 16-byte pieces per query
      const int UP = U > 64 ? 64 : U;                 // pieces per unit
      const int upq = U / UP;                         // units per query (1 or 2)
      const int lpu = UP < 32 ? UP : 32;              // lanes per unit
      const int upp = 32 / lpu, ipl = UP / lpu;       // units per pass, pieces per lane
      const int sub = lane % lpu;
      const int nunits = kTileQ * upq;
      const int npass = (nunits + upp - 1) / upp;
      constexpr int kWarps = kShThreads / 32;
      const int wslot = (warp + kWarps - 2) % kWarps;  // softmax warps first
      constexpr int kIpl = 2;                         // most pieces per lane
      constexpr int kNb = 4;                          // partials in flight per lane
      for (int ps = wslot; ps < npass; ps += kWarps) {
        const int unit = ps * upp + lane / lpu;
        const int wq = unit / upq, uh = unit - wq * upq;
        const bool qv = unit < nunits && i0 + wq < q1;
        float acc[kIpl][8], pm[kIpl], pi[kIpl];
        int pe[kIpl], ph[kIpl];
#pragma unroll
        for (int c = 0; c < kIpl; ++c) {
          pe[c] = 8 * (uh * UP + c * lpu + sub);      // element within the query's G*d_h
          ph[c] = pe[c] / D_H;
          const int RR = min(min(wq, kTileQ - 1) * G + ph[c], 127);
          pm[c] = s_mx[RR];
          pi[c] = s_inv[RR];
          const float4* src =
              reinterpret_cast<const float4*>(s_os + RR * L::kOsStride + (pe[c] - ph[c] * D_H));
          const float4 a0 = src[0], a1 = src[1];
          acc[c][0] = a0.x; acc[c][1] = a0.y; acc[c][2] = a0.z; acc[c][3] = a0.w;
          acc[c][4] = a1.x; acc[c][5] = a1.y; acc[c][6] = a1.z; acc[c][7] = a1.w;
        }
        const int npq = qv ? s_np[wq] : 0;
        for (int j = 0; j < npq; j += kNb) {
          int pos[kNb];
          uint4 u[kNb][kIpl];
          float lv[kNb][kIpl];
#pragma unroll
          for (int d = 0; d < kNb; ++d) pos[d] = j + d < npq ? s_pos[wq * kk + j + d] : -1;
          // every load of the batch is issued before any is used (ordered volatile loads)
#pragma unroll
          for (int d = 0; d < kNb; ++d)
#pragma unroll
            for (int c = 0; c < kIpl; ++c)
              if (pos[d] >= 0 && c < ipl) {
                u[d][c] = ldg_nc_v4(part_o + (int64_t)pos[d] * G * D_H + pe[c]);
                lv[d][c] = ldg_nc_f32(part_lse + (int64_t)pos[d] * G + ph[c]);
              }
#pragma unroll
          for (int d = 0; d < kNb; ++d)
#pragma unroll
            for (int c = 0; c < kIpl; ++c)
              if (pos[d] >= 0 && c < ipl) {
                const float wt = ex2(lv[d][c] - pm[c]) * pi[c];
                const uint32_t wd[4] = {u[d][c].x, u[d][c].y, u[d][c].z, u[d][c].w};
#pragma unroll
                for (int k2 = 0; k2 < 4; ++k2) {
                  const float2 f =
                      __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&wd[k2]));
                  ffma2(acc[c][2 * k2], acc[c][2 * k2 + 1], wt, wt, f.x, f.y, acc[c][2 * k2],
                        acc[c][2 * k2 + 1]);
                }
              }
        }
        if (qv) {
          __nv_bfloat16* orow = o + ((i0 + wq) * H_q + (int64_t)r * G) * D_H;
#pragma unroll
          for (int c = 0; c < kIpl; ++c)
            if (c < ipl) {
              uint4 v;
              v.x = pack_bf16x2(acc[c][0], acc[c][1]);
              v.y = pack_bf16x2(acc[c][2], acc[c][3]);
              v.z = pack_bf16x2(acc[c][4], acc[c][5]);
              v.w = pack_bf16x2(acc[c][6], acc[c][7]);
              *reinterpret_cast<uint4*>(orow + pe[c]) = v;
            }
        }
      }
    }
  }
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, L::kTmemCols);
  }
}

}  // namespace

template <int D_H>
static cudaError_t launch_shared_t(const CUtensorMap& tq, const CUtensorMap& tk,
                                   const CUtensorMap& tv, const void* q,
                                   const int* tile_list, const unsigned long long* tile_priv,
                                   const void* part_o,
                                   const float* part_lse, void* o, float* lse, int64_t N,
                                   int64_t q0, int64_t q1, int H_q, int H_kv, int kk,
                                   cudaStream_t st) {
  using L = ShSmem<D_H>;
  auto kern = k_attn_shared<D_H>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kAlloc);
  if (e != cudaSuccess) return e;
  const int64_t ntiles = (q1 - q0 + kTileQ - 1) / kTileQ;
  const float scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)D_H));
  kern<<<(unsigned)(ntiles * H_kv), kShThreads, L::kAlloc, st>>>(
      tq, tk, tv, static_cast<const __nv_bfloat16*>(q), tile_list, tile_priv,
      static_cast<const __nv_bfloat16*>(part_o), part_lse, static_cast<__nv_bfloat16*>(o), lse, N,
      q0, q1, H_q, H_q / H_kv, kk, ntiles, scale_log2);
  return cudaGetLastError();
}

cudaError_t launch_attn_shared(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                               const void* q,
                               const int* tile_list, const unsigned long long* tile_priv,
                               const void* part_o,
                               const float* part_lse, void* o, float* lse, int64_t N, int64_t q0,
                               int64_t q1, int H_q, int H_kv, int d_h, int kk, cudaStream_t st) {
  if (d_h == 128)
    return launch_shared_t<128>(tq, tk, tv, q, tile_list, tile_priv, part_o, part_lse, o, lse, N, q0, q1, H_q,
                                H_kv, kk, st);
  return launch_shared_t<64>(tq, tk, tv, q, tile_list, tile_priv, part_o, part_lse, o, lse, N, q0, q1, H_q,
                             H_kv, kk, st);
}

cudaError_t read_reset_shared_status(unsigned* out) {
  unsigned zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(out, g_shared_status, sizeof(unsigned));
  if (e != cudaSuccess) return e;
  return cudaMemcpyToSymbol(g_shared_status, &zero, sizeof(unsigned));
}

}  // namespace msa

// Shared-block pass of the sparse main branch («MiniMax-M3：MSA 技术报告速读», section 主分支,
// eq. O^(h)_i; LSE from section Kernel): the KV blocks that two or more queries of a 16-query
// tile selected, processed once for the tile on the 5th-generation tensor cores.
//
// One CTA = one tile (16 consecutive queries of KV group r).  Its 16*G <= 128 (query, head)
// rows are the M side of every UMMA:
//   warp 0   builds the tile's union of selections, keeps the shared blocks, then streams them
//            as 32-token half blocks (K and V, 3-D tensor maps over [N, H_kv, d_h], 128-byte
//            swizzle) through a 3-stage TMA ring;
//   warp 1   allocates TMEM and issues  S[buf] = Q K^T  (M=128, N=32) and  O += P V  (M=128,
//            N=d_h, V as an MN-major operand); S is double-buffered so the next half block's
//            QK^T runs while the softmax of this one is computed;
//   warps 2-5 own one row each (TMEM lane): they load Q, read S rows, mask queries that did not
//            select the block and keys after the query, and write P (bf16, 64-byte swizzle).
// Online softmax with a lazily moved reference max: a row's reference m moves only when a block
// max exceeds it by more than 2^8, so P <= 2^8 and O (in TMEM) is rescaled only then.  The
// result is exact either way -- O/l and m + log2 l use the same reference.
// The epilogue finishes each row: it combines the row's shared-block state (O in TMEM, fp32)
// with the row's private-block partials written by the block-major pass (k_attn_kvouter.cu, run
// before this kernel) in slot order, and writes O (bf16) and the natural-log LSE.
// Every wait is bounded; a timeout sets the device status word and the roles stop.
#include <climits>
#include <cmath>

#include "attn_tile.cuh"
#include "msa_internal.h"

namespace msa {
namespace {

__device__ unsigned g_shared_status = 0;

constexpr int kRing = 3;                 // half-block stages
constexpr int kHalfTok = 32;             // tokens per stage
constexpr int kShThreads = 192;          // producer, MMA, 4 softmax/epilogue warps
constexpr int kMaxShared = kMaxKeys / 2; // a shared block holds at least two selections

template <int D_H>
struct ShSmem {
  static constexpr int kHalves = D_H / 64;
  static constexpr int kQHalf = 128 * 128;          // 128 rows x 64 dims
  static constexpr int kBox = kHalfTok * 128;       // 32 tokens x 64 dims
  static constexpr int kKBytes = kHalves * kBox;
  static constexpr int kStage = 2 * kKBytes;        // K boxes, then V boxes
  static constexpr int kOffQ = 0;
  static constexpr int kOffRing = kOffQ + kHalves * kQHalf;
  static constexpr int kOffP = kOffRing + kRing * kStage;      // 128 rows x 32 keys, SW64
  static constexpr int kOffList = kOffP + 128 * 64;
  static constexpr int kOffBar = kOffList + kMaxShared * 4;
  // kv_full[kRing], kv_empty[kRing], s_full[2], s_free[2], p_full, p_free, q_ready, done
  static constexpr int kNumBars = 2 * kRing + 8;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;
  static constexpr int kBytes = kOffMisc + 16;
  static constexpr int kAlloc = kBytes + 1024;
  static constexpr uint32_t kTmemCols = 256;        // S[0] 0..31, S[1] 32..63, O from 128
  static_assert(kRing * kStage >= kMaxKeys * 8, "the union is built in the ring");
};

#define MSA_TMEM_LD32(taddr, r)                                                                 \
  asm volatile(                                                                                 \
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "                                                 \
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"                                 \
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"                \
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),     \
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), \
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),           \
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),           \
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])            \
      : "r"(taddr))

#define MSA_TMEM_ST64(taddr, r)                                                                 \
  asm volatile(                                                                                 \
      "tcgen05.st.sync.aligned.32x32b.x64.b32 [%0], "                                           \
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"                                \
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32,"                        \
      "%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,%48,"                        \
      "%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63,%64};" ::"r"(taddr),         \
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),   \
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),         \
      "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]),       \
      "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]),       \
      "r"(r[29]), "r"(r[30]), "r"(r[31]), "r"(r[32]), "r"(r[33]), "r"(r[34]), "r"(r[35]),       \
      "r"(r[36]), "r"(r[37]), "r"(r[38]), "r"(r[39]), "r"(r[40]), "r"(r[41]), "r"(r[42]),       \
      "r"(r[43]), "r"(r[44]), "r"(r[45]), "r"(r[46]), "r"(r[47]), "r"(r[48]), "r"(r[49]),       \
      "r"(r[50]), "r"(r[51]), "r"(r[52]), "r"(r[53]), "r"(r[54]), "r"(r[55]), "r"(r[56]),       \
      "r"(r[57]), "r"(r[58]), "r"(r[59]), "r"(r[60]), "r"(r[61]), "r"(r[62]), "r"(r[63])        \
      : "memory")

__device__ __forceinline__ void tmem_st_wait() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void fence_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ uint64_t desc_mn_sw128(uint32_t a, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((a & 0x3FFFFu) >> 4) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

template <int EPL>
__device__ __forceinline__ int shared_blocks(const int32_t* __restrict__ idx, int r, int64_t i0,
                                             int64_t q1, int64_t N, int kk, int* tmpU,
                                             unsigned* tmpM, int* s_list) {
  const int lane = threadIdx.x & 31;
  int x[EPL], rank[EPL];
  const int nU = tile_union<EPL>(idx, r, i0, q1, N, kk, x, rank, tmpU, tmpM);
  int nS = 0;
  for (int base = 0; base < nU; base += 32) {
    const int u = base + lane;
    const unsigned m = u < nU ? tmpM[u] : 0u;
    const bool keep = __popc(m) >= 2;
    const unsigned kb = __ballot_sync(kAllLanes, keep);
    if (keep) s_list[nS + __popc(kb & ((1u << lane) - 1u))] = (tmpU[u] << 16) | (int)m;
    nS += __popc(kb);
  }
  __syncwarp();
  return nS;
}

template <int D_H>
__global__ void __launch_bounds__(kShThreads, 2)
    k_attn_shared(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                  const __nv_bfloat16* __restrict__ q, const int32_t* __restrict__ idx,
                  const int* __restrict__ slotmap, const __nv_bfloat16* __restrict__ part_o,
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
  const uint32_t bar = sb + L::kOffBar;
  auto kv_full = [&](int s) { return bar + 8u * s; };
  auto kv_empty = [&](int s) { return bar + 8u * (kRing + s); };
  auto s_full = [&](int b) { return bar + 8u * (2 * kRing + b); };
  auto s_free = [&](int b) { return bar + 8u * (2 * kRing + 2 + b); };
  const uint32_t p_full = bar + 8u * (2 * kRing + 4), p_free = bar + 8u * (2 * kRing + 5);
  const uint32_t q_ready = bar + 8u * (2 * kRing + 6), done = bar + 8u * (2 * kRing + 7);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t bid = blockIdx.x;
  const int r = (int)(bid / ntiles);
  const int64_t i0 = q0 + (bid - (int64_t)r * ntiles) * kTileQ;
  const int rows = kTileQ * G;                       // 16 G <= 128 rows in use

  if (warp == 0) {
    int* tmpU = reinterpret_cast<int*>(smem + L::kOffRing);
    unsigned* tmpM = reinterpret_cast<unsigned*>(smem + L::kOffRing + kMaxKeys * 4);
    const int nS = with_epl(kk, [&](auto e) {
      return shared_blocks<decltype(e)::value>(idx, r, i0, q1, N, kk, tmpU, tmpM, s_list);
    });
    if (lane == 0) {
      *s_nS = nS;
      for (int s = 0; s < kRing; ++s) {
        mbar_init(kv_full(s), 1);
        mbar_init(kv_empty(s), 1);
      }
      for (int b = 0; b < 2; ++b) {
        mbar_init(s_full(b), 1);
        mbar_init(s_free(b), 4);
      }
      mbar_init(p_full, 4);
      mbar_init(p_free, 1);
      mbar_init(q_ready, 4);
      mbar_init(done, 1);
      fence_barrier_init();
    }
  } else if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), L::kTmemCols);
    tc_fence_before();
  } else {
    // softmax warps: gather the tile's Q rows (row R = query w * G + head h) into SW128 halves
    constexpr int kChunks = D_H / 8;
    for (int x = threadIdx.x - 64; x < rows * kChunks; x += 128) {
      const int R = x / kChunks, c = x - R * kChunks;
      const int w = R / G;
      const int64_t i = i0 + w;
      if (i >= q1) continue;
      const uint32_t off = (c >> 3) * L::kQHalf + R * 128 + (((c & 7) ^ (R & 7)) << 4);
      cp_async16(sb + L::kOffQ + off, q + (i * H_q + (int64_t)r * G + (R - w * G)) * D_H + c * 8);
    }
    asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
    fence_async_smem();
  }
  __syncthreads();
  tc_fence_after();
  const int nS = *s_nS;
  const int nH = 2 * nS;                              // half blocks
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------------ producer
    if (lane == 0) {
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
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_s = umma_idesc_bf16(128, kHalfTok);
      constexpr uint32_t idesc_o = umma_idesc_bf16(128, D_H) | (1u << 16);   // B MN-major
      bool ok = mbar_wait(q_ready, 0, &g_shared_status);
      auto issue_s = [&](int hb) -> bool {
        const int s = hb % kRing, b = hb & 1;
        if (!mbar_wait(kv_full(s), (hb / kRing) & 1, &g_shared_status)) return false;
        if (!mbar_wait(s_free(b), ((hb >> 1) & 1) ^ 1, &g_shared_status)) return false;
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
      for (int hb = 0; hb < nH && ok; ++hb) {
        if (hb + 1 < nH && !(ok = issue_s(hb + 1))) break;
        if (!(ok = mbar_wait(p_full, hb & 1, &g_shared_status))) break;
        tc_fence_after();
        const uint32_t vbase = sb + L::kOffRing + (hb % kRing) * L::kStage + L::kKBytes;
#pragma unroll
        for (int ks = 0; ks < kHalfTok / 16; ++ks)
          umma_bf16(tmem + 128, umma_desc_kmajor(sb + L::kOffP + ks * 32, 512, 64),
                    desc_mn_sw128(vbase + ks * 2048, L::kBox, 1024), idesc_o,
                    (hb > 0 || ks > 0) ? 1u : 0u);
        umma_commit(p_free);
        umma_commit(kv_empty(hb % kRing));
      }
      umma_commit(done);
      mbar_wait(done, 0, &g_shared_status);
    }
  } else {
    // ------------------------------------------------------ softmax and epilogue
    const int qd = warp & 3;                          // TMEM lane quarter
    const int R = 32 * qd + lane;
    const int w = R / G, h = R - (R / G) * G;
    const int64_t i = i0 + w;
    const bool valid = R < rows && i < q1;
    const uint32_t lanes = (uint32_t)(32 * qd) << 16;
    __syncwarp();
    if (lane == 0) mbar_arrive(q_ready);
    float m_ref = -INFINITY, l = 0.f;
    bool ok = true;
    for (int hb = 0; hb < nH && ok; ++hb) {
      const int ent = s_list[hb >> 1];
      const int64_t b = ent >> 16;
      const bool sel = valid && ((ent >> w) & 1);
      const int buf = hb & 1;
      if (!(ok = __all_sync(kAllLanes, mbar_wait(s_full(buf), (hb >> 1) & 1, &g_shared_status))))
        break;
      tc_fence_after();
      uint32_t sv[32];
      MSA_TMEM_LD32(tmem + lanes + 32 * buf, sv);
      tmem_ld_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(s_free(buf));

      float alpha = 1.f;
      uint32_t pk[16];
      if (sel) {
        const int64_t j0 = b * kBlock + (hb & 1) * kHalfTok;
        float bm = -INFINITY;
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          if (j0 + c > i) sv[c] = __float_as_uint(-INFINITY);
          bm = fmaxf(bm, __uint_as_float(sv[c]));
        }
        bm *= scale_log2;
        if (m_ref == -INFINITY) {
          m_ref = bm;                                 // this row's O and l are still zero
        } else if (bm > m_ref + 8.f) {
          alpha = ex2(m_ref - bm);
          m_ref = bm;
        }
        float ps = 0.f;
#pragma unroll
        for (int c = 0; c < 16; ++c) {
          const float p0 = ex2(__uint_as_float(sv[2 * c]) * scale_log2 - m_ref);
          const float p1 = ex2(__uint_as_float(sv[2 * c + 1]) * scale_log2 - m_ref);
          ps += p0 + p1;
          pk[c] = pack_bf16x2(p0, p1);
        }
        l = l * alpha + ps;
      } else {
#pragma unroll
        for (int c = 0; c < 16; ++c) pk[c] = 0u;
      }
      // P and O may be touched once the previous half block's O += P V has completed
      if (hb > 0 &&
          !(ok = __all_sync(kAllLanes, mbar_wait(p_free, (hb - 1) & 1, &g_shared_status))))
        break;
      if (__any_sync(kAllLanes, alpha != 1.f)) {
        tc_fence_after();
#pragma unroll
        for (int part = 0; part < D_H / 64; ++part) {
          uint32_t ov[64];
          MSA_TMEM_LD64(tmem + lanes + 128 + 64 * part, ov);
          tmem_ld_wait();
#pragma unroll
          for (int c = 0; c < 64; ++c) ov[c] = __float_as_uint(__uint_as_float(ov[c]) * alpha);
          MSA_TMEM_ST64(tmem + lanes + 128 + 64 * part, ov);
        }
        tmem_st_wait();
      }
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const uint32_t addr = sb + L::kOffP + R * 64 + ((c ^ ((R >> 1) & 3)) << 4);
        asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(addr), "r"(pk[4 * c]),
                     "r"(pk[4 * c + 1]), "r"(pk[4 * c + 2]), "r"(pk[4 * c + 3])
                     : "memory");
      }
      fence_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(p_full);
    }
    // ---- epilogue: shared-block state + private partials of this row, in slot order
    if (ok) ok = __all_sync(kAllLanes, mbar_wait(done, 0, &g_shared_status));
    tc_fence_after();
    const bool have_o = nH > 0 && ok;               // warp-uniform
    const int* sm = slotmap + ((int64_t)r * (q1 - q0) + (i - q0)) * kk;
    const float lse_s = l > 0.f ? m_ref + __log2f(l) : -INFINITY;
    float mx = lse_s;
    if (valid)
      for (int t = 0; t < kk; ++t) {
        const int pos = __ldg(sm + t);
        if (pos >= 0) mx = fmaxf(mx, __ldg(part_lse + (int64_t)pos * G + h));
      }
    const float w_s = lse_s == -INFINITY ? 0.f : ex2(lse_s - mx);
    float wsum = w_s;
    if (valid)
      for (int t = 0; t < kk; ++t) {
        const int pos = __ldg(sm + t);
        if (pos >= 0) wsum += ex2(__ldg(part_lse + (int64_t)pos * G + h) - mx);
      }
    const float inv_w = wsum > 0.f ? 1.f / wsum : 0.f;
    const float c_s = l > 0.f ? w_s / l : 0.f;      // weight of the TMEM accumulator
#pragma unroll
    for (int part = 0; part < D_H / 64; ++part) {
      uint32_t ov[64];
      if (have_o) {
        MSA_TMEM_LD64(tmem + lanes + 128 + 64 * part, ov);
        tmem_ld_wait();
      }
      if (valid) {
        float acc[64];
#pragma unroll
        for (int c = 0; c < 64; ++c) acc[c] = have_o ? __uint_as_float(ov[c]) * c_s : 0.f;
        for (int t = 0; t < kk; ++t) {
          const int pos = __ldg(sm + t);
          if (pos < 0) continue;
          const float wp = ex2(__ldg(part_lse + (int64_t)pos * G + h) - mx);
          const uint4* src =
              reinterpret_cast<const uint4*>(part_o + ((int64_t)pos * G + h) * D_H + 64 * part);
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            const uint4 u = __ldg(src + c);
            const uint32_t wd[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
            for (int k2 = 0; k2 < 4; ++k2) {
              const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&wd[k2]));
              acc[8 * c + 2 * k2] += wp * f.x;
              acc[8 * c + 2 * k2 + 1] += wp * f.y;
            }
          }
        }
        uint4* dst = reinterpret_cast<uint4*>(o + (i * H_q + (int64_t)r * G + h) * D_H + 64 * part);
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          uint4 v4;
          v4.x = pack_bf16x2(acc[8 * c + 0] * inv_w, acc[8 * c + 1] * inv_w);
          v4.y = pack_bf16x2(acc[8 * c + 2] * inv_w, acc[8 * c + 3] * inv_w);
          v4.z = pack_bf16x2(acc[8 * c + 4] * inv_w, acc[8 * c + 5] * inv_w);
          v4.w = pack_bf16x2(acc[8 * c + 6] * inv_w, acc[8 * c + 7] * inv_w);
          dst[c] = v4;
        }
      }
    }
    if (valid) lse[((int64_t)r * G + h) * N + i] = (mx + __log2f(wsum)) * 0.69314718055994531f;
    tc_fence_before();
  }

  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, L::kTmemCols);
  }
}

}  // namespace

template <int D_H>
static cudaError_t launch_shared_t(const CUtensorMap& tk, const CUtensorMap& tv, const void* q,
                                   const int32_t* idx, const int* slotmap, const void* part_o,
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
      tk, tv, static_cast<const __nv_bfloat16*>(q), idx, slotmap,
      static_cast<const __nv_bfloat16*>(part_o), part_lse, static_cast<__nv_bfloat16*>(o), lse, N,
      q0, q1, H_q, H_q / H_kv, kk, ntiles, scale_log2);
  return cudaGetLastError();
}

cudaError_t launch_attn_shared(const CUtensorMap& tk, const CUtensorMap& tv, const void* q,
                               const int32_t* idx, const int* slotmap, const void* part_o,
                               const float* part_lse, void* o, float* lse, int64_t N, int64_t q0,
                               int64_t q1, int H_q, int H_kv, int d_h, int kk, cudaStream_t st) {
  if (d_h == 128)
    return launch_shared_t<128>(tk, tv, q, idx, slotmap, part_o, part_lse, o, lse, N, q0, q1, H_q,
                                H_kv, kk, st);
  return launch_shared_t<64>(tk, tv, q, idx, slotmap, part_o, part_lse, o, lse, N, q0, q1, H_q,
                             H_kv, kk, st);
}

cudaError_t read_reset_shared_status(unsigned* out) {
  unsigned zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(out, g_shared_status, sizeof(unsigned));
  if (e != cudaSuccess) return e;
  return cudaMemcpyToSymbol(g_shared_status, &zero, sizeof(unsigned));
}

}  // namespace msa

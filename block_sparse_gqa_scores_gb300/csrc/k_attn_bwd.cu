// Backward of the sparse main branch («MiniMax-M3：MSA 技术报告速读», section 主分支 eq. O^(h)_i
// differentiated; the kernel section's persistent, load-balanced backward with pre-scheduled
// splits and an ordered merge).  For every row i, head h (group r) and selected visible token
// j in T_i, with s_j = Q[i,h].K[j,r]/sqrt(d_h) and the forward's LSE:
//   P_j  = exp(s_j - LSE[h,i]),   dP_j = dO[i,h] . V[j,r],   D = dO[i,h] . O[i,h]
//   dS_j = P_j (dP_j - D)
//   dQ[i,h] = sum_j dS_j K[j,r] / sqrt(d_h)
//   dK[j,r] = sum_{(i,h): j in T_i} dS_j Q[i,h] / sqrt(d_h),   dV[j,r] = sum_{(i,h)} P_j dO[i,h]
//
// Organisation (KV-outer, like the forward's block-major pass): every selection is bucketed by
// (group, block); a work tile stacks up to 128/G entries of one bucket, G rows each, into one
// 128-row UMMA tile.  Each bucket's tiles are cut into pieces of at most kPiece tiles (the
// pre-scheduled splits); a piece's dK and dV accumulate in TMEM over its tiles and leave as one
// fp32 partial, and pieces are dealt to persistent CTAs by equal shares of work tiles (hot blocks
// selected by most queries become many pieces spread over many CTAs).  Per tile:
//   S    = Q_stack  K_b^T            M=128 rows, N=64 keys, K=d_h        (tcgen05, TMEM)
//   dP   = dO_stack V_b^T            M=128 rows, N=64 keys, K=d_h
//   thread per row: P, dS -> shared memory (bf16, 128-byte swizzle)
//   dV^T += dO_stack^T P             M=d_h dims, N=64 keys, K=128 rows  (both operands MN-major)
//   dK^T += Q_stack^T dS             M=d_h dims, N=64 keys, K=128 rows
//   dQp  = dS K_b                    M=128 rows, N=d_h, K=64 keys       (K_b MN-major)
// and each row writes its dQ partial (bf16; staged in shared memory and stored by TMA at G = 8)
// at the fixed position of its (group, row, slot).
// Merges: dQ of a row sums its slots in slot order; dK, dV of a block sum the bucket's pieces in
// piece order.  The buckets list their selections in row order (row-ordered planning), so the
// work tiles and every sum's order are fixed: no atomic update of any result, and every output
// is the same bit for bit on every call.
// One CTA per SM (its tensor memory and shared memory), 128 threads; thread 0 issues the copies
// and MMAs, every thread owns one TMEM lane (row) in the epilogues.  Every wait is bounded.
#include <cmath>

#include "msa_device.cuh"
#include "msa_internal.h"

namespace msa {
namespace {

__device__ unsigned g_bwd_status = 0;

constexpr int kRowsB = 128;            // UMMA M of the row-major products
constexpr int kThreadsB = 128;
constexpr int kPiece = 64;             // most work tiles per piece (one dK/dV partial)
constexpr float kLog2eB = 1.442695040888963407f;

// TMEM columns: S [0,64), dP [64,128); dQp [0, d_h) over them once both are read;
// dV^T [128,192), dK^T [192,256) (lane = dim)
constexpr uint32_t kColDP = 64, kColDV = 128, kColDK = 192;

template <int D_H>
struct BwdSmem {
  static constexpr int kHalves = D_H / 64;
  static constexpr int kRowHalf = kRowsB * 128;    // 128 rows x 64 dims, SW128
  static constexpr int kKeyHalf = 64 * 128;        // 64 keys x 64 dims, SW128
  static constexpr int kRowTile = kHalves * kRowHalf;
  static constexpr int kOffQ = 0;
  static constexpr int kOffDO = kOffQ + kRowTile;
  // the second 64-dim block of the transposed A operands at d_h = 64 reads past the tile (its
  // results land in TMEM lanes that are never read); two row tiles keep it inside the buffer
  static constexpr int kOffK = kOffDO + (D_H == 64 ? 2 : 1) * kRowTile;
  static constexpr int kOffV = kOffK + kHalves * kKeyHalf;
  static constexpr int kOffP = kOffV + kHalves * kKeyHalf;      // P  [128 rows][64 keys] bf16
  static constexpr int kOffS = kOffP + kRowsB * 128;            // dS [128 rows][64 keys] bf16
  static constexpr int kOffBar = kOffS + kRowsB * 128;          // kv, rows, mma, drain
  static constexpr int kOffMisc = kOffBar + 32;
  static constexpr int kOffEnt = kOffMisc + 16;
  static constexpr int kBytes = kOffEnt + 4 * kRowsB;
  // more than half of the SM's shared memory: one CTA per SM
  static constexpr int kAlloc = kBytes + 1024 > 116 * 1024 ? kBytes + 1024 : 116 * 1024;
  static_assert(kAlloc <= 227 * 1024, "shared memory");
};

__device__ __forceinline__ void bwd_cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void bwd_cp_async_wait() {
  asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
}
__device__ __forceinline__ void bwd_fence_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void st_shared_v4(uint32_t a, uint32_t x, uint32_t y, uint32_t z,
                                             uint32_t w) {
  asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(a), "r"(x), "r"(y), "r"(z), "r"(w)
               : "memory");
}

// D[h, i] = dO[i, h, :] . O[i, h, :] in fp32, one warp per (row, head).
__global__ void __launch_bounds__(256)
    k_attn_bwd_delta(const __nv_bfloat16* __restrict__ o, const __nv_bfloat16* __restrict__ d_o,
                     float* __restrict__ delta, int64_t N, int H_q, int d_h) {
  const int64_t wid = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (wid >= N * H_q) return;
  const int64_t i = wid / H_q;
  const int h = (int)(wid - i * H_q);
  const __nv_bfloat162* a = reinterpret_cast<const __nv_bfloat162*>(o + wid * d_h);
  const __nv_bfloat162* b = reinterpret_cast<const __nv_bfloat162*>(d_o + wid * d_h);
  float acc = 0.f;
  for (int x = lane; x < d_h / 2; x += 32) {
    const float2 fa = __bfloat1622float2(a[x]), fb = __bfloat1622float2(b[x]);
    acc += fa.x * fb.x + fa.y * fb.y;
  }
#pragma unroll
  for (int m = 16; m > 0; m >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, m);
  if (lane == 0) delta[(int64_t)h * N + i] = acc;
}

// piece_off[b] = sum_{b' < b} ceil(tiles of b' / kPiece), with the total at index nb (one CTA).
constexpr int kScanB = 1024;
__global__ void __launch_bounds__(kScanB)
    k_attn_bwd_pieces(const int* __restrict__ tile_off, int* __restrict__ piece_off, int nb) {
  __shared__ int s_a[kScanB];
  const int tid = threadIdx.x;
  const int per = (nb + kScanB - 1) / kScanB;
  const int beg = min(nb, tid * per), end = min(nb, beg + per);
  int sum = 0;
  for (int b = beg; b < end; ++b) sum += (tile_off[b + 1] - tile_off[b] + kPiece - 1) / kPiece;
  s_a[tid] = sum;
  __syncthreads();
  for (int o = 1; o < kScanB; o <<= 1) {
    const int v = tid >= o ? s_a[tid - o] : 0;
    __syncthreads();
    s_a[tid] += v;
    __syncthreads();
  }
  int run = s_a[tid] - sum;
  for (int b = beg; b < end; ++b) {
    piece_off[b] = run;
    run += (tile_off[b + 1] - tile_off[b] + kPiece - 1) / kPiece;
  }
  if (tid == kScanB - 1) piece_off[nb] = s_a[tid];
}

struct BwdArgs {
  const __nv_bfloat16* q;
  const __nv_bfloat16* d_o;
  const float* lse;          // [H_q, N], natural log
  const float* delta;        // [H_q, N]
  const int* entries;
  const int* offset;
  const int* tile_off;
  const int* piece_off;
  __nv_bfloat16* part_dq;    // [H_kv, N, k, G, d_h]
  float* part_dkv;           // [pieces, 2, d_h, 64]: dK^T then dV^T
  int64_t N;
  int nb, nblk, H_kv, kk;
  float scale_log2;          // log2(e) / sqrt(d_h)
};

template <int D_H, int G>
__global__ void __launch_bounds__(kThreadsB, 1)
    k_attn_bwd_kvouter(const __grid_constant__ CUtensorMap tm_q,
                       const __grid_constant__ CUtensorMap tm_do,
                       const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v,
                       const __grid_constant__ CUtensorMap tm_dq, const BwdArgs a) {
  using L = BwdSmem<D_H>;
  constexpr int kEpt = kRowsB / G;
  constexpr int kChunks = D_H / 8;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t sb = smem_u32(smem);
  const uint32_t kv_bar = sb + L::kOffBar, row_bar = kv_bar + 8, mma_bar = kv_bar + 16;
  const uint32_t drain_bar = kv_bar + 24;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kOffMisc);
  int* s_ent = reinterpret_cast<int*>(smem + L::kOffEnt);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int H_q = a.H_kv * G;

  if (tid == 0) {
    mbar_init(kv_bar, 1);
    mbar_init(row_bar, 1);
    mbar_init(mma_bar, 1);
    mbar_init(drain_bar, 1);
    fence_barrier_init();
  }
  // Rows past a tile's entries keep whatever the buffer held; zeroed once here, they only ever
  // hold finite query rows afterwards, so their zero P and dS rows add exact zeros to dK and dV
  for (int x = tid; x < (L::kOffK - L::kOffQ) / 16; x += kThreadsB)
    st_shared_v4(sb + L::kOffQ + 16 * x, 0u, 0u, 0u, 0u);
  bwd_fence_async_smem();
  if (warp == 0) {
    tmem_alloc(smem_u32(tmem_slot), 256);
    tc_fence_before();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t lanes = (uint32_t)(32 * warp) << 16;
  uint32_t kv_ph = 0, row_ph = 0, mma_ph = 0;
  bool ok = true;
  // every thread waits on the barrier; the CTA proceeds only if all of them saw it complete
  auto wait_all = [&](uint32_t bar, uint32_t& ph) -> bool {
    const bool w = mbar_wait(bar, ph, &g_bwd_status);
    ph ^= 1u;
    return __syncthreads_and(w) != 0;
  };

  // this CTA's share of the work tiles; it takes the pieces that start inside it
  const int T = __ldg(a.tile_off + a.nb);
  const int per = (T + (int)gridDim.x - 1) / (int)gridDim.x;
  const int t_lo = (int)blockIdx.x * per, t_hi = min(T, t_lo + per);
  int b = 0;
  if (t_lo < t_hi) {
    int lo = 0, hi = a.nb;                                    // tile_off[lo] <= t_lo < tile_off[hi]
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (__ldg(a.tile_off + mid) <= t_lo) lo = mid; else hi = mid;
    }
    b = lo;
  }
  int m = t_lo < t_hi ? (t_lo - __ldg(a.tile_off + b) + kPiece - 1) / kPiece : 0;
  constexpr uint32_t idesc_s = umma_idesc_bf16(kRowsB, 64);
  // transposed products: A (dims x rows) and B (rows x keys) both MN-major
  constexpr uint32_t idesc_t = umma_idesc_bf16(128, 64) | (1u << 15) | (1u << 16);
  constexpr uint32_t idesc_q = umma_idesc_bf16(kRowsB, D_H) | (1u << 16);   // B (K_b) MN-major

  while (ok && t_lo < t_hi) {
    // the next piece starting in [t_lo, t_hi): bucket b, tiles [p0, p1)
    const int tb0 = __ldg(a.tile_off + b), tb1 = __ldg(a.tile_off + b + 1);
    const int p0 = tb0 + m * kPiece;
    if (p0 >= tb1) {
      if (++b >= a.nb) break;
      m = 0;
      continue;
    }
    if (p0 >= t_hi) break;
    const int p1 = min(tb1, p0 + kPiece);
    const int piece = __ldg(a.piece_off + b) + m;
    ++m;
    const int rb = b / a.nblk;
    const int blk = b - rb * a.nblk;
    // ---- K_b, V_b of the piece (TMA; rows past the sequence read as zeros)
    if (tid == 0) {
      mbar_expect_tx(kv_bar, (uint32_t)(2 * L::kHalves * L::kKeyHalf));
#pragma unroll
      for (int bx = 0; bx < L::kHalves; ++bx) {
        tma_load_3d(sb + L::kOffK + bx * L::kKeyHalf, &tm_k, kv_bar, 64 * bx, rb, blk * kBlock);
        tma_load_3d(sb + L::kOffV + bx * L::kKeyHalf, &tm_v, kv_bar, 64 * bx, rb, blk * kBlock);
      }
    }
    if (!(ok = wait_all(kv_bar, kv_ph))) break;
    for (int t = p0; t < p1 && ok; ++t) {
      const int e0 = __ldg(a.offset + b) + (t - tb0) * kEpt;
      const int n_e = min(kEpt, __ldg(a.offset + b + 1) - e0);
      if (tid < n_e) s_ent[tid] = __ldg(a.entries + e0 + tid);
      __syncthreads();
      // ---- the tile's stacked Q and dO rows
      if (G == 8) {
        if (warp == 0) {
          if (lane == 0) mbar_expect_tx(row_bar, (uint32_t)(2 * n_e * 8 * 128 * L::kHalves));
          __syncwarp();
          if (lane < n_e) {
            const int i = s_ent[lane] >> 6;
#pragma unroll
            for (int bx = 0; bx < L::kHalves; ++bx) {
              tma_load_3d(sb + L::kOffQ + bx * L::kRowHalf + lane * 1024, &tm_q, row_bar, 64 * bx,
                          rb * 8, i);
              tma_load_3d(sb + L::kOffDO + bx * L::kRowHalf + lane * 1024, &tm_do, row_bar,
                          64 * bx, rb * 8, i);
            }
          }
        }
        if (!(ok = wait_all(row_bar, row_ph))) break;
      } else {
        for (int x = tid; x < n_e * G * kChunks; x += kThreadsB) {
          const int R = x / kChunks, c = x - R * kChunks;
          const int e = R / G, h = R - e * G;
          const int64_t i = s_ent[e] >> 6;
          const uint32_t off = (c >> 3) * L::kRowHalf + R * 128 + (((c & 7) ^ (R & 7)) << 4);
          const int64_t src = (i * H_q + (int64_t)rb * G + h) * D_H + c * 8;
          bwd_cp_async16(sb + L::kOffQ + off, a.q + src);
          bwd_cp_async16(sb + L::kOffDO + off, a.d_o + src);
        }
        bwd_cp_async_wait();
        bwd_fence_async_smem();
        __syncthreads();
      }
      // ---- S = Q K_b^T and dP = dO V_b^T
      if (tid == 0) {
        bulk_wait_read_all();           // the previous tile's dQ stores have read the staging
        tc_fence_after();
#pragma unroll
        for (int ks = 0; ks < D_H / 16; ++ks) {
          const uint32_t koff = (ks >> 2) * L::kKeyHalf + (ks & 3) * 32;
          const uint32_t roff = (ks >> 2) * L::kRowHalf + (ks & 3) * 32;
          umma_bf16(tmem, umma_desc_kmajor(sb + L::kOffQ + roff, 1024, 128),
                    umma_desc_kmajor(sb + L::kOffK + koff, 1024, 128), idesc_s, ks > 0 ? 1u : 0u);
          umma_bf16(tmem + kColDP, umma_desc_kmajor(sb + L::kOffDO + roff, 1024, 128),
                    umma_desc_kmajor(sb + L::kOffV + koff, 1024, 128), idesc_s, ks > 0 ? 1u : 0u);
        }
        umma_commit(mma_bar);
      }
      if (!(ok = wait_all(mma_bar, mma_ph))) break;
      tc_fence_after();
      // ---- thread per row: P and dS into shared memory (bf16, [row][key], 128-byte swizzle)
      const int R = tid;
      const bool rv = R < n_e * G;
      const int e = R / G, h = R - e * G;
      const int ent = rv ? s_ent[e] : 0;
      const int64_t i = ent >> 6;
      {
        uint32_t sv[64], dp[64];
        MSA_TMEM_LD64(tmem + lanes, sv);
        MSA_TMEM_LD64(tmem + lanes + kColDP, dp);
        tmem_ld_wait();
        float lse2 = 0.f, dlt = 0.f;
        int cmax = -1;                                        // last visible key, -1: none
        if (rv) {
          const int64_t hr = (int64_t)(rb * G + h) * a.N + i;
          lse2 = __ldg(a.lse + hr) * kLog2eB;
          dlt = __ldg(a.delta + hr);
          cmax = blk == (int)(i >> 6) ? (int)(i - (int64_t)blk * kBlock) : kBlock - 1;
        }
#pragma unroll
        for (int cc = 0; cc < 8; ++cc) {
          uint32_t pw[4], dw[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int c = 8 * cc + 2 * u;
            float x0, x1;
            ffma2(x0, x1, __uint_as_float(sv[c]), __uint_as_float(sv[c + 1]), a.scale_log2,
                  a.scale_log2, -lse2, -lse2);
            const float p0 = c <= cmax ? ex2(x0) : 0.f;
            const float p1 = c + 1 <= cmax ? ex2(x1) : 0.f;
            const float d0 = c <= cmax ? p0 * (__uint_as_float(dp[c]) - dlt) : 0.f;
            const float d1 = c + 1 <= cmax ? p1 * (__uint_as_float(dp[c + 1]) - dlt) : 0.f;
            pw[u] = pack_bf16x2(p0, p1);
            dw[u] = pack_bf16x2(d0, d1);
          }
          const uint32_t sw = (uint32_t)(R * 128 + ((cc ^ (R & 7)) << 4));
          st_shared_v4(sb + L::kOffP + sw, pw[0], pw[1], pw[2], pw[3]);
          st_shared_v4(sb + L::kOffS + sw, dw[0], dw[1], dw[2], dw[3]);
        }
      }
      bwd_fence_async_smem();
      tc_fence_before();
      __syncthreads();
      // ---- dV^T += dO^T P, dK^T += Q^T dS (accumulated over the piece), dQp = dS K_b
      if (tid == 0) {
        tc_fence_after();
        const uint32_t acc = t > p0 ? 1u : 0u;
#pragma unroll
        for (int ks = 0; ks < kRowsB / 16; ++ks) {            // 16 rows per step
          const uint32_t roff = (uint32_t)ks * 2048;
          umma_bf16(tmem + kColDV, desc_mn_sw128(sb + L::kOffDO + roff, L::kRowHalf, 1024),
                    desc_mn_sw128(sb + L::kOffP + roff, 8192, 1024), idesc_t,
                    (acc | (ks > 0 ? 1u : 0u)));
          umma_bf16(tmem + kColDK, desc_mn_sw128(sb + L::kOffQ + roff, L::kRowHalf, 1024),
                    desc_mn_sw128(sb + L::kOffS + roff, 8192, 1024), idesc_t,
                    (acc | (ks > 0 ? 1u : 0u)));
        }
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)                        // 16 keys per step
          umma_bf16(tmem, umma_desc_kmajor(sb + L::kOffS + ks * 32, 1024, 128),
                    desc_mn_sw128(sb + L::kOffK + ks * 2048, L::kKeyHalf, 1024), idesc_q,
                    ks > 0 ? 1u : 0u);
        umma_commit(mma_bar);
      }
      if (!(ok = wait_all(mma_bar, mma_ph))) break;
      tc_fence_after();
      // ---- this row's dQ partial (bf16, unscaled; the merge applies 1/sqrt(d_h)).  At G = 8 the
      //      rows are staged over P and dS (free once the MMAs above completed) in the layout of a
      //      query box and stored by TMA, one 1-KB box per entry and half; otherwise row by row.
      {
        const int64_t slot = ((int64_t)rb * a.N + i) * a.kk + (ent & 63);
#pragma unroll
        for (int half = 0; half < D_H / 64; ++half) {
          uint32_t v[64];
          MSA_TMEM_LD64(tmem + lanes + 64 * half, v);
          tmem_ld_wait();
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            const uint32_t w0 = pack_bf16x2(__uint_as_float(v[8 * c]), __uint_as_float(v[8 * c + 1]));
            const uint32_t w1 = pack_bf16x2(__uint_as_float(v[8 * c + 2]), __uint_as_float(v[8 * c + 3]));
            const uint32_t w2 = pack_bf16x2(__uint_as_float(v[8 * c + 4]), __uint_as_float(v[8 * c + 5]));
            const uint32_t w3 = pack_bf16x2(__uint_as_float(v[8 * c + 6]), __uint_as_float(v[8 * c + 7]));
            if (G == 8) {
              st_shared_v4(sb + L::kOffP + half * (kRowsB * 128) + R * 128 + ((c ^ (R & 7)) << 4),
                           w0, w1, w2, w3);
            } else if (rv) {
              reinterpret_cast<uint4*>(a.part_dq + (slot * G + h) * D_H + 64 * half)[c] =
                  make_uint4(w0, w1, w2, w3);
            }
          }
        }
      }
      tc_fence_before();
      if (G == 8) bwd_fence_async_smem();
      __syncthreads();                                        // TMEM, s_ent and staging reused
      if (G == 8 && tid == 0) {
        for (int x = 0; x < n_e; ++x) {
          const int ex = s_ent[x];
          const int z = (int)(((int64_t)rb * a.N + (ex >> 6)) * a.kk + (ex & 63));
#pragma unroll
          for (int half = 0; half < D_H / 64; ++half)
            tma_store_3d(&tm_dq, sb + L::kOffP + half * (kRowsB * 128) + x * 1024, 64 * half, 0, z);
        }
        bulk_commit();
      }
      __syncthreads();                                        // s_ent read before it is reused
    }
    if (!ok) break;
    // ---- the piece's dK^T and dV^T (lane = dim): its partial
    tc_fence_after();
    {
      const int dim = tid;
      uint32_t kv[64];
      float* dst = a.part_dkv + (int64_t)piece * 2 * D_H * 64;
      MSA_TMEM_LD64(tmem + lanes + kColDK, kv);
      tmem_ld_wait();
      if (dim < D_H) {
        float4* d4 = reinterpret_cast<float4*>(dst + dim * 64);
#pragma unroll
        for (int c = 0; c < 16; ++c)
          d4[c] = make_float4(__uint_as_float(kv[4 * c]), __uint_as_float(kv[4 * c + 1]),
                              __uint_as_float(kv[4 * c + 2]), __uint_as_float(kv[4 * c + 3]));
      }
      MSA_TMEM_LD64(tmem + lanes + kColDV, kv);
      tmem_ld_wait();
      if (dim < D_H) {
        float4* d4 = reinterpret_cast<float4*>(dst + (D_H + dim) * 64);
#pragma unroll
        for (int c = 0; c < 16; ++c)
          d4[c] = make_float4(__uint_as_float(kv[4 * c]), __uint_as_float(kv[4 * c + 1]),
                              __uint_as_float(kv[4 * c + 2]), __uint_as_float(kv[4 * c + 3]));
      }
    }
    tc_fence_before();
    __syncthreads();
  }

  if (tid == 0) bulk_wait_all();                            // the dQ stores have completed
  if (!ok && tid == 0) {
    // a wait gave up: let whatever it waited for land (bounded) and every MMA issued complete
    // before the tensor memory is released
    mbar_wait(kv_bar, kv_ph ^ 1u, &g_bwd_status);
    mbar_wait(row_bar, row_ph ^ 1u, &g_bwd_status);
    umma_commit(drain_bar);
    mbar_wait(drain_bar, 0, &g_bwd_status);
  }
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 256);
  }
}

// dq[i, h, :] = (1/sqrt(d_h)) sum over the row's selections (slot order) of their partials; one
// thread per (row, head, 4 dims).
__global__ void __launch_bounds__(256)
    k_attn_bwd_dq_merge(const int32_t* __restrict__ idx, const __nv_bfloat16* __restrict__ part_dq,
                        float* __restrict__ dq, int64_t N, int H_kv, int G, int d_h, int kk,
                        float scale) {
  const int64_t x = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int q4 = d_h / 4;
  if (x >= N * H_kv * G * q4) return;
  const int d4 = (int)(x % q4);
  const int64_t ih = x / q4;                     // i * H_q + h
  const int H_q = H_kv * G;
  const int64_t i = ih / H_q;
  const int h = (int)(ih - i * H_q);
  const int r = h / G, hg = h - r * G;
  const int32_t* sel = idx + ((int64_t)r * N + i) * kk;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int t = 0; t < kk; ++t) {
    const int b = __ldg(sel + t);
    if (b < 0 || (int64_t)b > (i >> 6)) continue;
    const uint2 v = __ldg(reinterpret_cast<const uint2*>(
                        part_dq + ((((int64_t)r * N + i) * kk + t) * G + hg) * d_h) + d4);
    const float2 f0 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&v.x));
    const float2 f1 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&v.y));
    acc.x += f0.x;
    acc.y += f0.y;
    acc.z += f1.x;
    acc.w += f1.y;
  }
  reinterpret_cast<float4*>(dq + ih * d_h)[d4] =
      make_float4(acc.x * scale, acc.y * scale, acc.z * scale, acc.w * scale);
}

// dk / dv [N, H_kv, d_h] of block b of group r: the sum over the bucket's pieces (piece order)
// of their dK^T / dV^T partials; zeros for tokens no query selected.  One thread per
// (bucket, dim, 4 keys).
__global__ void __launch_bounds__(256)
    k_attn_bwd_dkv_merge(const int* __restrict__ piece_off, const float* __restrict__ part_dkv,
                         float* __restrict__ dk, float* __restrict__ dv, int64_t N, int H_kv,
                         int nblk, int d_h, float scale) {
  const int64_t x = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t per_b = (int64_t)d_h * 16;
  if (x >= (int64_t)H_kv * nblk * per_b) return;
  const int bkt = (int)(x / per_b);
  const int rem = (int)(x - (int64_t)bkt * per_b);
  const int dim = rem / 16, k4 = rem - dim * 16;
  const int r = bkt / nblk, blk = bkt - r * nblk;
  float4 sk = make_float4(0.f, 0.f, 0.f, 0.f), sv = sk;
  for (int p = __ldg(piece_off + bkt); p < __ldg(piece_off + bkt + 1); ++p) {
    const float* base = part_dkv + (int64_t)p * 2 * d_h * 64;
    const float4 a = __ldg(reinterpret_cast<const float4*>(base + dim * 64) + k4);
    const float4 c = __ldg(reinterpret_cast<const float4*>(base + (d_h + dim) * 64) + k4);
    sk.x += a.x; sk.y += a.y; sk.z += a.z; sk.w += a.w;
    sv.x += c.x; sv.y += c.y; sv.z += c.z; sv.w += c.w;
  }
  const float ks[4] = {sk.x, sk.y, sk.z, sk.w}, vs[4] = {sv.x, sv.y, sv.z, sv.w};
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const int64_t tok = (int64_t)blk * kBlock + 4 * k4 + u;
    if (tok >= N) break;
    const int64_t o = (tok * H_kv + r) * d_h + dim;
    dk[o] = ks[u] * scale;
    dv[o] = vs[u];
  }
}

struct BwdWs {
  size_t count, offset, tile_off, cursor, piece_off, cnt_mat, entries, delta, part_dq, part_dkv,
      total;
  int nb;
};

size_t a256(size_t x) { return (x + 255) & ~size_t(255); }

BwdWs bwd_layout(int64_t N, int H_q, int H_kv, int d_h, int kk) {
  BwdWs w{};
  const int G = H_q / H_kv;
  const int64_t nblk = (N + kBlock - 1) / kBlock;
  w.nb = (int)(H_kv * nblk);
  const size_t sel = (size_t)H_kv * N * kk;
  const size_t ept = (size_t)(kRowsB / G);
  // pieces <= sum_b (tiles_b / kPiece + 1) and tiles_b <= count_b / ept + 1
  const size_t pieces = 2 * (size_t)w.nb + sel / (ept * kPiece) + 1;
  size_t off = 0;
  auto take = [&](size_t bytes) { const size_t o = off; off = a256(off + bytes); return o; };
  w.count = take(4 * (size_t)(w.nb + 1));
  w.offset = take(4 * (size_t)(w.nb + 1));
  w.tile_off = take(4 * (size_t)(w.nb + 1));
  w.cursor = take(4 * (size_t)(w.nb + 1));
  w.piece_off = take(4 * (size_t)(w.nb + 1));
  w.cnt_mat = take(4 * (size_t)w.nb * ordered_bucket_ranges(N));
  w.entries = take(4 * sel);
  w.delta = take(4 * (size_t)H_q * N);
  w.part_dq = take(2 * sel * G * d_h);
  w.part_dkv = take(4 * pieces * 2 * d_h * 64);
  w.total = off;
  return w;
}

}  // namespace

size_t sparse_attn_bwd_ws_bytes(int64_t N, int H_q, int H_kv, int d_h, int kk) {
  return bwd_layout(N, H_q, H_kv, d_h, kk).total;
}

cudaError_t launch_sparse_attn_bwd(const void* q, const void* k, const void* v, const int32_t* idx,
                                   const void* o, const float* lse, const void* d_o, float* dq,
                                   float* dk, float* dv, int64_t N, int H_q, int H_kv, int d_h,
                                   int kk, void* ws, cudaStream_t st) {
  const BwdWs w = bwd_layout(N, H_q, H_kv, d_h, kk);
  const int G = H_q / H_kv;
  const int64_t nblk = (N + kBlock - 1) / kBlock;
  char* base = static_cast<char*>(ws);
  int* count = reinterpret_cast<int*>(base + w.count);
  int* offset = reinterpret_cast<int*>(base + w.offset);
  int* tile_off = reinterpret_cast<int*>(base + w.tile_off);
  int* cursor = reinterpret_cast<int*>(base + w.cursor);
  int* piece_off = reinterpret_cast<int*>(base + w.piece_off);
  int* cnt_mat = reinterpret_cast<int*>(base + w.cnt_mat);
  int* entries = reinterpret_cast<int*>(base + w.entries);
  float* delta = reinterpret_cast<float*>(base + w.delta);
  auto* part_dq = reinterpret_cast<__nv_bfloat16*>(base + w.part_dq);
  float* part_dkv = reinterpret_cast<float*>(base + w.part_dkv);
  const auto* qq = static_cast<const __nv_bfloat16*>(q);
  const auto* dd = static_cast<const __nv_bfloat16*>(d_o);

  // row-ordered buckets: the work tiles, and so the order of every dK / dV sum, are the same on
  // every call
  cudaError_t e = launch_bucket_selections_ordered(idx, N, H_kv, kk, kRowsB / G, count, offset,
                                                   tile_off, cursor, cnt_mat, entries, st);
  if (e != cudaSuccess) return e;
  k_attn_bwd_pieces<<<1, kScanB, 0, st>>>(tile_off, piece_off, w.nb);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  {
    const int64_t warps = N * H_q;
    k_attn_bwd_delta<<<(unsigned)((warps * 32 + 255) / 256), 256, 0, st>>>(
        static_cast<const __nv_bfloat16*>(o), dd, delta, N, H_q, d_h);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  CUtensorMap tq, tdo, tk, tv;
  if ((e = make_tma_3d_bf16(&tq, q, (uint64_t)d_h, (uint64_t)H_q, (uint64_t)N, 64, G, 1, 128)) !=
      cudaSuccess)
    return e;
  if ((e = make_tma_3d_bf16(&tdo, d_o, (uint64_t)d_h, (uint64_t)H_q, (uint64_t)N, 64, G, 1, 128)) !=
      cudaSuccess)
    return e;
  if ((e = make_tma_3d_bf16(&tk, k, (uint64_t)d_h, (uint64_t)H_kv, (uint64_t)N, 64, 1, 64, 128)) !=
      cudaSuccess)
    return e;
  if ((e = make_tma_3d_bf16(&tv, v, (uint64_t)d_h, (uint64_t)H_kv, (uint64_t)N, 64, 1, 64, 128)) !=
      cudaSuccess)
    return e;
  // the dQ partials as [H_kv * N * k slots, G, d_h]: one box = one selection's G heads x 64 dims
  CUtensorMap tdq;
  if ((e = make_tma_3d_bf16(&tdq, part_dq, (uint64_t)d_h, (uint64_t)G, (uint64_t)H_kv * N * kk, 64,
                            G, 1, 128)) != cudaSuccess)
    return e;
  int dev = 0, sms = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
    return e;
  BwdArgs args{qq, dd, lse, delta, entries, offset, tile_off, piece_off, part_dq, part_dkv, N,
               w.nb, (int)nblk, H_kv, kk,
               (float)(1.4426950408889634 / std::sqrt((double)d_h))};
  auto run = [&](auto kern, int smem) -> cudaError_t {
    cudaError_t x = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (x != cudaSuccess) return x;
    kern<<<sms, kThreadsB, smem, st>>>(tq, tdo, tk, tv, tdq, args);
    return cudaGetLastError();
  };
  auto dispatch = [&](auto dh) -> cudaError_t {
    constexpr int D = decltype(dh)::value;
    constexpr int S = BwdSmem<D>::kAlloc;
    switch (G) {
      case 1: return run(k_attn_bwd_kvouter<D, 1>, S);
      case 2: return run(k_attn_bwd_kvouter<D, 2>, S);
      case 4: return run(k_attn_bwd_kvouter<D, 4>, S);
      default: return run(k_attn_bwd_kvouter<D, 8>, S);
    }
  };
  e = d_h == 128 ? dispatch(std::integral_constant<int, 128>())
                 : dispatch(std::integral_constant<int, 64>());
  if (e != cudaSuccess) return e;
  const float scale = (float)(1.0 / std::sqrt((double)d_h));
  {
    const int64_t n = N * H_q * (d_h / 4);
    k_attn_bwd_dq_merge<<<(unsigned)((n + 255) / 256), 256, 0, st>>>(idx, part_dq, dq, N, H_kv, G,
                                                                    d_h, kk, scale);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  {
    const int64_t n = (int64_t)w.nb * d_h * 16;
    k_attn_bwd_dkv_merge<<<(unsigned)((n + 255) / 256), 256, 0, st>>>(piece_off, part_dkv, dk, dv,
                                                                     N, H_kv, (int)nblk, d_h,
                                                                     scale);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  return cudaSuccess;
}

cudaError_t read_reset_bwd_status(unsigned* out) {
  unsigned zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(out, g_bwd_status, sizeof(unsigned));
  if (e != cudaSuccess) return e;
  return cudaMemcpyToSymbol(g_bwd_status, &zero, sizeof(unsigned));
}

}  // namespace msa

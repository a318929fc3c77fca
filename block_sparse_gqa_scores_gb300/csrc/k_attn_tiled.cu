// Shared-block pass of the sparse main branch («MiniMax-M3：MSA 技术报告速读», section 主分支,
// eq. O^(h)_i, and the LSE of section Kernel): the KV blocks that two or more queries of an
// 8-query tile selected are read from L2 once for the tile.  Blocks only one query selected go
// to the block-major pass (k_attn_kvouter.cu); k_attn_merge combines both kinds of partial.
//
// One CTA = 8 consecutive queries of one KV group r: 8 consumer warps (warp w owns query
// i0+w and its G <= 8 heads) and one TMA producer warp.
//   1. The producer warp forms the union of the 8 queries' selected blocks with a per-block mask
//      of the queries that selected it (attn_tile.cuh) and keeps the blocks with >= 2 users.
//   2. It streams them as 32-token half blocks (K and V of group r, a 3-D tensor map over
//      [N, H_kv, d_h] with 128-byte swizzle) through a 6-stage ring.  When it fills a stage it
//      arrives on the stage's "empty" barrier on behalf of every warp whose query did not
//      select the block, so each consumer touches only its own stages.  Because a consumer may
//      skip whole ring turns, it first waits for the producer's count of issued stages to pass
//      its stage: the previous turn of that slot has then landed and been released, and the
//      next turn cannot be issued before this consumer releases it, so the slot's "full"
//      parity names exactly one turn.
//   3. A consumer computes on the blocks its query selected: S^T = K Q^T and O^T += V^T P^T
//      as m16n8k16 MMAs with the group's heads on N = 8, operands by ldmatrix /
//      ldmatrix.trans from the swizzled tiles, online softmax in the log2 domain.
//   4. Each warp writes its query's partial: O normalised by its own sum (bf16, [G, d_h]) and
//      the log2-domain LSE (-inf when the query shares no block with its tile).
// All mbarrier waits are bounded; a timeout sets the device status word and ends the loop.
#include <climits>
#include <cmath>

#include "attn_tile.cuh"
#include "msa_internal.h"

namespace msa {
namespace {

__device__ unsigned g_attn_status = 0;

constexpr int kQT = 8;                  // queries per CTA (one consumer warp each)
constexpr int kStages = 6;              // ring depth in half blocks
constexpr int kHalf = 32;               // tokens per stage
constexpr int kMaxK = 64;
constexpr int kThreads = 32 * (kQT + 1);
constexpr unsigned kFull = 0xffffffffu;

template <int D_H>
struct TiledSmem {
  static constexpr int kBoxBytes = kHalf * 128;           // 32 rows x 64 dims, 128-B swizzle
  static constexpr int kBoxes = D_H / 64;                 // 64-dim boxes per row
  static constexpr int kKBytes = kBoxes * kBoxBytes;
  static constexpr int kStageBytes = 2 * kKBytes;         // K boxes then V boxes
  static constexpr int kOffU = kStages * kStageBytes;
  static constexpr int kOffMask = kOffU + kQT * kMaxK * 4;
  static constexpr int kOffBar = kOffMask + kQT * kMaxK * 4;
  static constexpr int kOffMisc = kOffBar + 2 * kStages * 8;     // nU, issued-stage count
  static constexpr int kBytes = kOffMisc + 16;
  static constexpr int kAlloc = kBytes + 1024;
};

template <int EPL>
__device__ __forceinline__ int union_of(const int32_t* __restrict__ idx, int r, int64_t i0,
                                       int64_t i_end, int64_t N, int kk, int* s_U,
                                       unsigned* s_mask) {
  int x[EPL], rank[EPL];
  return tile_union<EPL>(idx, r, i0, i_end, N, kk, x, rank, s_U, s_mask);
}

template <int D_H>
__global__ void __launch_bounds__(kThreads, 2)
    k_sparse_attn_tiled(const __grid_constant__ CUtensorMap tm_k,
                        const __grid_constant__ CUtensorMap tm_v,
                        const __nv_bfloat16* __restrict__ q, const int32_t* __restrict__ idx,
                        __nv_bfloat16* __restrict__ tp_o, float* __restrict__ tp_lse, int64_t N,
                        int64_t q0, int64_t q1, int H_q, int G, int kk, int64_t ntiles,
                        float scale_log2) {
  using L = TiledSmem<D_H>;
  constexpr int KS = D_H / 16;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t sbase = smem_u32(smem);
  int* s_U = reinterpret_cast<int*>(smem + L::kOffU);
  unsigned* s_mask = reinterpret_cast<unsigned*>(smem + L::kOffMask);
  int* s_nU = reinterpret_cast<int*>(smem + L::kOffMisc);
  int* s_issued = s_nU + 1;
  const uint32_t bar0 = sbase + L::kOffBar;
  auto full = [&](int s) { return bar0 + 8u * s; };
  auto empty = [&](int s) { return bar0 + 8u * (kStages + s); };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t bid = blockIdx.x;
  const int r = (int)(bid / ntiles);
  const int64_t i0 = q0 + (bid - (int64_t)r * ntiles) * kQT;

  // ---- 1. the tile's shared blocks (producer warp), barrier init
  if (warp == kQT) {
    int nU;
    if (kk <= 4) nU = union_of<1>(idx, r, i0, q1, N, kk, s_U, s_mask);
    else if (kk <= 8) nU = union_of<2>(idx, r, i0, q1, N, kk, s_U, s_mask);
    else if (kk <= 16) nU = union_of<4>(idx, r, i0, q1, N, kk, s_U, s_mask);
    else if (kk <= 32) nU = union_of<8>(idx, r, i0, q1, N, kk, s_U, s_mask);
    else nU = union_of<16>(idx, r, i0, q1, N, kk, s_U, s_mask);
    int nS = 0;                                       // keep blocks with two or more users
    for (int base = 0; base < nU; base += 32) {
      const int u = base + lane;
      const int bu = u < nU ? s_U[u] : 0;
      const unsigned mu = u < nU ? s_mask[u] : 0u;
      const bool keep = __popc(mu) >= 2;
      const unsigned kb = __ballot_sync(kAllLanes, keep);
      __syncwarp();
      if (keep) {
        const int pos = nS + __popc(kb & ((1u << lane) - 1u));
        s_U[pos] = bu;
        s_mask[pos] = mu;
      }
      nS += __popc(kb);
      __syncwarp();
    }
    if (lane == 0) {
      *s_nU = nS;
      *s_issued = 0;
      for (int s = 0; s < kStages; ++s) {
        mbar_init(full(s), 1);
        mbar_init(empty(s), kQT);
      }
      fence_barrier_init();
    }
  }
  __syncthreads();
  const int nU = *s_nU;
  const int nst = 2 * nU;               // stage sequence: two half blocks per union block

  if (warp == kQT) {
    // -------------------------------------------------------------- producer
    if (lane == 0) {
      prefetch_tensormap(&tm_k);
      prefetch_tensormap(&tm_v);
      int last_round[kStages];
      for (int s = 0; s < kStages; ++s) last_round[s] = -1;
      for (int qd = 0; qd < nst; ++qd) {
        const int s = qd % kStages, round = qd / kStages;
        if (!mbar_wait(empty(s), (round & 1) ^ 1, &g_attn_status)) break;
        // the warps whose query did not select this block release the stage up front
        const int users = __popc(s_mask[qd >> 1]);
        if (users < kQT) mbar_arrive_cnt(empty(s), (uint32_t)(kQT - users));
        const int tok = s_U[qd >> 1] * kBlock + (qd & 1) * kHalf;
        const uint32_t dst = sbase + s * L::kStageBytes;
        mbar_expect_tx(full(s), L::kStageBytes);
#pragma unroll
        for (int bx = 0; bx < L::kBoxes; ++bx) {
          tma_load_3d(dst + bx * L::kBoxBytes, &tm_k, full(s), 64 * bx, r, tok);
          tma_load_3d(dst + L::kKBytes + bx * L::kBoxBytes, &tm_v, full(s), 64 * bx, r, tok);
        }
        last_round[s] = round;
        *reinterpret_cast<volatile int*>(s_issued) = qd + 1;
      }
      for (int s = 0; s < kStages; ++s)            // no copy may be in flight at exit
        if (last_round[s] >= 0) mbar_wait(full(s), last_round[s] & 1, &g_attn_status);
    }
    return;
  }

  // ------------------------------------------------------------------ consumers
  const int c = lane & 3, r4 = lane >> 2;
  const int64_t i = i0 + warp;
  const bool valid = i < q1;
  const int hq0 = r * G;

  uint32_t qf[KS][2];
  {
    const bool hv = valid && r4 < G;
    const uint32_t* qh =
        reinterpret_cast<const uint32_t*>(q + (i * H_q + hq0 + (hv ? r4 : 0)) * D_H);
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
      qf[ks][0] = hv ? qh[8 * ks + c] : 0u;
      qf[ks][1] = hv ? qh[8 * ks + 4 + c] : 0u;
    }
  }
  float oacc[KS][4];
#pragma unroll
  for (int mt = 0; mt < KS; ++mt)
#pragma unroll
    for (int e = 0; e < 4; ++e) oacc[mt][e] = 0.f;
  float m_run[2] = {-INFINITY, -INFINITY};
  float l_run[2] = {0.f, 0.f};

  // per-lane ldmatrix row offsets inside a 32-row swizzled box
  const int krow_a = (lane & 7) + 8 * ((lane >> 3) & 1);   // S^T A operand (K rows)
  const int kchk_a = lane >> 4;
  const int vrow_b = (lane & 7) + 8 * (lane >> 4);          // O^T A operand (V rows, trans)
  const int vchk_b = (lane >> 3) & 1;

  bool ok = valid;
  for (int qd = 0; qd < nst && ok; ++qd) {
    const int u = qd >> 1;
    if (!((s_mask[u] >> warp) & 1u)) continue;      // stage released by the producer
    const int s = qd % kStages, round = qd / kStages;
    if (!wait_counter_above(s_issued, qd, &g_attn_status) ||
        !mbar_wait(full(s), round & 1, &g_attn_status)) {
      ok = false;
      break;
    }
    {
      const int64_t j0 = (int64_t)s_U[u] * kBlock + (qd & 1) * kHalf;
      const uint32_t kb = sbase + s * L::kStageBytes;
      const uint32_t vb = kb + L::kKBytes;

      float sacc[2][4];
#pragma unroll
      for (int mt = 0; mt < 2; ++mt) {
#pragma unroll
        for (int e = 0; e < 4; ++e) sacc[mt][e] = 0.f;
        const int kr = 16 * mt + krow_a;
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
          const int chunk = 2 * (ks & 3) + kchk_a;
          uint32_t a[4];
          ldmatrix_x4(a, kb + (ks >> 2) * L::kBoxBytes + kr * 128 + ((chunk ^ (kr & 7)) << 4));
          mma_16816(sacc[mt], a, qf[ks][0], qf[ks][1]);
        }
      }
      float x[2][4];
#pragma unroll
      for (int mt = 0; mt < 2; ++mt) {
        const int64_t jlo = j0 + 16 * mt + r4, jhi = jlo + 8;
        x[mt][0] = jlo <= i ? sacc[mt][0] * scale_log2 : -INFINITY;
        x[mt][1] = jlo <= i ? sacc[mt][1] * scale_log2 : -INFINITY;
        x[mt][2] = jhi <= i ? sacc[mt][2] * scale_log2 : -INFINITY;
        x[mt][3] = jhi <= i ? sacc[mt][3] * scale_log2 : -INFINITY;
      }
      float p[2][4];
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        float mb = fmax3(x[0][hh], x[0][hh + 2], fmaxf(x[1][hh], x[1][hh + 2]));
        mb = fmaxf(mb, __shfl_xor_sync(kFull, mb, 4));
        mb = fmaxf(mb, __shfl_xor_sync(kFull, mb, 8));
        mb = fmaxf(mb, __shfl_xor_sync(kFull, mb, 16));
        const float m_new = fmaxf(m_run[hh], mb);
        float alpha = 1.f;
        if (m_new == -INFINITY) {
          p[0][hh] = p[0][hh + 2] = p[1][hh] = p[1][hh + 2] = 0.f;
        } else {
          alpha = ex2(m_run[hh] - m_new);
          p[0][hh] = ex2(x[0][hh] - m_new);
          p[0][hh + 2] = ex2(x[0][hh + 2] - m_new);
          p[1][hh] = ex2(x[1][hh] - m_new);
          p[1][hh + 2] = ex2(x[1][hh + 2] - m_new);
        }
        m_run[hh] = m_new;
        l_run[hh] = l_run[hh] * alpha + (p[0][hh] + p[0][hh + 2]) + (p[1][hh] + p[1][hh + 2]);
#pragma unroll
        for (int mt = 0; mt < KS; ++mt) {
          oacc[mt][hh] *= alpha;
          oacc[mt][hh + 2] *= alpha;
        }
      }
      uint32_t pb[2][2];
#pragma unroll
      for (int mt = 0; mt < 2; ++mt) {
        pb[mt][0] = movmatrix_trans(pack_bf16x2(p[mt][0], p[mt][1]));   // keys 16mt + 0..7
        pb[mt][1] = movmatrix_trans(pack_bf16x2(p[mt][2], p[mt][3]));   // keys 16mt + 8..15
      }
#pragma unroll
      for (int mtd = 0; mtd < KS; ++mtd) {
        const int chunk = 2 * mtd + vchk_b;
        const int bx = chunk >> 3, cc = chunk & 7;
#pragma unroll
        for (int k2 = 0; k2 < 2; ++k2) {
          const int vr = 16 * k2 + vrow_b;
          uint32_t a[4];
          ldmatrix_x4_trans(a, vb + bx * L::kBoxBytes + vr * 128 + ((cc ^ (vr & 7)) << 4));
          mma_16816(oacc[mtd], a, pb[k2][0], pb[k2][1]);
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(empty(s));
  }

  // ---- epilogue: this warp's query
  float inv[2], lsum[2];
#pragma unroll
  for (int hh = 0; hh < 2; ++hh) {
    float t = l_run[hh];
    t += __shfl_xor_sync(kFull, t, 4);
    t += __shfl_xor_sync(kFull, t, 8);
    t += __shfl_xor_sync(kFull, t, 16);
    lsum[hh] = t;
    inv[hh] = t > 0.f ? 1.f / t : 0.f;
  }
  if (valid) {
    const int64_t unit = (int64_t)r * (q1 - q0) + (i - q0);   // partial row of this query
    if (r4 == 0) {
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const int h = 2 * c + hh;
        if (h < G) tp_lse[unit * G + h] = lsum[hh] > 0.f ? m_run[hh] + __log2f(lsum[hh]) : -INFINITY;
      }
    }
    uint32_t* orow = reinterpret_cast<uint32_t*>(tp_o + (unit * G + (r4 < G ? r4 : 0)) * D_H);
#pragma unroll
    for (int mtd = 0; mtd < KS; ++mtd) {
      const uint32_t lo = movmatrix_trans(pack_bf16x2(oacc[mtd][0] * inv[0], oacc[mtd][1] * inv[1]));
      const uint32_t hi = movmatrix_trans(pack_bf16x2(oacc[mtd][2] * inv[0], oacc[mtd][3] * inv[1]));
      if (r4 < G) {
        orow[8 * mtd + c] = lo;          // dims 16mtd + 2c, +1
        orow[8 * mtd + 4 + c] = hi;      // dims 16mtd + 8 + 2c, +1
      }
    }
  }
}

template <int D_H>
cudaError_t launch_tiled(const CUtensorMap& tk, const CUtensorMap& tv, const void* q,
                         const int32_t* idx, void* tp_o, float* tp_lse, int64_t N, int64_t q0,
                         int64_t q1, int H_q, int H_kv, int kk, cudaStream_t stream) {
  using L = TiledSmem<D_H>;
  auto kern = k_sparse_attn_tiled<D_H>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kAlloc);
  if (e != cudaSuccess) return e;
  const int64_t ntiles = (q1 - q0 + kQT - 1) / kQT;
  const float scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)D_H));
  kern<<<(unsigned)(ntiles * H_kv), kThreads, L::kAlloc, stream>>>(
      tk, tv, static_cast<const __nv_bfloat16*>(q), idx, static_cast<__nv_bfloat16*>(tp_o), tp_lse,
      N, q0, q1, H_q, H_q / H_kv, kk, ntiles, scale_log2);
  return cudaGetLastError();
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

constexpr int64_t kChunkRows = 16384;     // query rows per pass (bounds the workspace)

struct AttnWs {
  size_t count, offset, tile_off, cursor, entries, slotmap, part_o, part_lse, tp_o, tp_lse, total;
  int64_t qc;
  int nb;
};

AttnWs attn_layout(int64_t N, int H_q, int H_kv, int d_h, int kk) {
  AttnWs w{};
  const int G = H_q / H_kv;
  w.qc = ((N < kChunkRows ? N : kChunkRows) + kQT - 1) / kQT * kQT;
  const int64_t nblk = (N + kBlock - 1) / kBlock;
  w.nb = (int)(H_kv * nblk);
  const size_t sel = (size_t)H_kv * w.qc * kk;            // selections of one chunk
  size_t off = 0;
  auto take = [&](size_t bytes) { const size_t o = off; off = align256(off + bytes); return o; };
  w.count = take(4 * (size_t)(w.nb + 1));
  w.offset = take(4 * (size_t)(w.nb + 1));
  w.tile_off = take(4 * (size_t)(w.nb + 1));
  w.cursor = take(4 * (size_t)(w.nb + 1));
  w.entries = take(4 * sel);
  w.slotmap = take(4 * sel);
  w.part_o = take(2 * sel * G * d_h);
  w.part_lse = take(4 * sel * G);
  w.tp_o = take(2 * (size_t)H_kv * w.qc * G * d_h);
  w.tp_lse = take(4 * (size_t)H_kv * w.qc * G);
  w.total = off;
  return w;
}

}  // namespace

size_t sparse_attn_ws_bytes(int64_t N, int H_q, int H_kv, int d_h, int kk) {
  return attn_layout(N, H_q, H_kv, d_h, kk).total;
}

// The main branch over query chunks: plan (count) -> scan -> plan (scatter) -> block-major pass
// over private selections -> shared-block pass -> merge.  Everything is enqueued on `stream`.
cudaError_t launch_sparse_attn_fwd(const void* q, const void* k, const void* v, const int32_t* idx,
                                   void* o, float* lse, int64_t N, int H_q, int H_kv, int d_h,
                                   int kk, void* ws, cudaStream_t stream) {
  const AttnWs w = attn_layout(N, H_q, H_kv, d_h, kk);
  char* base = static_cast<char*>(ws);
  int* count = reinterpret_cast<int*>(base + w.count);
  int* offset = reinterpret_cast<int*>(base + w.offset);
  int* tile_off = reinterpret_cast<int*>(base + w.tile_off);
  int* cursor = reinterpret_cast<int*>(base + w.cursor);
  int* entries = reinterpret_cast<int*>(base + w.entries);
  int* slotmap = reinterpret_cast<int*>(base + w.slotmap);
  void* part_o = base + w.part_o;
  float* part_lse = reinterpret_cast<float*>(base + w.part_lse);
  void* tp_o = base + w.tp_o;
  float* tp_lse = reinterpret_cast<float*>(base + w.tp_lse);

  CUtensorMap tk, tv;
  cudaError_t e = make_tma_3d_bf16(&tk, k, (uint64_t)d_h, (uint64_t)H_kv, (uint64_t)N, 64, 1, kHalf, 128);
  if (e != cudaSuccess) return e;
  e = make_tma_3d_bf16(&tv, v, (uint64_t)d_h, (uint64_t)H_kv, (uint64_t)N, 64, 1, kHalf, 128);
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 148;
  if (cudaGetDevice(&dev) == cudaSuccess)
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int64_t nblk = (N + kBlock - 1) / kBlock;
  const int G = H_q / H_kv;
  for (int64_t q0 = 0; q0 < N; q0 += w.qc) {
    const int64_t q1 = q0 + w.qc < N ? q0 + w.qc : N;
    if ((e = cudaMemsetAsync(count, 0, 4 * (size_t)w.nb, stream)) != cudaSuccess) return e;
    if ((e = launch_attn_plan(idx, N, H_kv, kk, q0, q1, q1 - q0, nblk, 0, count, offset, cursor,
                              entries, slotmap, stream)) != cudaSuccess) return e;
    if ((e = launch_attn_scan(count, offset, tile_off, cursor, w.nb, 128 / G, stream)) != cudaSuccess)
      return e;
    if ((e = launch_attn_plan(idx, N, H_kv, kk, q0, q1, q1 - q0, nblk, 1, count, offset, cursor,
                              entries, slotmap, stream)) != cudaSuccess) return e;
    if ((e = launch_attn_kvouter(q, k, v, entries, offset, tile_off, w.nb, nblk, N, q0, H_q, H_kv,
                                 d_h, 2 * sms, part_o, part_lse, stream)) != cudaSuccess) return e;
    e = d_h == 128 ? launch_tiled<128>(tk, tv, q, idx, tp_o, tp_lse, N, q0, q1, H_q, H_kv, kk, stream)
                   : launch_tiled<64>(tk, tv, q, idx, tp_o, tp_lse, N, q0, q1, H_q, H_kv, kk, stream);
    if (e != cudaSuccess) return e;
    if ((e = launch_attn_merge(tp_o, tp_lse, slotmap, part_o, part_lse, o, lse, N, H_q, H_kv, d_h,
                               kk, q0, q1, stream)) != cudaSuccess) return e;
  }
  return cudaSuccess;
}

cudaError_t read_reset_attn_status(unsigned* out) {
  unsigned zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(out, g_attn_status, sizeof(unsigned));
  if (e != cudaSuccess) return e;
  return cudaMemcpyToSymbol(g_attn_status, &zero, sizeof(unsigned));
}

}  // namespace msa

// Decode index branch: for one new query per sequence, block scores of the whole cache
// («MiniMax-M3：MSA 技术报告速读», section 索引分支, eqs. S^idx and M^idx at row i = L-1).
//
// This is the byte-dominant part of decode: the shared index key cache is streamed once
// (128 B per token at d_idx = 64).  The grid is (chunk of 1024 tokens, sequence); chunks past
// a sequence's end exit at once.  Each warp takes whole 64-token blocks; the dot products of
// 16 tokens with the H_kv <= 8 index heads are one m16n8k16 MMA per 16 dims (tokens on M,
// heads on N), with the index-key rows loaded from global memory straight into A fragments
// as 16-byte vectors (the contracted dim is permuted the same way in the q_idx fragment).
// Every token of the cache is visible to the last row, so only the cache end is masked.  The
// cache is packed or paged (CacheMap): a 64-token block is contiguous either way, so a warp finds
// the cache row of its block once and reads the block's rows from there.
#include <math.h>

#include "msa_device.cuh"
#include "msa_internal.h"

namespace msa {
namespace {

constexpr int kDecWarps = 4;
constexpr int kChunkTokens = 1024;
constexpr unsigned kFull = 0xffffffffu;

template <int D_IDX, bool PAGED>
__global__ void __launch_bounds__(32 * kDecWarps)
    k_decode_block_scores(const __nv_bfloat16* __restrict__ q_idx,
                          const __nv_bfloat16* __restrict__ k_idx, const CacheMap cm,
                          float* __restrict__ Mdec, int H_kv, int64_t max_len, int64_t nblk_max,
                          float scale) {
  constexpr int KS = D_IDX / 16;           // k-steps
  constexpr int KCH = D_IDX / 32;          // 16-B chunks per thread per token row
  pdl_launch_dependents();                 // the selection may be scheduled under this grid's tail
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int c = lane & 3, r4 = lane >> 2;
  const int64_t s = blockIdx.y;
  const int64_t L = cm.len<PAGED>(s, max_len);
  const __nv_bfloat16* kseq = k_idx + cm.seq_row<PAGED>(s) * D_IDX;   // packed: the sequence
  const int64_t first = (int64_t)blockIdx.x * kChunkTokens;
  if (first >= L) return;
  const int64_t last_blk = (L - 1) >> 6;

  // q_idx^T fragments: head n = r4 (zero beyond H_kv), dims permuted like the key loads
  uint32_t qf[KS][2];
  {
    const bool valid = r4 < H_kv;
    const uint32_t* qh = reinterpret_cast<const uint32_t*>(q_idx + (s * H_kv + r4) * D_IDX);
#pragma unroll
    for (int ks = 0; ks < KS; ++ks)
#pragma unroll
      for (int hl = 0; hl < 2; ++hl) {
        const int t = 2 * ks + hl;
        const int d = 8 * (c + 4 * (t >> 2)) + 2 * (t & 3);
        qf[ks][hl] = valid ? qh[d >> 1] : 0u;
      }
  }
  for (int64_t b = (first >> 6) + warp; b <= last_blk && b < ((first + kChunkTokens) >> 6);
       b += kDecWarps) {
    float best[2] = {-INFINITY, -INFINITY};          // heads 2c, 2c+1
    // token rows: packed, from the sequence's first row; paged, from the block's page
    const __nv_bfloat16* kb =
        PAGED ? k_idx + (cm.block_row<true>(s, b, 0) - b * kBlock) * D_IDX : kseq;
#pragma unroll
    for (int mt = 0; mt < 4; ++mt) {
      const int64_t jlo = b * kBlock + 16 * mt + r4, jhi = jlo + 8;
      const bool vlo = jlo < L, vhi = jhi < L;
      uint4 kr[2][KCH];
#pragma unroll
      for (int u = 0; u < KCH; ++u) {
        kr[0][u] = vlo ? ldg_nc_v4(kb + jlo * D_IDX + 8 * (c + 4 * u)) : make_uint4(0, 0, 0, 0);
        kr[1][u] = vhi ? ldg_nc_v4(kb + jhi * D_IDX + 8 * (c + 4 * u)) : make_uint4(0, 0, 0, 0);
      }
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int ks = 0; ks < KS; ++ks) {
        const int t0 = 2 * ks, t1 = 2 * ks + 1;
        uint32_t a[4];
        a[0] = reinterpret_cast<const uint32_t*>(&kr[0][t0 >> 2])[t0 & 3];
        a[1] = reinterpret_cast<const uint32_t*>(&kr[1][t0 >> 2])[t0 & 3];
        a[2] = reinterpret_cast<const uint32_t*>(&kr[0][t1 >> 2])[t1 & 3];
        a[3] = reinterpret_cast<const uint32_t*>(&kr[1][t1 >> 2])[t1 & 3];
        mma_16816(acc, a, qf[ks][0], qf[ks][1]);
      }
      best[0] = fmax3(best[0], vlo ? acc[0] : -INFINITY, vhi ? acc[2] : -INFINITY);
      best[1] = fmax3(best[1], vlo ? acc[1] : -INFINITY, vhi ? acc[3] : -INFINITY);
    }
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      float m = best[hh];
      m = fmaxf(m, __shfl_xor_sync(kFull, m, 4));
      m = fmaxf(m, __shfl_xor_sync(kFull, m, 8));
      m = fmaxf(m, __shfl_xor_sync(kFull, m, 16));
      best[hh] = m;
    }
    if (r4 == 0) {
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const int head = 2 * c + hh;
        if (head < H_kv) Mdec[(s * H_kv + head) * nblk_max + b] = best[hh] * scale;
      }
    }
  }
}

}  // namespace

cudaError_t launch_decode_block_scores(const void* q_idx, const void* k_idx_cache,
                                       const CacheMap& cm, float* Mdec, int S, int H_kv, int d_idx,
                                       int64_t max_len, int64_t nblk_max, cudaStream_t stream) {
  const dim3 grid((unsigned)((max_len + kChunkTokens - 1) / kChunkTokens), (unsigned)S);
  const float scale = (float)(1.0 / sqrt((double)d_idx));
  const auto* q = static_cast<const __nv_bfloat16*>(q_idx);
  const auto* kc = static_cast<const __nv_bfloat16*>(k_idx_cache);
  auto run = [&](auto kern) {
    kern<<<grid, 32 * kDecWarps, 0, stream>>>(q, kc, cm, Mdec, H_kv, max_len, nblk_max, scale);
  };
  if (cm.pages) {
    if (d_idx == 64) run(k_decode_block_scores<64, true>); else run(k_decode_block_scores<32, true>);
  } else {
    if (d_idx == 64) run(k_decode_block_scores<64, false>); else run(k_decode_block_scores<32, false>);
  }
  return cudaGetLastError();
}

}  // namespace msa

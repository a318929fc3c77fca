// Decode tail of MSA («MiniMax-M3：MSA 技术报告速读», section 索引分支 eq. I^(r)_i and section
// 主分支 eq. O^(h)_i with the LSE of section Kernel): for one new token per sequence, the per-group
// top-k selection over the block scores the index-key scan wrote, then exact softmax attention of
// the group's G query heads over the visible tokens of the selected blocks, in one CTA per
// (sequence, group) -- no selection array, split partials or merge kernel between the stages.
//
//   selection   the row's candidate blocks are cut into segments, one per warp; each warp keeps
//               its segment's k-1 best (select_core.cuh), then warp 0 keeps the k-1 best of those
//               (exactly the single-warp selection) and appends the local block
//   attention   warps form quads; quad g takes the selected blocks g, g + kQuads, ...; warp w of a
//               quad owns keys [16w, 16w+16) of each of them.  The G <= 8 heads are the N=8 side of
//               the m16n8k16 MMA with the keys (S^T = K Q^T) or the head dims (O^T += V^T P^T) as
//               its M side; P goes from the S^T accumulator to the P^T operand with one movmatrix
//               transpose per 8x8 tile.  K and V rows are loaded from global memory straight into
//               MMA fragments as 16-byte vectors (the contracted head dim is permuted identically
//               in K and Q^T; V keys are paired with byte permutes, output rows un-permuted).
//               Online softmax per warp in the log2 domain
//   merge       the warps' (max, sum, O) states combined in shared memory in warp order, then O
//               (bf16) and the natural-log LSE written directly
// Results do not depend on timing: the selection is exact, and every sum runs in a fixed order.
#include <math.h>

#include "msa_internal.h"
#include "select_core.cuh"

namespace msa {
namespace {

constexpr int kTailWarps = 16;                 // 4 quads of 4 warps
// rows of at most this many candidate blocks (a 512K-token cache) are copied to shared memory
// before the selection, with every load in flight at once
constexpr int kRowCap = 8192;
constexpr int kQuads = kTailWarps / 4;
constexpr unsigned kFull = 0xffffffffu;

template <int D_H>
struct TailSmem {
  int cnt[kTailWarps];
  float tau[kTailWarps];                        // the segments' bounds on the (k-1)-th best
  int blocks[64];                               // the row's selection (ascending, -1 padded)
  float m[kTailWarps][8];
  float l[kTailWarps][8];
  union {                                       // selection scratch, then the warps' O states
    struct {
      sel::SelScratch sc[kTailWarps];
      float row[kRowCap];                       // the row's block scores
    } s;
    float o[kTailWarps][8][D_H];
  } u;
};

struct AttnParams {
  const __nv_bfloat16* q;
  const __nv_bfloat16* k;
  const __nv_bfloat16* v;
  const float* Mdec;  // block scores [S * H_kv, nblk_max]
  int32_t* idx_out;   // [S, H_kv, k] or null
  __nv_bfloat16* o;   // [S, H_q, D_H]
  float* lse;         // [S, H_q], natural log
  CacheMap cm;        // where each sequence's cache rows are (packed or paged)
  int64_t max_len;    // length bound
  int64_t nblk_max;
  int H_q, H_kv, G, kk, S;
  float scale_log2;   // log2(e) / sqrt(d_h)
};

template <int D_H, bool PAGED>
__global__ void __launch_bounds__(32 * kTailWarps) k_decode_tail(const AttnParams p) {
  constexpr int KS = D_H / 16;             // k-steps of S^T, m-tiles of O^T
  constexpr int KCH = D_H / 32;            // 16-B K chunks per thread per key row
  constexpr int VCH = D_H / 64;            // 16-B V chunks per thread per key
  extern __shared__ __align__(16) uint8_t tail_raw[];
  TailSmem<D_H>& sm = *reinterpret_cast<TailSmem<D_H>*>(tail_raw);
  pdl_launch_dependents();
  pdl_wait();                               // the block scores are written

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int c = lane & 3, r4 = lane >> 2;

  // ---------------------------------------------------------------- the problem
  const int64_t sr = blockIdx.x;            // (sequence, group)
  const int64_t s = sr / p.H_kv;
  const int r = (int)(sr - s * p.H_kv);
  const int64_t L = p.cm.len<PAGED>(s, p.max_len);
  const int64_t srow = p.cm.seq_row<PAGED>(s);
  const int64_t kv_stride = (int64_t)p.H_kv * D_H;          // elements between tokens
  const __nv_bfloat16* kseq = p.k + (srow * p.H_kv + r) * D_H;   // packed: the sequence's rows
  const __nv_bfloat16* vseq = p.v + (srow * p.H_kv + r) * D_H;
  const int64_t i = L - 1;                  // the new token's position
  const __nv_bfloat16* qrow = p.q + s * (int64_t)p.H_q * D_H;
  const int kk = p.kk;

  // ---------------------------------------------------------------- selection
  {
    const int64_t l = i >> 6;
    const float* Mrow = p.Mdec + sr * p.nblk_max;
    if (l + 1 <= kk) {
      for (int x = threadIdx.x; x < kk; x += 32 * kTailWarps) sm.blocks[x] = x <= l ? x : -1;
    } else {
      const int K1 = kk - 1, n = (int)l;
      int nseg = sel::kBuf / K1;
      nseg = nseg > kTailWarps ? kTailWarps : (nseg < 1 ? 1 : nseg);
      const int seg = (n + nseg - 1) / nseg;
      // the row's scores into shared memory, all loads of a thread issued together (the
      // segment passes below then read shared memory instead of one L2 round trip per step)
      const bool staged = n <= kRowCap;
      if (staged) {
        constexpr int kPer = kRowCap / (32 * kTailWarps);
        float v[kPer];
#pragma unroll
        for (int u = 0; u < kPer; ++u) {
          const int x = threadIdx.x + u * 32 * kTailWarps;
          v[u] = x < n ? __ldg(Mrow + x) : 0.f;
        }
#pragma unroll
        for (int u = 0; u < kPer; ++u) {
          const int x = threadIdx.x + u * 32 * kTailWarps;
          if (x < n) sm.u.s.row[x] = v[u];
        }
        __syncthreads();
      }
      // every segment's bound is a bound for the whole row: the largest of them lets each
      // segment keep only the blocks that can still be among the row's k-1 best, so warp 0
      // merges a few dozen candidates instead of k-1 per segment
      const int b0 = min(n, warp * seg), b1 = min(n, b0 + seg);
      if (warp < nseg) {
        const float t = b1 > b0 ? (staged ? sel::segment_bound<true>(sm.u.s.row, b0, b1, K1)
                                          : sel::segment_bound(Mrow, b0, b1, K1))
                                : -INFINITY;
        if (lane == 0) sm.tau[warp] = t;
      }
      __syncthreads();
      float tg = -INFINITY;
      for (int x = 0; x < nseg; ++x) tg = fmaxf(tg, sm.tau[x]);
      if (warp < nseg) {
        int cnt = 0;
        if (b1 > b0)
          cnt = staged
                    ? sel::select_segment_from<true>(sm.u.s.row, b0, b1, K1, tg, sm.u.s.sc[warp])
                    : sel::select_segment_from(Mrow, b0, b1, K1, tg, sm.u.s.sc[warp]);
        if (lane == 0) sm.cnt[warp] = cnt;
      }
      __syncthreads();
      if (warp == 0) {
        // the segments' survivors after warp 0's own, in segment (= block) order
        int cnt = sm.cnt[0];
        for (int w = 1; w < nseg; ++w) {
          const int cw = sm.cnt[w];
          for (int x = lane; x < cw; x += 32) {
            sm.u.s.sc[0].v[cnt + x] = sm.u.s.sc[w].v[x];
            sm.u.s.sc[0].b[cnt + x] = sm.u.s.sc[w].b[x];
          }
          cnt += cw;
        }
        __syncwarp();
        if (cnt > K1) {
          sel::compact(sm.u.s.sc[0], cnt, K1);
          cnt = K1;
        }
        for (int x = lane; x < K1; x += 32) sm.blocks[x] = x < cnt ? sm.u.s.sc[0].b[x] : -1;
        if (lane == 0) sm.blocks[K1] = (int32_t)l;
      }
    }
    __syncthreads();
    if (p.idx_out != nullptr)
      for (int x = threadIdx.x; x < kk; x += 32 * kTailWarps) p.idx_out[sr * kk + x] = sm.blocks[x];
  }
  const int quad = warp >> 2, wq = warp & 3;   // this warp: keys [16 wq, 16 wq + 16) of its blocks

  // Q^T fragments (B operand of S^T = K Q^T): head n = r4, dims permuted as the K loads.
  uint32_t qf[KS][2];
  {
    const bool valid = r4 < p.G;
    const uint32_t* qh = reinterpret_cast<const uint32_t*>(qrow + (int64_t)(r * p.G + r4) * D_H);
#pragma unroll
    for (int ks = 0; ks < KS; ++ks)
#pragma unroll
      for (int hl = 0; hl < 2; ++hl) {
        const int t = 2 * ks + hl;                       // fragment word index
        const int chunk = c + 4 * (t >> 2);
        const int d = 8 * chunk + 2 * (t & 3);
        qf[ks][hl] = valid ? qh[d >> 1] : 0u;
      }
  }

  float oacc[KS][4];
#pragma unroll
  for (int mt = 0; mt < KS; ++mt)
#pragma unroll
    for (int e = 0; e < 4; ++e) oacc[mt][e] = 0.f;
  float m_run[2] = {-INFINITY, -INFINITY};
  float l_run[2] = {0.f, 0.f};


  for (int t = quad; t < kk; t += kQuads) {
    const int b = sm.blocks[t];
    if (b < 0) continue;
    // keys are indexed by position; a paged block's rows are shifted to its page
    const __nv_bfloat16* kbase = kseq;
    const __nv_bfloat16* vbase = vseq;
    if (PAGED) {
      const int64_t shift = (p.cm.block_row<true>(s, b, 0) - (int64_t)b * kBlock) * p.H_kv * D_H;
      kbase = p.k + shift + r * D_H;
      vbase = p.v + shift + r * D_H;
    }
    const int64_t j0 = (int64_t)b * kBlock + 16 * wq;       // first key of this warp's slice
    const int64_t jlo = j0 + r4, jhi = j0 + r4 + 8;
    const bool vlo = jlo <= i, vhi = jhi <= i;

    // ---- K rows lo/hi (A operand of S^T), chunks c, c+4, ...
    uint4 kr[2][KCH];
#pragma unroll
    for (int u = 0; u < KCH; ++u) {
      kr[0][u] = vlo ? ldg_nc_v4(kbase + jlo * kv_stride + 8 * (c + 4 * u)) : make_uint4(0, 0, 0, 0);
      kr[1][u] = vhi ? ldg_nc_v4(kbase + jhi * kv_stride + 8 * (c + 4 * u)) : make_uint4(0, 0, 0, 0);
    }
    // ---- V rows of keys 2c, 2c+1, 2c+8, 2c+9 (A operand of O^T), chunks r4 (+8)
    uint4 vr[4][VCH];
#pragma unroll
    for (int kq = 0; kq < 4; ++kq) {
      const int64_t j = j0 + 2 * c + (kq & 1) + 8 * (kq >> 1);
      const bool ok = j <= i;
#pragma unroll
      for (int u = 0; u < VCH; ++u)
        vr[kq][u] = ok ? ldg_nc_v4(vbase + j * kv_stride + 8 * (r4 + 8 * u)) : make_uint4(0, 0, 0, 0);
    }

    // ---- S^T = K Q^T  (16 keys x 8 heads)
    float s[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
      const int t0w = 2 * ks, t1w = 2 * ks + 1;
      const uint32_t* lo = reinterpret_cast<const uint32_t*>(&kr[0][t0w >> 2]);
      const uint32_t* hi = reinterpret_cast<const uint32_t*>(&kr[1][t0w >> 2]);
      uint32_t a[4];
      a[0] = lo[t0w & 3];
      a[1] = hi[t0w & 3];
      a[2] = reinterpret_cast<const uint32_t*>(&kr[0][t1w >> 2])[t1w & 3];
      a[3] = reinterpret_cast<const uint32_t*>(&kr[1][t1w >> 2])[t1w & 3];
      mma_16816(s, a, qf[ks][0], qf[ks][1]);
    }
    // scores in log2 units; keys after the query are masked
    float x[4];
    x[0] = vlo ? s[0] * p.scale_log2 : -INFINITY;
    x[1] = vlo ? s[1] * p.scale_log2 : -INFINITY;
    x[2] = vhi ? s[2] * p.scale_log2 : -INFINITY;
    x[3] = vhi ? s[3] * p.scale_log2 : -INFINITY;

    // ---- online softmax per head column (heads 2c, 2c+1)
    float pr[4];
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      float mb = fmaxf(x[hh], x[hh + 2]);
      mb = fmaxf(mb, __shfl_xor_sync(kFull, mb, 4));
      mb = fmaxf(mb, __shfl_xor_sync(kFull, mb, 8));
      mb = fmaxf(mb, __shfl_xor_sync(kFull, mb, 16));
      const float m_new = fmaxf(m_run[hh], mb);
      float alpha, p0, p1;
      if (m_new == -INFINITY) {
        alpha = 1.f;
        p0 = p1 = 0.f;
      } else {
        alpha = ex2(m_run[hh] - m_new);
        p0 = ex2(x[hh] - m_new);
        p1 = ex2(x[hh + 2] - m_new);
      }
      m_run[hh] = m_new;
      l_run[hh] = l_run[hh] * alpha + p0 + p1;
      pr[hh] = p0;
      pr[hh + 2] = p1;
#pragma unroll
      for (int mt = 0; mt < KS; ++mt) {
        oacc[mt][hh] *= alpha;
        oacc[mt][hh + 2] *= alpha;
      }
    }
    // P^T operand: transpose the two 8x8 (key x head) tiles
    const uint32_t pb0 = movmatrix_trans(pack_bf16x2(pr[0], pr[1]));   // keys 0-7
    const uint32_t pb1 = movmatrix_trans(pack_bf16x2(pr[2], pr[3]));   // keys 8-15

    // ---- O^T += V^T P^T: m-tile mt covers dims lo(mt) and hi(mt) of this thread
#pragma unroll
    for (int mt = 0; mt < KS; ++mt) {
      // element index inside the owned chunk(s): lo rows -> chunk 0, hi rows -> chunk VCH-1
      const int elo = (D_H == 128) ? mt : mt;
      const int ehi = (D_H == 128) ? mt : 4 + mt;
      const int clo = 0, chi = VCH - 1;
      auto pick = [&](const uint4& wa, const uint4& wb, int e) -> uint32_t {
        const uint32_t* pa = reinterpret_cast<const uint32_t*>(&wa);
        const uint32_t* pbw = reinterpret_cast<const uint32_t*>(&wb);
        return (e & 1) ? prmt_hi(pa[e >> 1], pbw[e >> 1]) : prmt_lo(pa[e >> 1], pbw[e >> 1]);
      };
      uint32_t a[4];
      a[0] = pick(vr[0][clo], vr[1][clo], elo);   // dim lo, keys 2c, 2c+1
      a[1] = pick(vr[0][chi], vr[1][chi], ehi);   // dim hi, keys 2c, 2c+1
      a[2] = pick(vr[2][clo], vr[3][clo], elo);   // dim lo, keys 2c+8, 2c+9
      a[3] = pick(vr[2][chi], vr[3][chi], ehi);   // dim hi, keys 2c+8, 2c+9
      mma_16816(oacc[mt], a, pb0, pb1);
    }
  }

  // ---- per-warp state -> shared memory
#pragma unroll
  for (int hh = 0; hh < 2; ++hh) {
    float lsum = l_run[hh];
    lsum += __shfl_xor_sync(kFull, lsum, 4);
    lsum += __shfl_xor_sync(kFull, lsum, 8);
    lsum += __shfl_xor_sync(kFull, lsum, 16);
    if (r4 == 0) {
      sm.m[warp][2 * c + hh] = m_run[hh];
      sm.l[warp][2 * c + hh] = lsum;
    }
  }
  // this thread's dims: lo(mt) = base_lo + mt, hi(mt) = base_hi + mt
  const int base_lo = 8 * r4;
  const int base_hi = (D_H == 128) ? 64 + 8 * r4 : 8 * r4 + 4;
#pragma unroll
  for (int mt = 0; mt < KS; ++mt) {
    sm.u.o[warp][2 * c][base_lo + mt] = oacc[mt][0];
    sm.u.o[warp][2 * c + 1][base_lo + mt] = oacc[mt][1];
    sm.u.o[warp][2 * c][base_hi + mt] = oacc[mt][2];
    sm.u.o[warp][2 * c + 1][base_hi + mt] = oacc[mt][3];
  }
  __syncthreads();

  // ---- merge the warps in warp order: thread -> (head, 8-dim chunk); O and LSE written
  constexpr int kChunks = D_H / 8;
  for (int wi = threadIdx.x; wi < p.G * kChunks; wi += 32 * kTailWarps) {
    const int h = wi / kChunks, d0 = (wi - h * kChunks) * 8;
    float mx = -INFINITY;
#pragma unroll
    for (int w = 0; w < kTailWarps; ++w) mx = fmaxf(mx, sm.m[w][h]);
    float L2 = 0.f, acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int w = 0; w < kTailWarps; ++w) {
      const float wgt = mx == -INFINITY ? 0.f : ex2(sm.m[w][h] - mx);
      L2 += wgt * sm.l[w][h];
#pragma unroll
      for (int e = 0; e < 8; ++e) acc[e] += wgt * sm.u.o[w][h][d0 + e];
    }
    const float inv = L2 > 0.f ? 1.f / L2 : 0.f;
    const int hq = r * p.G + h;
    uint4 pk;
    pk.x = pack_bf16x2(acc[0] * inv, acc[1] * inv);
    pk.y = pack_bf16x2(acc[2] * inv, acc[3] * inv);
    pk.z = pack_bf16x2(acc[4] * inv, acc[5] * inv);
    pk.w = pack_bf16x2(acc[6] * inv, acc[7] * inv);
    *reinterpret_cast<uint4*>(p.o + (s * p.H_q + hq) * D_H + d0) = pk;
    if (d0 == 0) p.lse[s * p.H_q + hq] = (mx + __log2f(L2)) * 0.69314718055994531f;
  }
}

}  // namespace

cudaError_t launch_decode_tail(const void* q, const void* k_cache, const void* v_cache,
                               const float* Mdec, int64_t nblk_max, const CacheMap& cm, int S,
                               int64_t max_len, int H_q, int H_kv, int d_h, int kk,
                               int32_t* idx_out, void* o, float* lse, cudaStream_t stream) {
  AttnParams p{};
  p.q = static_cast<const __nv_bfloat16*>(q);
  p.k = static_cast<const __nv_bfloat16*>(k_cache);
  p.v = static_cast<const __nv_bfloat16*>(v_cache);
  p.Mdec = Mdec;
  p.idx_out = idx_out;
  p.o = static_cast<__nv_bfloat16*>(o);
  p.lse = lse;
  p.cm = cm;
  p.max_len = max_len;
  p.nblk_max = nblk_max;
  p.S = S;
  p.H_q = H_q;
  p.H_kv = H_kv;
  p.G = H_q / H_kv;
  p.kk = kk;
  p.scale_log2 = (float)(1.4426950408889634 / sqrt((double)d_h));
  const dim3 grid((unsigned)((int64_t)S * H_kv));
  // may start under the index-key scan's tail (it waits for the block scores)
  auto run = [&](auto kern, size_t smem) -> cudaError_t {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    return launch_pdl(kern, grid, dim3(32 * kTailWarps), smem, stream, p);
  };
  if (d_h == 128) {
    constexpr size_t S128 = sizeof(TailSmem<128>);
    return cm.pages ? run(k_decode_tail<128, true>, S128) : run(k_decode_tail<128, false>, S128);
  }
  constexpr size_t S64 = sizeof(TailSmem<64>);
  return cm.pages ? run(k_decode_tail<64, true>, S64) : run(k_decode_tail<64, false>, S64);
}

}  // namespace msa

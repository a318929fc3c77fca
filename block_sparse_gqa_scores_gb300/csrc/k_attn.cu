// Decode attention of MSA («MiniMax-M3：MSA 技术报告速读», section 主分支, eq. O^(h)_i, and
// the LSE of section Kernel): exact softmax attention of the G query heads of group r of one new
// token over the visible tokens of its selected blocks, split into block ranges whose partials
// are merged in a fixed order (the kernel section's pre-scheduled splits with a two-stage merge
// and no atomics).
//
// Layout of the work: one CTA = 4 warps per (sequence, group, split).  Warp w owns keys
// [16w, 16w+16) of every selected block, so a block is read by the 4 warps side by side.  The
// G <= 8 heads of the group are the N=8 side of the m16n8k16 MMA with the keys (S^T = K Q^T) or
// the head dims (O^T += V^T P^T) as its M side, which wastes no MMA lane on the single query; P
// goes from the S^T accumulator to the P^T operand with one movmatrix transpose per 8x8 tile.
// K and V rows are loaded from global memory directly into MMA fragments as 16-byte vectors:
//   * S^T: the contracted head dim is permuted identically in K (A operand) and Q^T (B), so a
//     thread's A fragment words are whole 16-byte chunks of a K row;
//   * O^T: a thread owns 8 (d_h=64) or 16 (d_h=128) head dims of V for 4 keys and pairs keys
//     with byte permutes; the output rows are un-permuted when stored.
// Online softmax per warp in the log2 domain (scale*log2 e folded into the scores), then the
// four warps' (max, sum, O) states are merged in shared memory in a fixed order.
#include <math.h>

#include "msa_device.cuh"
#include "msa_internal.h"

namespace msa {
namespace {

constexpr int kWarps = 4;
constexpr unsigned kFull = 0xffffffffu;

template <int D_H>
struct AttnSmem {
  float m[kWarps][8];
  float l[kWarps][8];
  float o[kWarps][8][D_H];
};

struct AttnParams {
  const __nv_bfloat16* q;
  const __nv_bfloat16* k;
  const __nv_bfloat16* v;
  const int32_t* idx;
  float* part_o;      // decode split partials [S*H_kv*nsplit, G, D_H] (normalised)
  float* part_lse;    // decode split partials [S*H_kv*nsplit, G] (log2 units)
  CacheMap cm;        // where each sequence's cache rows are (packed or paged)
  int64_t max_len;    // length bound
  int H_q, H_kv, G, kk, nsplit, S;
  float scale_log2;   // log2(e) / sqrt(d_h)
};

template <int D_H, bool PAGED>
__global__ void __launch_bounds__(32 * kWarps) k_sparse_attn(const AttnParams p) {
  constexpr int KS = D_H / 16;             // k-steps of S^T, m-tiles of O^T
  constexpr int KCH = D_H / 32;            // 16-B K chunks per thread per key row
  constexpr int VCH = D_H / 64;            // 16-B V chunks per thread per key
  __shared__ AttnSmem<D_H> sm;
  pdl_launch_dependents();                  // the merge may be scheduled under this grid's tail

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int c = lane & 3, r4 = lane >> 2;

  // ---------------------------------------------------------------- the problem
  const int64_t unit = blockIdx.x;          // (sequence, group, split)
  const int split = (int)(unit % p.nsplit);
  const int64_t sr = unit / p.nsplit;
  const int64_t s = sr / p.H_kv;
  const int r = (int)(sr - s * p.H_kv);
  const int64_t L = p.cm.len<PAGED>(s, p.max_len);
  const int64_t srow = p.cm.seq_row<PAGED>(s);
  const int64_t kv_stride = (int64_t)p.H_kv * D_H;          // elements between tokens
  const __nv_bfloat16* kseq = p.k + (srow * p.H_kv + r) * D_H;   // packed: the sequence's rows
  const __nv_bfloat16* vseq = p.v + (srow * p.H_kv + r) * D_H;
  const int64_t i = L - 1;                  // the new token's position
  const int32_t* sel = p.idx + sr * p.kk;
  const __nv_bfloat16* qrow = p.q + s * (int64_t)p.H_q * D_H;
  const int per = (p.kk + p.nsplit - 1) / p.nsplit;
  const int t0 = split * per;
  const int t1 = min(p.kk, t0 + per);

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


  pdl_wait();                               // the selection is written
  for (int t = t0; t < t1; ++t) {
    const int b = __ldg(sel + t);
    if (b < 0) continue;
    // keys are indexed by position; a paged block's rows are shifted to its page
    const __nv_bfloat16* kbase = kseq;
    const __nv_bfloat16* vbase = vseq;
    if (PAGED) {
      const int64_t shift = (p.cm.block_row<true>(s, b, 0) - (int64_t)b * kBlock) * p.H_kv * D_H;
      kbase = p.k + shift + r * D_H;
      vbase = p.v + shift + r * D_H;
    }
    const int64_t j0 = (int64_t)b * kBlock + 16 * warp;     // first key of this warp's slice
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
    sm.o[warp][2 * c][base_lo + mt] = oacc[mt][0];
    sm.o[warp][2 * c + 1][base_lo + mt] = oacc[mt][1];
    sm.o[warp][2 * c][base_hi + mt] = oacc[mt][2];
    sm.o[warp][2 * c + 1][base_hi + mt] = oacc[mt][3];
  }
  __syncthreads();

  // ---- merge the 4 warps: thread -> (head, 8-dim chunk)
  constexpr int kChunks = D_H / 8;
  for (int wi = threadIdx.x; wi < p.G * kChunks; wi += 32 * kWarps) {
    const int h = wi / kChunks, d0 = (wi - h * kChunks) * 8;
    float mx = -INFINITY;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) mx = fmaxf(mx, sm.m[w][h]);
    float wgt[kWarps], L = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      wgt[w] = mx == -INFINITY ? 0.f : ex2(sm.m[w][h] - mx);
      L += wgt[w] * sm.l[w][h];
    }
    const float inv = L > 0.f ? 1.f / L : 0.f;
    float ov[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      float acc = 0.f;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) acc += wgt[w] * sm.o[w][h][d0 + e];
      ov[e] = acc * inv;
    }
    const float lse2 = L > 0.f ? mx + __log2f(L) : -INFINITY;
    float* po = p.part_o + (unit * p.G + h) * D_H + d0;
#pragma unroll
    for (int e = 0; e < 8; ++e) po[e] = ov[e];
    if (d0 == 0) p.part_lse[unit * p.G + h] = lse2;
  }
}

// Decode: combine the split partials of each (sequence, head) in split order.
template <int D_H>
__global__ void __launch_bounds__(128) k_decode_merge(const float* __restrict__ part_o,
                                                      const float* __restrict__ part_lse,
                                                      __nv_bfloat16* __restrict__ o,
                                                      float* __restrict__ lse, int H_q, int H_kv,
                                                      int G, int nsplit) {
  pdl_wait();                                    // the split partials are written
  const int64_t sr = blockIdx.x;                 // (s, r)
  const int64_t s = sr / H_kv;
  const int r = (int)(sr - s * H_kv);
  constexpr int kChunks = D_H / 8;
  for (int wi = threadIdx.x; wi < G * kChunks; wi += blockDim.x) {
    const int h = wi / kChunks, d0 = (wi - h * kChunks) * 8;
    float mx = -INFINITY;
    for (int sp = 0; sp < nsplit; ++sp) mx = fmaxf(mx, part_lse[(sr * nsplit + sp) * G + h]);
    float L = 0.f, acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    for (int sp = 0; sp < nsplit; ++sp) {
      const int64_t u = sr * nsplit + sp;
      const float w = mx == -INFINITY ? 0.f : ex2(part_lse[u * G + h] - mx);
      L += w;
      const float* po = part_o + (u * G + h) * D_H + d0;
#pragma unroll
      for (int e = 0; e < 8; ++e) acc[e] += w * po[e];
    }
    const float inv = L > 0.f ? 1.f / L : 0.f;
    const int hq = r * G + h;
    uint4 pk;
    pk.x = pack_bf16x2(acc[0] * inv, acc[1] * inv);
    pk.y = pack_bf16x2(acc[2] * inv, acc[3] * inv);
    pk.z = pack_bf16x2(acc[4] * inv, acc[5] * inv);
    pk.w = pack_bf16x2(acc[6] * inv, acc[7] * inv);
    *reinterpret_cast<uint4*>(o + (s * H_q + hq) * D_H + d0) = pk;
    if (d0 == 0) lse[s * H_q + hq] = (mx + __log2f(L)) * 0.69314718055994531f;
  }
}

}  // namespace

cudaError_t launch_sparse_attn_decode(const void* q, const void* k_cache, const void* v_cache,
                                      const int32_t* idx, const CacheMap& cm, int S,
                                      int64_t max_len, int H_q, int H_kv, int d_h, int kk,
                                      int nsplit, float* part_o, float* part_lse, void* o,
                                      float* lse, cudaStream_t stream) {
  AttnParams p{};
  p.q = static_cast<const __nv_bfloat16*>(q);
  p.k = static_cast<const __nv_bfloat16*>(k_cache);
  p.v = static_cast<const __nv_bfloat16*>(v_cache);
  p.idx = idx;
  p.cm = cm;
  p.part_o = part_o;
  p.part_lse = part_lse;
  p.max_len = max_len;
  p.S = S;
  p.H_q = H_q;
  p.H_kv = H_kv;
  p.G = H_q / H_kv;
  p.kk = kk;
  p.nsplit = nsplit;
  p.scale_log2 = (float)(1.4426950408889634 / sqrt((double)d_h));
  const dim3 grid((unsigned)((int64_t)S * H_kv * nsplit));
  const dim3 mgrid((unsigned)((int64_t)S * H_kv));
  auto* ob = static_cast<__nv_bfloat16*>(o);
  // both launches may start under the previous kernel's tail (they wait for its results)
  auto run = [&](auto attn, auto merge) -> cudaError_t {
    cudaError_t e = launch_pdl(attn, grid, dim3(32 * kWarps), 0, stream, p);
    if (e != cudaSuccess) return e;
    return launch_pdl(merge, mgrid, dim3(128), 0, stream, (const float*)part_o,
                      (const float*)part_lse, ob, lse, H_q, H_kv, p.G, nsplit);
  };
  if (d_h == 128)
    return cm.pages ? run(k_sparse_attn<128, true>, k_decode_merge<128>)
                    : run(k_sparse_attn<128, false>, k_decode_merge<128>);
  return cm.pages ? run(k_sparse_attn<64, true>, k_decode_merge<64>)
                  : run(k_sparse_attn<64, false>, k_decode_merge<64>);
}

}  // namespace msa

// Block-major ("KV-outer") pass of the sparse main branch («MiniMax-M3：MSA 技术报告速读»,
// section 主分支 eq. O^(h)_i; the kernel section's organisation in which a selected KV block
// gathers the queries that chose it and stacks them to fill tensor-core MMAs).
//
// Input: the private selections of a query chunk -- (query, slot) pairs whose block fewer than
// kSharedMin queries of the same 16-query tile selected -- bucketed by (group r, block b).  A work tile is up
// to 128/G entries of one bucket; their G heads stack into the 128 rows of one UMMA tile:
//   S = Q_stack [128 x d_h] . K_b^T [d_h x 64]       tcgen05, bf16 -> fp32 in TMEM
//   row-wise softmax over the block's visible keys   one thread per row (TMEM lane)
//   O = P [128 x 64] . V_b [64 x d_h]                tcgen05, V as an MN-major operand
// and every row writes a partial: O normalised by its own sum (bf16) and its log2-domain LSE,
// at the fixed position of its (group, query, slot) -- a query's partials are contiguous, so the
// merge reads them in order without an index.
// A partial covers exactly one block, so no rescaling is needed; the epilogue of the
// shared-block pass (k_attn_shared.cu) combines a row's partials with its shared-block state in
// slot order.
// Q rows (by TMA, one box per query, at G = 8; by cp.async otherwise), K_b and V_b (cp.async)
// land in 128-byte-swizzled tiles (the canonical K-major / MN-major SW128 layouts).  P reuses Q's shared memory and O reuses S's TMEM
// columns, so three CTAs fit on an SM.  The next tile's K_b (if its bucket differs) is loaded
// as soon as S = Q K^T has completed, and its query rows and V_b once O = P V has completed,
// so those loads run under the softmax and the epilogue.  Persistent grid; each CTA takes a contiguous range of
// work tiles (consecutive tiles often share K_b, V_b) and finds each tile's bucket by binary
// search over the per-bucket tile offsets.
#include <cmath>

#include "msa_device.cuh"
#include "msa_internal.h"

namespace msa {
namespace {

__device__ unsigned g_kvo_status = 0;

constexpr int kRowsT = 128;                // UMMA M
constexpr int kThreadsKvo = 128;           // 4 warps: TMEM lane quarters

template <int D_H>
struct KvoSmem {
  static constexpr int kHalves = D_H / 64;
  static constexpr int kQHalf = kRowsT * 128;     // 128 rows x 64 dims
  static constexpr int kKHalf = 64 * 128;         // 64 keys x 64 dims
  static constexpr int kOffQ = 0;
  static constexpr int kOffP = 0;                 // P (128 rows x 64 keys) reuses Q's first half
  static constexpr int kOffK = kOffQ + kHalves * kQHalf;
  static constexpr int kOffV = kOffK + kHalves * kKHalf;
  static constexpr int kOffBar = kOffV + kHalves * kKHalf;
  static constexpr int kOffMisc = kOffBar + 16;
  static constexpr int kOffEnt = kOffMisc + 16;   // entries of this tile and the next (<= 128 each)
  static constexpr int kBytes = kOffEnt + 2 * kRowsT * 4;
  static constexpr int kAlloc = kBytes + 1024;
  static constexpr uint32_t kTmemCols = D_H;      // S (64 columns), then O over the same columns
};

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
}
__device__ __forceinline__ void fence_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// MN-major operand, 128-byte swizzle: 64-element MN blocks `lbo` bytes apart, 8-row K groups
// `sbo` bytes apart.
__device__ __forceinline__ uint64_t umma_desc_mnmajor(uint32_t smem_addr, uint32_t lbo,
                                                      uint32_t sbo) {
  return (uint64_t)((smem_addr & 0x3FFFFu) >> 4) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
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

template <int D_H>
__global__ void __launch_bounds__(kThreadsKvo, 3)
    k_attn_kvouter(const __grid_constant__ CUtensorMap tm_q,
                   const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ k,
                   const __nv_bfloat16* __restrict__ v, const int* __restrict__ entries,
                   const int* __restrict__ offset, const int* __restrict__ tile_off, int nbuckets,
                   int64_t nblk, int64_t N, int64_t q0, int64_t nq, int H_q, int H_kv, int G,
                   int kk, int ept,
                   __nv_bfloat16* __restrict__ part_o, float* __restrict__ part_lse,
                   float scale_log2) {
  using L = KvoSmem<D_H>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t sb = smem_u32(smem);
  const uint32_t mma_bar = sb + L::kOffBar, q_bar = sb + L::kOffBar + 8;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kOffMisc);
  int* s_ent = reinterpret_cast<int*>(smem + L::kOffEnt);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tid = threadIdx.x;

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
  // S lives in columns [0, 64); O overwrites columns [0, d_h) once S has been read
  const uint32_t tmem_s = tmem, tmem_o = tmem;

  const int total_tiles = tile_off[nbuckets];
  const int64_t kv_stride = (int64_t)H_kv * D_H;             // elements between tokens
  constexpr int kChunks = D_H / 8;                           // 16-B chunks per row
  uint32_t phase = 0;
  bool ok = true;

  // a contiguous range of work tiles per CTA: consecutive tiles often share a bucket (K_b, V_b)
  const int per = (total_tiles + gridDim.x - 1) / gridDim.x;
  const int t_beg = blockIdx.x * per;
  const int t_end = min(total_tiles, t_beg + per);
  // bucket of the first tile: last b with tile_off[b] <= t_beg (binary search, once per CTA);
  // later tiles advance it, since a CTA's tiles are consecutive
  int bucket = 0;
  if (t_beg < t_end) {
    int lo = 0, hi = nbuckets;                               // tile_off[lo] <= t_beg < tile_off[hi]
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (__ldg(tile_off + mid) <= t_beg) lo = mid; else hi = mid;
    }
    bucket = lo;
  }
  int next_off = t_beg < t_end ? __ldg(tile_off + bucket + 1) : 0;   // first tile of bucket + 1
  // tile -> (bucket, first entry, entries), advancing (bkt, nxt) from the previous tile's
  auto describe = [&](int tile, int& bkt, int& nxt, int& e0, int& n_e) {
    while (nxt <= tile) {
      ++bkt;
      nxt = __ldg(tile_off + bkt + 1);
    }
    e0 = __ldg(offset + bkt) + (tile - __ldg(tile_off + bkt)) * ept;
    n_e = min(ept, __ldg(offset + bkt + 1) - e0);
  };
  // K_b and/or V_b of a bucket into their buffers (rows past the sequence: zeros, so p = 0)
  auto load_kv = [&](int bkt, bool do_k, bool do_v) {
    const int rb = (int)(bkt / nblk);
    const int64_t bb = bkt - (int64_t)rb * nblk;
    const __nv_bfloat16* kb = k + (bb * kBlock * H_kv + rb) * (int64_t)D_H;
    const __nv_bfloat16* vb = v + (bb * kBlock * H_kv + rb) * (int64_t)D_H;
    for (int x = tid; x < kBlock * kChunks; x += kThreadsKvo) {
      const int j = x / kChunks, c = x - j * kChunks;
      const uint32_t off = (c >> 3) * L::kKHalf + j * 128 + (((c & 7) ^ (j & 7)) << 4);
      if (bb * kBlock + j < N) {
        if (do_k) cp_async16(sb + L::kOffK + off, kb + j * kv_stride + c * 8);
        if (do_v) cp_async16(sb + L::kOffV + off, vb + j * kv_stride + c * 8);
      } else {
        if (do_k)
          asm volatile("st.shared.v4.b32 [%0], {%1,%1,%1,%1};" ::"r"(sb + L::kOffK + off), "r"(0u)
                       : "memory");
        if (do_v)
          asm volatile("st.shared.v4.b32 [%0], {%1,%1,%1,%1};" ::"r"(sb + L::kOffV + off), "r"(0u)
                       : "memory");
      }
    }
  };
  // the stacked query rows of a tile (entry e's G heads are rows e*G .. e*G+G-1): at G = 8 an
  // entry is one 1-KB swizzle atom per 64-dim half, a single TMA box issued by lane e of warp 0
  // and counted on q_bar; otherwise every thread gathers 16-byte pieces with cp.async
  auto gather_q = [&](int bkt, const int* ent, int n_ent) {
    const int rb = (int)(bkt / nblk);
    if (G == 8) {
      // one lane of warp 0 per entry: the boxes are issued in parallel, not one after another
      if (warp == 0) {
        if (lane == 0) mbar_expect_tx(q_bar, (uint32_t)(n_ent * 8 * 128 * L::kHalves));
        __syncwarp();
        if (lane < n_ent) {
          const int i = (int)(q0 + (ent[lane] >> 6));
#pragma unroll
          for (int bx = 0; bx < L::kHalves; ++bx)
            tma_load_3d(sb + L::kOffQ + bx * L::kQHalf + lane * 1024, &tm_q, q_bar, 64 * bx,
                        rb * 8, i);
        }
      }
      return;
    }
    const int rows = n_ent * G;
    for (int x = tid; x < rows * kChunks; x += kThreadsKvo) {
      const int R = x / kChunks, c = x - R * kChunks;
      const int e = R / G, h = R - e * G;
      const int64_t i = q0 + (ent[e] >> 6);
      const uint32_t off = (c >> 3) * L::kQHalf + R * 128 + (((c & 7) ^ (R & 7)) << 4);
      cp_async16(sb + L::kOffQ + off, q + (i * H_q + (int64_t)rb * G + h) * D_H + c * 8);
    }
  };

  int e0 = 0, n_e = 0;
  if (t_beg < t_end) {
    describe(t_beg, bucket, next_off, e0, n_e);
    load_kv(bucket, true, true);
    if (tid < n_e) s_ent[tid] = __ldg(entries + e0 + tid);
    __syncthreads();
    gather_q(bucket, s_ent, n_e);
  }
  uint32_t qphase = 0;
  for (int tile = t_beg; tile < t_end && ok; ++tile) {
    const int cur = (tile - t_beg) & 1;
    const int* ent_cur = s_ent + cur * kRowsT;
    const int r = (int)(bucket / nblk);
    const int64_t b = bucket - (int64_t)r * nblk;
    const int rows = n_e * G;
    cp_async_wait_all();                                     // this tile's Q (and K_b, V_b)
    fence_async_smem();
    bool qok = true;
    if (G == 8 && tid == 0) qok = mbar_wait(q_bar, qphase, &g_kvo_status);   // Q by TMA
    qphase ^= 1u;
    ok = __syncthreads_and(qok);
    if (!ok) break;

    // ---- S = Q_stack K_b^T
    if (tid == 0) {
      tc_fence_after();
      constexpr uint32_t idesc = umma_idesc_bf16(kRowsT, 64);
#pragma unroll
      for (int ks = 0; ks < D_H / 16; ++ks) {
        const uint32_t a = sb + L::kOffQ + (ks >> 2) * L::kQHalf + (ks & 3) * 32;
        const uint32_t bk = sb + L::kOffK + (ks >> 2) * L::kKHalf + (ks & 3) * 32;
        umma_bf16(tmem_s, umma_desc_kmajor(a, 1024, 128), umma_desc_kmajor(bk, 1024, 128), idesc,
                  ks > 0 ? 1u : 0u);
      }
      umma_commit(mma_bar);
    }
    ok = __syncthreads_and(mbar_wait(mma_bar, phase, &g_kvo_status));
    if (!ok) break;
    phase ^= 1u;
    tc_fence_after();

    // ---- K_b is free: the next tile's entries and, for a new bucket, its K_b
    const bool has_next = tile + 1 < t_end;
    int n_bucket = bucket, n_next = next_off, n_e0 = 0, n_ne = 0;
    if (has_next) {
      describe(tile + 1, n_bucket, n_next, n_e0, n_ne);
      if (tid < n_ne) s_ent[(cur ^ 1) * kRowsT + tid] = __ldg(entries + n_e0 + tid);
    }
    const bool new_bucket = has_next && n_bucket != bucket;
    if (new_bucket) load_kv(n_bucket, true, false);
    asm volatile("cp.async.commit_group;" ::: "memory");

    // ---- softmax of row R = 32*warp + lane over the block's visible keys
    const int R = 32 * warp + lane;
    const bool rv = R < rows;
    int64_t i = 0, slot_pos = 0;
    int h = 0;
    float mx = 0.f, l = 0.f;
    {
      uint32_t s[64];
      MSA_TMEM_LD64(tmem_s + ((uint32_t)(32 * warp) << 16), s);
      tmem_ld_wait();
      if (rv) {
        const int e = R / G;
        h = R - e * G;
        const int ent = ent_cur[e];
        slot_pos = ((int64_t)r * nq + (ent >> 6)) * kk + (ent & 63);
        i = q0 + (ent >> 6);
        if (b == (i >> 6)) {                                // local block: keys j <= i only
          const int lim = (int)(i - b * kBlock);
#pragma unroll
          for (int c = 0; c < 64; ++c)
            if (c > lim) s[c] = __float_as_uint(-INFINITY);
        }
        mx = rowmax64(s) * scale_log2;
      }
      uint32_t pk[32];
      float l0 = 0.f, l1 = 0.f;
#pragma unroll
      for (int c = 0; c < 32; ++c) {
        float x0, x1;
        ffma2(x0, x1, __uint_as_float(s[2 * c]), __uint_as_float(s[2 * c + 1]), scale_log2,
              scale_log2, -mx, -mx);
        const float p0 = rv ? ex2(x0) : 0.f;
        const float p1 = rv ? ex2(x1) : 0.f;
        fadd2(l0, l1, l0, l1, p0, p1);
        pk[c] = pack_bf16x2(p0, p1);
      }
      l = l0 + l1;
#pragma unroll
      for (int cc = 0; cc < 8; ++cc) {
        const uint32_t addr = sb + L::kOffP + R * 128 + ((cc ^ (R & 7)) << 4);
        asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(addr), "r"(pk[4 * cc]),
                     "r"(pk[4 * cc + 1]), "r"(pk[4 * cc + 2]), "r"(pk[4 * cc + 3])
                     : "memory");
      }
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();

    // ---- O = P V_b  (V_b: keys x dims, dims contiguous -> MN-major B operand)
    if (tid == 0) {
      tc_fence_after();
      constexpr uint32_t idesc = umma_idesc_bf16(kRowsT, D_H) | (1u << 16);   // B MN-major
#pragma unroll
      for (int ks = 0; ks < 4; ++ks) {
        const uint32_t a = sb + L::kOffP + ks * 32;
        const uint32_t bv = sb + L::kOffV + ks * 2048;      // 16 keys = two 8-row groups
        umma_bf16(tmem_o, umma_desc_kmajor(a, 1024, 128), umma_desc_mnmajor(bv, L::kKHalf, 1024),
                  idesc, ks > 0 ? 1u : 0u);
      }
      umma_commit(mma_bar);
    }
    ok = __syncthreads_and(mbar_wait(mma_bar, phase, &g_kvo_status));
    if (!ok) break;
    phase ^= 1u;
    tc_fence_after();

    // ---- Q (holding P) and V_b are free once O = P V is done: the next tile's rows, V_b
    if (new_bucket) load_kv(n_bucket, false, true);
    if (has_next) gather_q(n_bucket, s_ent + (cur ^ 1) * kRowsT, n_ne);
    asm volatile("cp.async.commit_group;" ::: "memory");

    // ---- epilogue: normalised partial (bf16) and log2-domain LSE of each row
    {
      const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
      for (int half = 0; half < D_H / 64; ++half) {
        uint32_t o[64];
        MSA_TMEM_LD64(tmem_o + ((uint32_t)(32 * warp) << 16) + 64 * half, o);
        tmem_ld_wait();
        if (rv) {
          uint4* dst = reinterpret_cast<uint4*>(part_o + (slot_pos * G + h) * D_H + 64 * half);
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            uint4 w;
            w.x = pack_bf16x2(__uint_as_float(o[8 * c + 0]) * inv, __uint_as_float(o[8 * c + 1]) * inv);
            w.y = pack_bf16x2(__uint_as_float(o[8 * c + 2]) * inv, __uint_as_float(o[8 * c + 3]) * inv);
            w.z = pack_bf16x2(__uint_as_float(o[8 * c + 4]) * inv, __uint_as_float(o[8 * c + 5]) * inv);
            w.w = pack_bf16x2(__uint_as_float(o[8 * c + 6]) * inv, __uint_as_float(o[8 * c + 7]) * inv);
            dst[c] = w;
          }
        }
      }
      if (rv) part_lse[slot_pos * G + h] = mx + __log2f(l);
    }
    tc_fence_before();
    __syncthreads();
    bucket = n_bucket;
    next_off = n_next;
    e0 = n_e0;
    n_e = n_ne;
  }
  cp_async_wait_all();                                       // no copy left in flight

  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, L::kTmemCols);
  }
}

}  // namespace

int kvouter_smem_bytes(int d_h) {
  return d_h == 128 ? KvoSmem<128>::kAlloc : KvoSmem<64>::kAlloc;
}

cudaError_t launch_attn_kvouter(const void* q, const void* k, const void* v, const int* entries,
                                const int* offset, const int* tile_off, int nbuckets, int64_t nblk,
                                int64_t N, int64_t q0, int64_t q1, int H_q, int H_kv, int d_h,
                                int kk, int grid, void* part_o, float* part_lse,
                                cudaStream_t stream) {
  const int G = H_q / H_kv;
  const float scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)d_h));
  const auto* qq = static_cast<const __nv_bfloat16*>(q);
  // Q as [N, H_q, d_h]: one box = one query's G heads x 64 dims, 128-byte swizzle
  CUtensorMap tq;
  cudaError_t me = make_tma_3d_bf16(&tq, q, (uint64_t)d_h, (uint64_t)H_q, (uint64_t)N, 64, G, 1, 128);
  if (me != cudaSuccess) return me;
  const auto* kp = static_cast<const __nv_bfloat16*>(k);
  const auto* vv = static_cast<const __nv_bfloat16*>(v);
  auto* po = static_cast<__nv_bfloat16*>(part_o);
  if (d_h == 128) {
    auto kern = k_attn_kvouter<128>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         KvoSmem<128>::kAlloc);
    if (e != cudaSuccess) return e;
    kern<<<grid, kThreadsKvo, KvoSmem<128>::kAlloc, stream>>>(tq, qq, kp, vv, entries, offset, tile_off,
                                                             nbuckets, nblk, N, q0, q1 - q0, H_q, H_kv, G,
                                                             kk, kRowsT / G, po, part_lse, scale_log2);
  } else {
    auto kern = k_attn_kvouter<64>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         KvoSmem<64>::kAlloc);
    if (e != cudaSuccess) return e;
    kern<<<grid, kThreadsKvo, KvoSmem<64>::kAlloc, stream>>>(tq, qq, kp, vv, entries, offset, tile_off,
                                                            nbuckets, nblk, N, q0, q1 - q0, H_q, H_kv, G,
                                                            kk, kRowsT / G, po, part_lse, scale_log2);
  }
  return cudaGetLastError();
}

cudaError_t read_reset_kvo_status(unsigned* out) {
  unsigned zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(out, g_kvo_status, sizeof(unsigned));
  if (e != cudaSuccess) return e;
  return cudaMemcpyToSymbol(g_kvo_status, &zero, sizeof(unsigned));
}

}  // namespace msa

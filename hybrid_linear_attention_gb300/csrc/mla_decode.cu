// mla_decode.cu -- absorbed gated-MLA decode over the 576-wide latent cache.
//
// "Ling-3.1-flash: Grouped Routing and Two Different MLA Caches", sections "MLA's expanded
// reference path" and "Why weight absorption keeps the same attention function": each cached
// position keeps its 512-wide normalised latent c_t and the 64-wide rotated positional key r_t
// shared by the 64 heads.  With the key up-projection W_K,i moved into the query
// (q~_i = W_K,i^T q_i^N) the score of head i is scale * [q~_i ; q_i^R] . [c_t ; r_t] over the
// same 576-wide key for every head; the latent itself is the attention value, and the value
// up-projection W_V,i comes after the weighted sum; a per-head sigmoid gate scales the head's
// 128-wide output.
//
// Kernels (the two projections around the attention are in mla_proj.cu):
//   mla_latent_kernel   per sequence, all 64 heads: S = Q C^T over 64-position tiles of the
//                       cache (tcgen05, M = 64 heads, Q and C K-major, fp32 in TMEM), online
//                       softmax on the CUDA cores, Z^T += C^T P^T with the same C tile read
//                       MN-major and P written K-major over the tile's positional block
//                       (tcgen05, 4 M-slices of 128 latent channels); Z rescaled in TMEM when
//                       a head's max moves.
//   mla_combine_kernel  the split partial sums merged to a common maximum.
#include "kda_common.cuh"
#include "kda_internal.h"
#include "kda_tc_ptx.cuh"

#include <cuda.h>
#include <cudaTypedefs.h>
#include <atomic>
#include <cstdlib>
#include <mutex>

#include <cstring>

namespace kda {
namespace {

using namespace tc;

constexpr int MH = 64;        // heads
constexpr int ML = 512;       // latent width
constexpr int MR = 64;        // positional-key width
constexpr int MK = ML + MR;   // cached key width
constexpr int TP = 64;        // cached positions per tile
constexpr int KB = MK / 64;   // 64-element key blocks (128 bytes of bf16)
constexpr int PFD = 2;       // tiles ahead of the one being loaded that are fetched into L2
constexpr int MLA_NT = 384;   // eight softmax warps (two per TMEM lane quarter) + four issuer warps

// shared memory of the latent kernel (1024-byte aligned base): Q [KB][64 heads][128 B]
// (72 KB, K-major) and two cache tiles [KB][64 positions][128 B] (72 KB each, TMA, 128-byte
// swizzle).  A tile's last (positional) block becomes P = its softmax weights, [64 heads]
// [64 positions] bf16, once the score product has read it.
constexpr uint32_t BLK = TP * 128;                 // one key block of a tile
constexpr uint32_t TILE = KB * BLK;
constexpr uint32_t M_OFF_Q = 0;
constexpr uint32_t M_OFF_C = KB * MH * 128;
constexpr uint32_t M_SMEM = M_OFF_C + 2 * TILE + 1024;
constexpr uint32_t M_TM_S = 0;    // S: 2 buffers of 64 columns; M = 64 heads in lanes 32 w + 0..15
constexpr uint32_t M_TM_S2 = 128;  // the second partial sum of S (key blocks 5-8), 2 buffers
constexpr uint32_t M_TM_Z = 256;  // Z^T: 4 slices of 128 lanes (latent) x 64 columns (heads)
// MB_SF0/1: the softmax warps have read S buffer 0 / 1 (it may be overwritten)
enum { MB_Q = 0, MB_C0, MB_C1, MB_S0, MB_S1, MB_SF0, MB_SF1, MB_P, MB_Z, MB_N };

struct MlaMaps {
  CUtensorMap q, c;
};

// 2^x on the special-function unit (relative error ~2^-22; the weights are bf16 operands)
__device__ __forceinline__ float ex2f_sfu(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
// a tensor tile fetched into L2 only (no shared memory, no barrier)
__device__ __forceinline__ void tma_prefetch_3d(const CUtensorMap *map, int c0, int c1, int c2) {
  asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(c0), "r"(c1), "r"(c2)
               : "memory");
}
// offset of (row r, 16-byte chunk j) in a 128-byte-swizzled block
__device__ __forceinline__ uint32_t sw128_row(int r, int j) {
  return (uint32_t)r * 128u + ((uint32_t)(j ^ (r & 7)) << 4);
}

// Warps 0-7: softmax and rescale (warp w reads TMEM lanes 32 (w & 3) .. + 31; in S, whose
// M = 64 rows sit in lanes 32 (w & 3) + 0..15, lane l < 16 of warps w and w + 4 owns head
// 16 (w & 3) + l, the first warp for a tile's positions 0-31 and the second for 32-63; each
// owner hands the upper 16 of its 32 scores to lane l + 16, so every lane takes 16 weights).
// Warps 8-11: TMA loads and tensor-core issue (S products on 8 and 9, Z products on 10 and
// 11).  The sides meet only on mbarriers: C tile landed, S ready, S read, P ready, Z done.
__global__ void __launch_bounds__(MLA_NT, 1)
    mla_latent_kernel(const MlaArgs a, const __grid_constant__ MlaMaps maps) {
  extern __shared__ uint8_t mraw[];
  const uint32_t raw = smem_u32(mraw);
  const uint32_t pad = ((raw + 1023u) & ~1023u) - raw;
  uint8_t *sm = mraw + pad;
  const uint32_t sb = raw + pad;
  __shared__ __align__(8) uint64_t s_bar[MB_N];
  __shared__ uint32_t s_tmem;
  __shared__ volatile uint32_t s_abort;
  __shared__ uint32_t s_loads[2], s_smmas[2], s_mmas;
  __shared__ int s_stop;  // the softmax warps' exit decision, taken by one thread per tile
  __shared__ float s_alpha[MH], s_l[MH], s_mfin[MH];
  __shared__ float s_pmax[2][MH], s_lpart[MH];  // a tile's half maxima; the second half's l
  __shared__ int s_rescale[2];  // by tile parity: set by the head owners, reset after use

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int b = blockIdx.x;
  int len = a.lengths[b];
  if (len < 0 || len > a.L_max) {  // a length outside the cache: flagged, nothing attended
    if (tid == 0 && a.err) atomicOr(a.err, ERR_BAD_INDEX);
    len = 0;
  }
  // split-KV: CTA (b, split) walks tiles [tbase, tbase + ntiles) of its sequence
  const int all_tiles = (len + TP - 1) / TP;
  const int per_split = (all_tiles + (int)gridDim.y - 1) / (int)gridDim.y;
  const int tbase = (int)blockIdx.y * per_split;
  const int ntiles = all_tiles - tbase < per_split ? (all_tiles - tbase > 0 ? all_tiles - tbase : 0)
                                                   : per_split;
  auto bar = [&](int i) { return smem_u32(&s_bar[i]); };
  if (tid == 0) {
    // S and Z each complete on the commits of two issuing threads
    for (int i = 0; i < MB_N; ++i)
      mbar_init(bar(i), i == MB_S0 || i == MB_S1 || i == MB_Z ? 2 : 1);
    mbar_fence_init();
    s_abort = 0;
    s_rescale[0] = s_rescale[1] = 0;
    s_stop = 0;
    s_loads[0] = s_loads[1] = 0;  // tiles requested into each buffer (the drain's parity)
    s_mmas = 0;                   // value products issued
    s_smmas[0] = s_smmas[1] = 0;  // score products issued into each S buffer
  }
  if (warp == 0) tmem_alloc(smem_u32(&s_tmem), 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tm = s_tmem;
  auto wait = [&](int i, uint32_t parity) {
    if (!mbar_wait(bar(i), parity)) s_abort = 1;
    return s_abort == 0;
  };

  if (warp >= 8) {
    // ---- issuers (lane 0 of warps 8-11).  One thread issues a tcgen05 product every ~90
    //      cycles here (measured; two issuing warps reach ~50 between them), so the products
    //      are spread over four warps: warps 8 and 9 issue S of each tile, as two partial sums
    //      over key blocks 0-4 and 5-8, once the tile has landed and the softmax has read that
    //      S buffer's previous tile, so S(t+1) runs while tile t is soft-maxed; warps 10 and
    //      11 issue Z of each tile (latent slices 0-1 | 2-3) once its P is written, and warp
    //      10 then loads the tile two ahead into the buffer Z has finished reading.  Warp 8
    //      loads the queries and the first two tiles.
    if (lane == 0 && ntiles > 0) {
      auto load_tile = [&](int t) {
        const int j = t & 1;
        ++s_loads[j];
        mbar_expect_tx(bar(MB_C0 + j), TILE);
        for (int kb = 0; kb < KB; ++kb)
          tma_load_3d(sb + M_OFF_C + j * TILE + kb * BLK, &maps.c, 64 * kb, TP * (tbase + t), b,
                      bar(MB_C0 + j));
        if (t + PFD < ntiles)  // the tile PFD further on, into L2 while this one is used:
                               // its own load then waits on L2, not on HBM
          for (int kb = 0; kb < KB; ++kb)
            tma_prefetch_3d(&maps.c, 64 * kb, TP * (tbase + t + PFD), b);
      };
      if (warp < 10) {
        // S = Q C^T: M = 64 heads (A = Q), N = 64 positions (B = C), both K-major
        constexpr uint32_t ID_S = idesc(1, 64, 64, 0, 0);
        const int kb0 = warp == 8 ? 0 : 5, kb1 = warp == 8 ? 5 : KB;
        const uint32_t d0 = warp == 8 ? M_TM_S : M_TM_S2;
        if (warp == 8) {
          mbar_expect_tx(bar(MB_Q), KB * MH * 128);
          for (int kb = 0; kb < KB; ++kb)
            tma_load_3d(sb + M_OFF_Q + kb * MH * 128, &maps.q, 64 * kb, 0, b, bar(MB_Q));
          load_tile(0);
          if (ntiles > 1) load_tile(1);
        }
        const bool go = wait(MB_Q, 0);
        for (int t = 0; t < ntiles && go; ++t) {
          const int j = t & 1;
          if (!wait(MB_C0 + j, (uint32_t)((t >> 1) & 1))) break;  // tile t landed
          // S buffer j was last read by the softmax of tile t - 2
          if (t >= 2 && !wait(MB_SF0 + j, (uint32_t)(((t >> 1) - 1) & 1))) break;
          tc_fence_after();
          for (int kb = kb0; kb < kb1; ++kb)
            for (int ks = 0; ks < 4; ++ks) {
              const uint64_t ad = sdesc_sw128(sb + M_OFF_Q + kb * MH * 128 + ks * 32, 16, 1024);
              const uint64_t bd =
                  sdesc_sw128(sb + M_OFF_C + j * TILE + kb * BLK + ks * 32, 16, 1024);
              mma_bf16_ss(tm + d0 + 64 * j, ad, bd, ID_S, (kb != kb0 || ks) ? 1u : 0u);
            }
          mma_commit(bar(MB_S0 + j));
          if (warp == 8) ++s_smmas[j];
        }
      } else {
        // Z^T = C^T P^T: M = 128 latent (A = C^T, MN-major), N = 64 heads (B = P, K-major)
        constexpr uint32_t ID_Z = idesc(1, 128, 64, 1, 0);
        const int sl0 = warp == 10 ? 0 : 2;
        for (int t = 0; t < ntiles; ++t) {
          const int j = t & 1;
          if (!wait(MB_P, (uint32_t)(t & 1))) break;  // P(t) written, Z rescaled
          tc_fence_after();
          const uint32_t tile = sb + M_OFF_C + j * TILE;
          for (int sl = sl0; sl < sl0 + 2; ++sl)
            for (int ks = 0; ks < TP / 16; ++ks) {
              // A = C^T: latent 128 sl .. 128 sl + 127 = key blocks 2 sl, 2 sl + 1 (BLK
              // apart), positions 16 ks .. 16 ks + 15 (two 8-row groups of 1 KB); B = P rows
              const uint64_t ad = sdesc_sw128(tile + 2 * sl * BLK + ks * 2048, BLK, 1024);
              const uint64_t bd = sdesc_sw128(tile + (KB - 1) * BLK + ks * 32, 16, 1024);
              mma_bf16_ss(tm + M_TM_Z + 64 * sl, ad, bd, ID_Z, (t > 0 || ks > 0) ? 1u : 0u);
            }
          mma_commit(bar(MB_Z));
          if (warp == 10) {
            ++s_mmas;
            if (t + 2 < ntiles) {  // buffer j is free once both halves of Z(t) have read it
              if (!wait(MB_Z, (uint32_t)(t & 1))) break;
              load_tile(t + 2);
            }
          }
        }
      }
    }
  } else {
    // ---- softmax warps: warps w and w + 4 share TMEM lane quarter w & 3, the first taking
    //      positions 0-31 of a tile and the second 32-63; the tile's maximum is exchanged
    //      through shared memory, and each half keeps its own running sum l (both halves
    //      scale by the same factor, so l is their sum at the end) -------------------------
    const int qw = warp & 3, hf = warp >> 2;
    const uint32_t lane_off = (uint32_t)(32 * qw) << 16;
    const bool owner = lane < 16;          // lane l < 16 owns head 16 (w & 3) + l (with l + 16)
    const int hd = 16 * qw + (lane & 15);
    float m_run = -INFINITY, l_run = 0.f;
    for (int t = 0; t < ntiles; ++t) {
      const int j = t & 1;
      // a wait that runs out only raises s_abort: the eight warps leave together, after a
      // named barrier, on one thread's reading of it (never between named barriers)
      wait(MB_S0 + j, (uint32_t)((t >> 1) & 1));
      tc_fence_after();
      uint8_t *tile = sm + M_OFF_C + j * TILE;
      const int p0 = TP * (tbase + t) + 32 * hf;  // this half's first position
      float x[32];
      {
        float v[32];
        tmem_ld32(tm + lane_off + M_TM_S + 64 * j + 32 * hf, x);
        tmem_ld32(tm + lane_off + M_TM_S2 + 64 * j + 32 * hf, v);
        tmem_wait_ld();
#pragma unroll
        for (int c = 0; c < 32; ++c)
          x[c] = p0 + c < len ? (x[c] + v[c]) * a.scale_log2 : -INFINITY;
      }
      // the owner of head hd (lane l < 16) hands its scores for positions 16-31 of this half
      // to lane l + 16, so all 32 lanes take 16 weights each
      const int sub = lane >> 4;
      float xs[16];
#pragma unroll
      for (int c = 0; c < 16; ++c) {
        const float up = __shfl_sync(0xffffffffu, x[16 + c], lane & 15);
        xs[c] = sub ? up : x[c];
      }
      float mt = -INFINITY;
#pragma unroll
      for (int c = 0; c < 16; ++c) mt = fmaxf(mt, xs[c]);
      mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 16));
      if (owner) s_pmax[hf][hd] = mt;
      tc_fence_before();
      asm volatile("bar.sync 1, 256;" ::: "memory");
      if (tid == 0) mbar_arrive(bar(MB_SF0 + j));  // S buffer j has been read
      {
        // the running maximum: the largest weight is exactly 1 (no bf16 rounding on the
        // dominant term; a reference allowed to lag by up to 2^8 measured 1.04e-2 of RMS on
        // peaked rows, over the bound)
        const float mn = fmaxf(m_run, fmaxf(mt, s_pmax[hf ^ 1][hd]));
        const float al = mn == -INFINITY ? 1.f : ex2f_sfu(m_run - mn);  // 2^(-inf) = 0
        float ls = 0.f;
        uint8_t *prow = tile + (KB - 1) * BLK;
#pragma unroll
        for (int q = 0; q < 2; ++q) {  // this lane's 16 weights: two 16-byte chunks of P's row
          uint32_t w[4];
#pragma unroll
          for (int y = 0; y < 4; ++y) {
            const float e0 = xs[8 * q + 2 * y] == -INFINITY ? 0.f : ex2f_sfu(xs[8 * q + 2 * y] - mn);
            const float e1 =
                xs[8 * q + 2 * y + 1] == -INFINITY ? 0.f : ex2f_sfu(xs[8 * q + 2 * y + 1] - mn);
            const __nv_bfloat16 b0 = __float2bfloat16_rn(e0), b1 = __float2bfloat16_rn(e1);
            ls += __bfloat162float(b0) + __bfloat162float(b1);  // the weights the product uses
            w[y] = (uint32_t)__bfloat16_as_ushort(b0) | ((uint32_t)__bfloat16_as_ushort(b1) << 16);
          }
          *reinterpret_cast<uint4 *>(prow + sw128_row(hd, 4 * hf + 2 * sub + q)) =
              make_uint4(w[0], w[1], w[2], w[3]);
        }
        l_run = l_run * al + ls;  // this lane's part of the head's normaliser
        m_run = mn;
        if (hf == 0 && owner) {
          s_alpha[hd] = al;
          if (t > 0 && al != 1.f) s_rescale[j] = 1;
        }
      }
      // a position past the sequence: its latent row must not reach Z (its memory may hold
      // anything, and 0 x NaN is NaN)
      if (tid < TP && TP * (tbase + t) + tid >= len) {
#pragma unroll 1
        for (int kb = 0; kb < KB - 1; ++kb)
#pragma unroll
          for (int q = 0; q < 8; ++q)
            *reinterpret_cast<uint4 *>(tile + kb * BLK + sw128_row(tid, q)) =
                make_uint4(0, 0, 0, 0);
      }
      // all of the above overlaps the previous tile's value product; the rescale needs it done
      if (t > 0) wait(MB_Z, (uint32_t)((t - 1) & 1));
      tc_fence_after();
      asm volatile("bar.sync 1, 256;" ::: "memory");
      if (s_rescale[j]) {  // Z^T columns of the heads whose maximum moved: slices 2 hf, 2 hf + 1
#pragma unroll 1
        for (int sl = 2 * hf; sl < 2 * hf + 2; ++sl) {  // a slice's 64 columns per round trip
          float v[32], w2[32];
          const uint32_t col = M_TM_Z + 64 * sl;
          tmem_ld32(tm + lane_off + col, v);
          tmem_ld32(tm + lane_off + col + 32, w2);
          tmem_wait_ld();
#pragma unroll
          for (int c = 0; c < 32; ++c) v[c] *= s_alpha[c], w2[c] *= s_alpha[32 + c];
          tmem_st32(tm + lane_off + col, v);
          tmem_st32(tm + lane_off + col + 32, w2);
        }
        tmem_wait_st();
      }
      fence_proxy_async();  // P and the zeroed rows feed the tensor core
      tc_fence_before();
      if (tid == 0) s_stop = s_abort;
      asm volatile("bar.sync 1, 256;" ::: "memory");
      if (tid == 0) {
        s_rescale[j] = 0;
        mbar_arrive(bar(MB_P));
      }
      if (s_stop) break;
    }
    l_run += __shfl_xor_sync(0xffffffffu, l_run, 16);  // lanes l and l + 16: one head
    if (owner) {
      if (hf == 0) s_l[hd] = l_run, s_mfin[hd] = m_run;
      else s_lpart[hd] = l_run;
    }
  }
  __syncthreads();
  if (tid < MH) s_l[tid] += s_lpart[tid];
  __syncthreads();

  // ---- z = Z / l per head (softmax warps: thread = latent channel of its lane quarter;
  //      warps w and w + 4 take slices 0-1 and 2-3) ------------------------------------------
  if (warp < 8) {
    // the warp shares the outcome (its tensor-memory loads below are warp-wide)
    const bool done = __all_sync(0xffffffffu, ntiles > 0 && !s_abort &&
                                                  wait(MB_Z, (uint32_t)((ntiles - 1) & 1))) != 0;
    tc_fence_after();
    const int qw = warp & 3, hf = warp >> 2;
    const uint32_t lane_off = (uint32_t)(32 * qw) << 16;
    // one split: z = Z / l; several: this split's unnormalised Z with its (m, l) per head
    const bool split = gridDim.y > 1;
    const size_t row = (size_t)blockIdx.y * a.B + b;
    float *z = split ? a.part + row * MH * ML : a.z + (size_t)b * MH * ML;
#pragma unroll 1
    for (int sl = 2 * hf; sl < 2 * hf + 2; ++sl)
#pragma unroll 1
      for (int hh = 0; hh < 2; ++hh) {
        float v[32];
        if (done) {
          tmem_ld32(tm + lane_off + M_TM_Z + 64 * sl + 32 * hh, v);
          tmem_wait_ld();
        }
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          const int head = 32 * hh + c;
          const float l = s_l[head];
          z[(size_t)head * ML + 128 * sl + 32 * qw + lane] =
              split ? (done ? v[c] : 0.f) : ((done && l > 0.f) ? v[c] / l : 0.f);
        }
      }
    if (split && tid < MH) {  // (m in log2 units, l) of each head; an empty range: (-inf, 0)
      float *ml = a.part + (size_t)gridDim.y * a.B * MH * ML + (row * MH + tid) * 2;
      ml[0] = done ? s_mfin[tid] : -INFINITY;
      ml[1] = done ? s_l[tid] : 0.f;
    }
  }
  if (tid == 128 && s_abort) {
    // a bounded wait ran out: let the copies and products in flight land (bounded) before
    // the CTA releases its memory, then report it
    for (int j = 0; j < 2; ++j)
      if (s_loads[j]) mbar_wait(bar(MB_C0 + j), (s_loads[j] - 1) & 1);
    for (int j = 0; j < 2; ++j)
      if (s_smmas[j]) mbar_wait(bar(MB_S0 + j), (s_smmas[j] - 1) & 1);
    if (s_mmas) mbar_wait(bar(MB_Z), (s_mmas - 1) & 1);
    if (a.err) atomicOr(a.err, ERR_MBAR_TIMEOUT);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tm, 512);
}

// z[b][h] = sum_s 2^(m_s - M) Z_s / sum_s 2^(m_s - M) l_s over the splits (M = max_s m_s).
// The splits' (m, l) come into shared memory once (one thread each); the partial sums' loads
// do not depend on the running sums, so eight of them are in flight at a time.
__global__ void __launch_bounds__(128) mla_combine_kernel(const MlaArgs a, int n_split) {
  __shared__ float s_m[64], s_l[64];  // n_split <= 64
  const int b = blockIdx.x, h = blockIdx.y, tid = threadIdx.x;
  const float *ml = a.part + (size_t)n_split * a.B * MH * ML;
  if (tid < n_split) {
    const float *p = ml + (((size_t)tid * a.B + b) * MH + h) * 2;
    s_m[tid] = p[0];
    s_l[tid] = p[1];
  }
  __syncthreads();
  float M = -INFINITY;
  for (int sp = 0; sp < n_split; ++sp) M = fmaxf(M, s_m[sp]);
  float acc[4] = {0.f, 0.f, 0.f, 0.f}, L = 0.f;
#pragma unroll 8
  for (int sp = 0; sp < n_split; ++sp) {  // an empty split (m = -inf) has Z = 0, l = 0: weight 0
    const float m = s_m[sp];
    const float w = m == -INFINITY ? 0.f : exp2f(m - M);
    const size_t row = (size_t)sp * a.B + b;
    const float4 zz = *reinterpret_cast<const float4 *>(a.part + (row * MH + h) * ML + 4 * tid);
    L = fmaf(w, s_l[sp], L);
    acc[0] = fmaf(w, zz.x, acc[0]), acc[1] = fmaf(w, zz.y, acc[1]);
    acc[2] = fmaf(w, zz.z, acc[2]), acc[3] = fmaf(w, zz.w, acc[3]);
  }
  const float r = L > 0.f ? 1.f / L : 0.f;
  *reinterpret_cast<float4 *>(a.z + ((size_t)b * MH + h) * ML + 4 * tid) =
      make_float4(acc[0] * r, acc[1] * r, acc[2] * r, acc[3] * r);
}


// [n3][rows][576] bf16, boxes of 64 elements x box_rows rows, 128-byte swizzle
bool mla_map(CUtensorMap *m, const void *ptr, int64_t rows, int64_t n3, uint32_t box_rows) {
  auto fn = tensor_map_encoder();
  if (!fn) return false;
  cuuint64_t dims[3] = {(cuuint64_t)MK, (cuuint64_t)rows, (cuuint64_t)n3};
  cuuint64_t strides[2] = {(cuuint64_t)MK * 2, (cuuint64_t)rows * MK * 2};
  cuuint32_t box[3] = {64, box_rows, 1};
  cuuint32_t es[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(ptr), dims, strides, box,
            es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// the split partial sums of one mla_decode_latent_noalloc call (one wave of CTAs on up to
// 191 SMs fits); cudaGetSymbolAddress gives each device's copy
constexpr size_t MLA_STATIC_SCRATCH = (size_t)24 << 20;
__device__ __align__(256) unsigned char g_mla_scratch[MLA_STATIC_SCRATCH];

}  // namespace

size_t mla_static_scratch_bytes() { return MLA_STATIC_SCRATCH; }

// The device address of this device's copy of the buffer, looked up with that device current
// (a host-side name of a __device__ array is not a device address).  Looked up on every call,
// under a lock: the lookup is cheap next to the launches, and a cached address would outlive
// a device reset that reloads the module.
void *mla_static_scratch() {
  static std::mutex lock;
  std::lock_guard<std::mutex> guard(lock);
  void *p = nullptr;
  if (cudaGetSymbolAddress(&p, g_mla_scratch) != cudaSuccess) return nullptr;
  return p;
}

// a split count set by mla_set_split_override (0: none)
std::atomic<int> g_split_override{0};

// splits per sequence: as many CTAs as fill the SMs in one wave (one CTA per SM fits; a
// second, partial wave costs more than the split saves), each split at least 8 tiles (512
// positions); mla_set_split_override(n) forces n (1..64, tuning and tests)
int mla_preferred_split(int n_seqs, int64_t cache_len) {
  if (const int n = g_split_override.load()) return n;
  int dev = 0, nsm = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || nsm < 1)
    nsm = 1;
  if (n_seqs < 1) return 1;
  const int64_t tiles = (cache_len + TP - 1) / TP;
  int64_t want = nsm / n_seqs;
  const int64_t most = tiles / 8 > 1 ? tiles / 8 : 1;
  if (want > most) want = most;
  if (want > 64) want = 64;
  return want > 1 ? (int)want : 1;
}

bool mla_set_split(int n) {
  if (n < 0 || n > 64) return false;
  g_split_override.store(n);
  return true;
}

size_t mla_split_bytes(int n_split, int n_seqs) {
  return n_split > 1 ? (size_t)n_split * n_seqs * MH * (ML + 2) * sizeof(float) : 0;
}

bool mla_latent_supported() {
  int dev = 0, major = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess)
    return false;
  return major == 10 && tensor_map_encoder() != nullptr;
}

cudaError_t launch_mla_latent(const MlaArgs &a, cudaStream_t s) {
  if (a.B == 0) return cudaSuccess;
  MlaMaps maps;
  memset(&maps, 0, sizeof maps);
  if (!mla_map(&maps.q, a.q_cat, MH, a.B, MH) ||
      !mla_map(&maps.c, a.cache, a.L_max > 0 ? a.L_max : 1, a.B, TP))
    return cudaErrorInvalidValue;
  static std::atomic<bool> attr_set[64];  // the opt-in done, per device (idempotent if raced)
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !attr_set[dev].load()) {
    cudaError_t e = cudaFuncSetAttribute(mla_latent_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, M_SMEM);
    if (e != cudaSuccess) return e;
    attr_set[dev].store(true);
  }
  const int ns = a.n_split > 1 ? a.n_split : 1;
  mla_latent_kernel<<<dim3(a.B, ns), MLA_NT, M_SMEM, s>>>(a, maps);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || ns == 1) return e;
  mla_combine_kernel<<<dim3(a.B, MH), 128, 0, s>>>(a, ns);
  return cudaGetLastError();
}

}  // namespace kda

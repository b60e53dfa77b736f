// kda_prefill_tc.cu -- chunked KDA prefill on the 5th-generation tensor cores (sm_103a).
//
// What it computes is the per-head recurrence of the KDA token mixer ("Ling-3.1-flash: a
// 560B hybrid-attention MoE, counted from its safetensors headers", section "How KDA and MLA
// split the work", the state equation; delta-rule write and the -5 log-retention bound from
// "Ling-3.1-flash: Grouped Routing and Two Different MLA Caches", section "KDA replaces a
// token list with a recurrent matrix").  Chunks of C = 64 tokens are processed with the
// WY/UT form of the delta rule, which reaches the token recurrence exactly in exact
// arithmetic.  With per-channel cumulative log-retention gam_r (inclusive of token r) and
// Gamma_r = exp(gam_r), inside a chunk starting from state S:
//     A[r,s] = beta_r sum_i k_ri k_si exp(gam_ri - gam_si)   (s < r)
//     P[r,s] = sum_i q_ri k_si exp(gam_ri - gam_si)          (s <= r)
//     T = (I + A)^-1 = I + T'
//     U = beta V + T' beta V,  W = beta (K*Gamma) + T' beta (K*Gamma)
//     u = U - W S                                           (corrected writes)
//     O = (Q*Gamma) S + P u
//     S <- Diag(Gamma_C) S + (K * Gamma_C/Gamma)^T u
// The pairwise decay exp(gam_r - gam_s) spans up to 64 * 5 = 320 nats, beyond fp32's range
// as a product of two factors, so A and P are built per 16-token row block R with the
// block start gam_R0 as reference: k_r exp(gam_r - gam_R0) in [e^-80, 1] against
// k_s exp(gam_R0 - gam_s), which is <= 1 for s before the block and <= e^80 inside it.
//
// Work layout: one CTA (256 threads, one CTA per SM) per (head, sequence); chunks walked in
// order.  The fp32 state lives in tensor memory, transposed (lane = value channel j,
// column = key channel i), and is fed to the tensor core directly as the A operand.
//   TMEM columns   [0,128) S^T   [128,256) T1   [256,384) T2   [384,512) T3
// MMA precision: intra-chunk products and S^T-reads in tf32 (operands rounded to nearest);
// the state update S += Kbar^T u as three bf16 products (hi*hi + hi*lo + lo*hi), which
// keeps the state at fp32-level accuracy.  Inputs arrive by TMA in 128-byte-swizzled tiles.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "kda_common.cuh"
#include "kda_prefill_tc.h"
#include "kda_tc_ptx.cuh"

namespace kda {
namespace {

using namespace tc;

constexpr int C = 64, D = 128, NT = 256;
constexpr float LOG2E = 1.4426950408889634f;

// Dynamic shared memory map (bytes from a 1024-aligned base).
constexpr uint32_t OFF_Q = 0;          // q   bf16 [64][128], 2 swizzled boxes of 64 channels
constexpr uint32_t OFF_K = 16384;      // k
constexpr uint32_t OFF_V = 32768;      // v
constexpr uint32_t OFF_G = 49152;      // g -> cumulative log2-retention, fp32, 4 boxes of 32
constexpr uint32_t OFF_GATE = 81920;   // gate logits bf16
constexpr uint32_t OFF_X = 98304;      // 64 KB: AP operand rows / T scratch / [W;Q~] / u hi,lo
constexpr uint32_t OFF_T = 163840;     // 16 KB: T' (tf32, K-major) / Kbar hi (bf16, MN-major)
constexpr uint32_t OFF_P = 180224;     // 16 KB: P' (tf32, K-major)
constexpr uint32_t OFF_A = 196608;     // 16 KB: A (fp32 plain) / Kbar lo
constexpr uint32_t SMEM_BYTES = 212992 + 1024;

constexpr uint32_t TM_S = 0, TM_1 = 128, TM_2 = 256, TM_3 = 384, TM_COLS = 512;

enum { BAR_Q = 0, BAR_K, BAR_V, BAR_G, BAR_GATE, BAR_MMA, NBAR };

// byte offset of (row, channel) in a TMA 128B-swizzled tile of 128-byte rows, element size E
template <int E>
__device__ __forceinline__ uint32_t swz(int row, int ch) {
  constexpr int PER = 128 / E;  // elements per box row
  const uint32_t b = (uint32_t)((ch % PER) * E);
  return (uint32_t)(ch / PER) * 8192u + (uint32_t)row * 128u + ((((b >> 4) ^ (row & 7))) << 4) +
         (b & 15u);
}
// K-major 128B-swizzled tf32 operand with NR rows: panels of 32 channels, NR*128 bytes each
template <int NR>
__device__ __forceinline__ uint32_t kmaj_f32(int row, int ch) {
  const uint32_t b = (uint32_t)((ch & 31) * 4);
  return (uint32_t)(ch >> 5) * (NR * 128u) + (uint32_t)row * 128u +
         ((((b >> 4) ^ (row & 7))) << 4) + (b & 15u);
}
// K-major bf16 operand [rows][64]: a single 128-byte panel
__device__ __forceinline__ uint32_t kmaj_bf16_64(int row, int k) {
  const uint32_t b = (uint32_t)(k * 2);
  return (uint32_t)row * 128u + ((((b >> 4) ^ (row & 7))) << 4) + (b & 15u);
}
// MN-major bf16 operand [K rows][128 MN]: 8-row K groups of two 1 KB MN atoms
__device__ __forceinline__ uint32_t mnmaj_bf16_128(int k, int mn) {
  const uint32_t b = (uint32_t)((mn & 63) * 2);
  return (uint32_t)(k >> 3) * 2048u + (uint32_t)(mn >> 6) * 1024u + (uint32_t)(k & 7) * 128u +
         ((((b >> 4) ^ (k & 7))) << 4) + (b & 15u);
}

__device__ __forceinline__ float bf_at(const uint8_t *tile, int row, int ch) {
  return __bfloat162float(*reinterpret_cast<const bf16 *>(tile + swz<2>(row, ch)));
}
__device__ __forceinline__ float f_at(const uint8_t *tile, int row, int ch) {
  return *reinterpret_cast<const float *>(tile + swz<4>(row, ch));
}

// eight bf16 (channels 8c..8c+7) / four fp32 (channels 4c..4c+3) of row `row`
__device__ __forceinline__ void bf_row8(const uint8_t *tile, int row, int c8, float (&o)[8]) {
  const uint32_t off = (uint32_t)(c8 >> 3) * 8192u + (uint32_t)row * 128u +
                       ((uint32_t)((c8 & 7) ^ (row & 7)) << 4);
  const uint4 u = *reinterpret_cast<const uint4 *>(tile + off);
  o[0] = __uint_as_float(u.x << 16), o[1] = __uint_as_float(u.x & 0xffff0000u);
  o[2] = __uint_as_float(u.y << 16), o[3] = __uint_as_float(u.y & 0xffff0000u);
  o[4] = __uint_as_float(u.z << 16), o[5] = __uint_as_float(u.z & 0xffff0000u);
  o[6] = __uint_as_float(u.w << 16), o[7] = __uint_as_float(u.w & 0xffff0000u);
}
// two fp32 -> packed bf16 pair (round to nearest even), low half = first
__device__ __forceinline__ uint32_t pack_bf2(float a, float b) {
  return (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(a)) |
         ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(b)) << 16);
}
__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }
__device__ __forceinline__ float4 f_row4(const uint8_t *tile, int row, int c4) {
  const uint32_t off = (uint32_t)(c4 >> 3) * 8192u + (uint32_t)row * 128u +
                       ((uint32_t)((c4 & 7) ^ (row & 7)) << 4);
  return *reinterpret_cast<const float4 *>(tile + off);
}

struct Maps {
  CUtensorMap q, k, v, g, gate;
};

template <typename ST, bool GATE>
__global__ void __launch_bounds__(NT, 1)
    prefill_tc_kernel(const TcArgs a, const __grid_constant__ Maps maps) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ float s_beta[C], s_rq[C], s_rk[C], s_pd[C];
  __shared__ float s_g0[D][4];  // log2-retention just before each 16-token block
  __shared__ float s_gC[D], s_GC[D];
  __shared__ float s_red[4][C];
  __shared__ __align__(8) uint64_t s_bar[NBAR];
  __shared__ uint32_t s_tmem, s_abort, s_pend, s_ppar[NBAR];

  const uint32_t raw_u32 = smem_u32(smem_raw);
  const uint32_t pad = (1024u - (raw_u32 & 1023u)) & 1023u;
  uint8_t *sm = smem_raw + pad;
  const uint32_t sb = raw_u32 + pad;

  const int h = blockIdx.x, n = blockIdx.y;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int H = a.H;
  const int64_t bos = a.cu_seqlens[n];
  int64_t eos = a.cu_seqlens[n + 1];
  if (eos < bos) eos = bos;
  const int nchunks = (int)((eos - bos + C - 1) / C);
  const int quarter = warp & 3, half = warp >> 2;
  const int j = 32 * quarter + lane;                    // this thread's TMEM lane
  const uint32_t lane_off = (uint32_t)(32 * quarter) << 16;

  auto bar = [&](int b) { return smem_u32(&s_bar[b]); };

  if (tid == 0) {
    for (int b = 0; b < NBAR; ++b) mbar_init(bar(b), 1);
    mbar_fence_init();
    s_abort = 0;
    s_pend = 0;
    for (int b = 0; b < NBAR; ++b) s_ppar[b] = 0;
  }
  if (warp == 0) tmem_alloc(smem_u32(&s_tmem), TM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tm = s_tmem;

  // issue the TMA loads of chunk c for the buffers in `mask` (thread 0 only)
  auto issue = [&](uint32_t mask, int c) {
    const int t0 = (int)(bos + (int64_t)c * C);
    fence_proxy_async();
    if (mask & (1u << BAR_Q)) {
      mbar_expect_tx(bar(BAR_Q), 16384);
      tma_load_3d(sb + OFF_Q, &maps.q, 0, h, t0, bar(BAR_Q));
      tma_load_3d(sb + OFF_Q + 8192, &maps.q, 64, h, t0, bar(BAR_Q));
    }
    if (mask & (1u << BAR_K)) {
      mbar_expect_tx(bar(BAR_K), 16384);
      tma_load_3d(sb + OFF_K, &maps.k, 0, h, t0, bar(BAR_K));
      tma_load_3d(sb + OFF_K + 8192, &maps.k, 64, h, t0, bar(BAR_K));
    }
    if (mask & (1u << BAR_V)) {
      mbar_expect_tx(bar(BAR_V), 16384);
      tma_load_3d(sb + OFF_V, &maps.v, 0, h, t0, bar(BAR_V));
      tma_load_3d(sb + OFF_V + 8192, &maps.v, 64, h, t0, bar(BAR_V));
    }
    if (mask & (1u << BAR_G)) {
      mbar_expect_tx(bar(BAR_G), 32768);
      for (int bx = 0; bx < 4; ++bx)
        tma_load_3d(sb + OFF_G + 8192 * bx, &maps.g, 32 * bx, h, t0, bar(BAR_G));
    }
    if (GATE && (mask & (1u << BAR_GATE))) {
      mbar_expect_tx(bar(BAR_GATE), 16384);
      tma_load_3d(sb + OFF_GATE, &maps.gate, 0, h, t0, bar(BAR_GATE));
      tma_load_3d(sb + OFF_GATE + 8192, &maps.gate, 64, h, t0, bar(BAR_GATE));
    }
    for (int b = 0; b < NBAR; ++b)
      if (mask & (1u << b)) s_ppar[b] = (uint32_t)(c & 1);
    s_pend |= mask;
  };
  auto commit = [&](uint32_t parity) {  // thread 0: MMAs issued, completion pending
    mma_commit(bar(BAR_MMA));
    s_ppar[BAR_MMA] = parity;
    s_pend |= 1u << BAR_MMA;
  };
  // bounded wait on a barrier phase; on time-out flag the error and abort the CTA
  auto wait = [&](int b, uint32_t parity) {
    if (!mbar_wait(bar(b), parity)) {
      s_abort = 1;
      if (a.err) atomicOr(a.err, ERR_MBAR_TIMEOUT);
    } else if (tid == 0) {
      s_pend &= ~(1u << b);
    }
  };
  auto sync = [&]() {
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    return s_abort == 0;
  };

  // ---- initial state: S^T[j][i] = S0[i][j] ---------------------------------------------
  {
    const ST *s0 = a.init_state
                       ? reinterpret_cast<const ST *>(a.init_state) + ((size_t)n * H + h) * D * D
                       : nullptr;
#pragma unroll
    for (int g32 = 0; g32 < 2; ++g32) {
      float v[32];
      const int i0 = 64 * half + 32 * g32;
#pragma unroll
      for (int x = 0; x < 32; ++x) v[x] = s0 ? to_f(s0[(size_t)(i0 + x) * D + j]) : 0.f;
      tmem_st32(tm + lane_off + TM_S + i0, v);
    }
    tmem_wait_st();
  }
  if (tid == 0 && nchunks > 0)
    issue((1u << BAR_Q) | (1u << BAR_K) | (1u << BAR_V) | (1u << BAR_G) |
              (GATE ? (1u << BAR_GATE) : 0u),
          0);
  bool ok = sync();

  const uint32_t ID_AP = idesc(2, 128, 64, 0, 0);
  const uint32_t ID_S = idesc(2, 128, 128, 0, 0);
  const uint32_t ID_UPD = idesc(1, 128, 128, 0, 1);
  uint32_t mma_par = 0;

  for (int c = 0; c < nchunks && ok; ++c) {
    const int64_t t0 = bos + (int64_t)c * C;
    const int nv = (int)((eos - t0) < C ? (eos - t0) : C);
    const uint32_t par = (uint32_t)(c & 1);
    const bool more = c + 1 < nchunks;

    if (tid < C) s_beta[tid] = tid < nv ? a.beta[(size_t)(t0 + tid) * H + h] : 0.f;
    wait(BAR_Q, par);
    wait(BAR_K, par);
    wait(BAR_G, par);

    // ---- P1: row norms and q.k (threads 0..63); log2-retention prefix sums (128..255) ---
    if (tid < C) {
      const int r = tid;
      float sq = 0.f, sk = 0.f, sqk = 0.f;
      if (r < nv) {
#pragma unroll 2
        for (int c8 = 0; c8 < 16; ++c8) {
          float qv[8], kv[8];
          bf_row8(sm + OFF_Q, r, c8, qv);
          bf_row8(sm + OFF_K, r, c8, kv);
#pragma unroll
          for (int y = 0; y < 8; ++y)
            sq = fmaf(qv[y], qv[y], sq), sk = fmaf(kv[y], kv[y], sk), sqk = fmaf(qv[y], kv[y], sqk);
        }
      }
      const float rq = r < nv ? (a.qk_l2norm ? rsqrtf(sq + a.l2_eps) : 1.f) : 0.f;
      const float rk = r < nv ? (a.qk_l2norm ? rsqrtf(sk + a.l2_eps) : 1.f) : 0.f;
      s_rq[r] = rq, s_rk[r] = rk, s_pd[r] = sqk * rq * rk;
    } else if (tid >= 128) {
      const int i = tid - 128;
      float acc = 0.f;
      for (int r = 0; r < C; ++r) {
        if ((r & 15) == 0) s_g0[i][r >> 4] = acc;
        float *p = reinterpret_cast<float *>(sm + OFF_G + swz<4>(r, i));
        if (r < nv) acc += fmaxf(*p, a.g_min) * LOG2E;
        *p = acc;
      }
      s_gC[i] = acc;
      s_GC[i] = exp2f(acc);
    }
    if (!(ok = sync())) break;

    // ---- P2: AP operands.  A-side in TMEM: rows m of pair pi hold
    //      Khat^(R)[s] = k_s exp(gam_R0 - gam_s) for R = 2pi + m/64, s = m % 64 (zero past
    //      block R); B-side rows in smem: [Ktil_R; Qtil_R] for the pair's two blocks. ------
    {
      const int pi = half, m = j;
      const int R = 2 * pi + (m >> 6), s = m & 63;
      const bool live = s < nv && s <= 16 * R + 15;
      const float rk = s_rk[s];
      const uint32_t dst = tm + lane_off + (pi == 0 ? TM_1 : TM_3);
#pragma unroll 1
      for (int g32 = 0; g32 < 4; ++g32) {
        float v[32];
        if (live) {
#pragma unroll
          for (int c8 = 0; c8 < 4; ++c8) {
            float kv[8];
            bf_row8(sm + OFF_K, s, 4 * g32 + c8, kv);
            const float4 ga = f_row4(sm + OFF_G, s, 8 * g32 + 2 * c8);
            const float4 gb = f_row4(sm + OFF_G, s, 8 * g32 + 2 * c8 + 1);
            const float gg[8] = {ga.x, ga.y, ga.z, ga.w, gb.x, gb.y, gb.z, gb.w};
#pragma unroll
            for (int y = 0; y < 8; ++y) {
              const int i = 32 * g32 + 8 * c8 + y;
              v[8 * c8 + y] = to_tf32(kv[y] * rk * exp2f(s_g0[i][R] - gg[y]));
            }
          }
        } else {
#pragma unroll
          for (int x = 0; x < 32; ++x) v[x] = 0.f;
        }
        tmem_st32(dst + 32 * g32, v);
      }
    }
    {
      const int row = tid >> 1, ph = tid & 1;  // 128 rows, two threads per row
      const int pi = row >> 6, w = row & 63;
      const int R = 2 * pi + (w >> 5), isq = (w >> 4) & 1, r = 16 * R + (w & 15);
      const bool live = r < nv;
      const float rx = isq ? s_rq[r] : s_rk[r];
      const uint8_t *src = sm + (isq ? OFF_Q : OFF_K);
#pragma unroll 1
      for (int c8 = 0; c8 < 8; ++c8) {
        const int i0 = 64 * ph + 8 * c8;
        float xv[8], o[8];
        bf_row8(src, r, i0 >> 3, xv);
        const float4 ga = f_row4(sm + OFF_G, r, i0 >> 2);
        const float4 gb = f_row4(sm + OFF_G, r, (i0 >> 2) + 1);
        const float gg[8] = {ga.x, ga.y, ga.z, ga.w, gb.x, gb.y, gb.z, gb.w};
#pragma unroll
        for (int y = 0; y < 8; ++y)
          o[y] = live ? to_tf32(xv[y] * rx * exp2f(gg[y] - s_g0[i0 + y][R])) : 0.f;
        *reinterpret_cast<float4 *>(sm + OFF_X + kmaj_f32<128>(row, i0)) =
            make_float4(o[0], o[1], o[2], o[3]);
        *reinterpret_cast<float4 *>(sm + OFF_X + kmaj_f32<128>(row, i0 + 4)) =
            make_float4(o[4], o[5], o[6], o[7]);
      }
    }
    tmem_wait_st();
    fence_proxy_async();
    if (!(ok = sync())) break;
    if (tid == 0) {
#pragma unroll
      for (int pi = 0; pi < 2; ++pi)
        for (int ks = 0; ks < 16; ++ks) {
          const uint64_t bd =
              sdesc_sw128(sb + OFF_X + (ks >> 2) * 16384 + 64 * pi * 128 + (ks & 3) * 32, 16, 1024);
          mma_tf32_ts(tm + TM_2 + 64 * pi, tm + (pi == 0 ? TM_1 : TM_3) + 8 * ks, bd, ID_AP,
                      ks > 0);
        }
      commit(mma_par);
    }
    wait(BAR_MMA, mma_par);
    mma_par ^= 1;
    tc_fence_after();

    // ---- P3: A (beta-scaled, strict lower, fp32) and P' (strict lower, tf32) ------------
    {
      const int pi = half, m = j, R = 2 * pi + (m >> 6), s = m & 63;
      float v[32];
      tmem_ld32(tm + lane_off + TM_2 + 64 * pi + 32 * (m >> 6), v);
      tmem_wait_ld();
#pragma unroll
      for (int x = 0; x < 16; ++x) {
        const int r = 16 * R + x;
        const bool low = s < r;
        reinterpret_cast<float *>(sm + OFF_A)[r * 64 + s] = low ? s_beta[r] * v[x] : 0.f;
        *reinterpret_cast<float *>(sm + OFF_P + kmaj_f32<64>(r, s)) =
            low ? to_tf32(v[16 + x]) : 0.f;
      }
    }
    wait(BAR_V, par);
    // (beta V)^T and (beta K Gamma)^T as tf32 A operands in T1 (lane = channel, col = token)
    {
      float v[32];
#pragma unroll 1
      for (int g32 = 0; g32 < 2; ++g32) {
#pragma unroll
        for (int x = 0; x < 32; ++x) {
          const int s = 32 * g32 + x;
          if (s >= nv) {
            v[x] = 0.f;
          } else if (half == 0) {
            v[x] = to_tf32(s_beta[s] * bf_at(sm + OFF_V, s, j));
          } else {
            const float kk = bf_at(sm + OFF_K, s, j) * s_rk[s];
            v[x] = to_tf32(s_beta[s] * kk * exp2f(f_at(sm + OFF_G, s, j)));
          }
        }
        tmem_st32(tm + lane_off + TM_1 + 64 * half + 32 * g32, v);
      }
    }
    tmem_wait_st();
    if (!(ok = sync())) break;

    // ---- P4: T = (I + A)^-1 by blocks of 16; T fp32 in X[0,16K), scratch X[16K,32K) ------
    float *Am = reinterpret_cast<float *>(sm + OFF_A);
    float *Tm = reinterpret_cast<float *>(sm + OFF_X);
    float *Mm = reinterpret_cast<float *>(sm + OFF_X + 16384);
    if (tid < 64) {  // diagonal blocks by forward substitution, one column per thread
      const int R = tid >> 4, cc = tid & 15, b0 = 16 * R;
      float x[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        float acc = 0.f;
#pragma unroll
        for (int k = 0; k < i; ++k)
          if (k >= cc) acc = fmaf(Am[(b0 + i) * 64 + b0 + k], x[k], acc);
        x[i] = i < cc ? 0.f : (i == cc ? 1.f : -acc);
      }
#pragma unroll
      for (int i = 0; i < 16; ++i) Tm[(b0 + i) * 64 + b0 + cc] = x[i];
    }
    if (!(ok = sync())) break;
    for (int dist = 1; dist <= 3; ++dist) {
      const int npairs = 4 - dist;
      for (int e = tid; e < npairs * 256; e += NT) {
        const int p = e >> 8, ai = (e >> 4) & 15, bi = e & 15;
        const int R = dist + p, S = R - dist;
        float acc = 0.f;
        for (int Q = S; Q < R; ++Q)
#pragma unroll
          for (int y = 0; y < 16; ++y)
            acc = fmaf(Am[(16 * R + ai) * 64 + 16 * Q + y], Tm[(16 * Q + y) * 64 + 16 * S + bi], acc);
        Mm[e] = acc;
      }
      __syncthreads();
      for (int e = tid; e < npairs * 256; e += NT) {
        const int p = e >> 8, ai = (e >> 4) & 15, bi = e & 15;
        const int R = dist + p, S = R - dist;
        float acc = 0.f;
#pragma unroll
        for (int x = 0; x < 16; ++x)
          acc = fmaf(Tm[(16 * R + ai) * 64 + 16 * R + x], Mm[(p << 8) + x * 16 + bi], acc);
        Tm[(16 * R + ai) * 64 + 16 * S + bi] = -acc;
      }
      __syncthreads();
    }
    {  // T' = T - I (strict lower), tf32 K-major [r][s]
      const int r = tid >> 2, s0 = (tid & 3) * 16;
#pragma unroll
      for (int c4 = 0; c4 < 4; ++c4) {
        float4 o4;
        float *o = reinterpret_cast<float *>(&o4);
#pragma unroll
        for (int x = 0; x < 4; ++x) {
          const int s = s0 + 4 * c4 + x;
          o[x] = s < r ? to_tf32(Tm[r * 64 + s]) : 0.f;
        }
        *reinterpret_cast<float4 *>(sm + OFF_T + kmaj_f32<64>(r, s0 + 4 * c4)) = o4;
      }
    }
    fence_proxy_async();
    if (!(ok = sync())) break;

    // ---- P5: U' = T' (beta V), W' = T' (beta K Gamma) on the tensor core ----------------
    if (tid == 0) {
      for (int w = 0; w < 2; ++w)
        for (int ks = 0; ks < 8; ++ks) {
          const uint64_t bd = sdesc_sw128(sb + OFF_T + (ks >> 2) * 8192 + (ks & 3) * 32, 16, 1024);
          mma_tf32_ts(tm + TM_2 + 64 * w, tm + TM_1 + 64 * w + 8 * ks, bd, ID_AP, ks > 0);
        }
      commit(mma_par);
    }
    // meanwhile: Qtil = q Gamma into rows 64..127 of the [W; Qtil] operand (X)
    {
      const int i = tid & 127, r0 = 32 * (tid >> 7);
#pragma unroll 4
      for (int x = 0; x < 32; ++x) {
        const int r = r0 + x;
        const float val = r < nv ? bf_at(sm + OFF_Q, r, i) * s_rq[r] * exp2f(f_at(sm + OFF_G, r, i))
                                 : 0.f;
        *reinterpret_cast<float *>(sm + OFF_X + kmaj_f32<128>(64 + r, i)) = to_tf32(val);
      }
    }
    wait(BAR_MMA, mma_par);
    mma_par ^= 1;
    tc_fence_after();

    // ---- P6: U = beta V + U' (kept in T1, fp32); W = beta K Gamma + W' -> X rows 0..63 ---
    {
      float v[32];
#pragma unroll 1
      for (int g32 = 0; g32 < 2; ++g32) {
        tmem_ld32(tm + lane_off + TM_2 + 64 * half + 32 * g32, v);
        tmem_wait_ld();
        if (half == 0) {
#pragma unroll
          for (int x = 0; x < 32; ++x) {
            const int s = 32 * g32 + x;
            if (s < nv) v[x] += s_beta[s] * bf_at(sm + OFF_V, s, j);
          }
          tmem_st32(tm + lane_off + TM_1 + 32 * g32, v);
        } else {
#pragma unroll
          for (int x = 0; x < 32; ++x) {
            const int r = 32 * g32 + x;
            const float kk = r < nv ? bf_at(sm + OFF_K, r, j) * s_rk[r] : 0.f;
            const float w = r < nv ? s_beta[r] * kk * exp2f(f_at(sm + OFF_G, r, j)) + v[x] : 0.f;
            *reinterpret_cast<float *>(sm + OFF_X + kmaj_f32<128>(r, j)) = to_tf32(w);
          }
        }
      }
    }
    tmem_wait_st();
    fence_proxy_async();
    if (!(ok = sync())) break;
    if (tid == 0 && more) issue((1u << BAR_Q) | (1u << BAR_V), c + 1);

    // ---- P7: [W; Qtil] S on the tensor core (A = S^T from TMEM) ------------------------
    if (tid == 0) {
      for (int ks = 0; ks < 16; ++ks) {
        const uint64_t bd = sdesc_sw128(sb + OFF_X + (ks >> 2) * 16384 + (ks & 3) * 32, 16, 1024);
        mma_tf32_ts(tm + TM_3, tm + TM_S + 8 * ks, bd, ID_S, ks > 0);
      }
      commit(mma_par);
    }
    // meanwhile: Kbar = k Gamma_C / Gamma as bf16 hi (T region) + lo (A region), MN-major
    {
      const int i = tid & 127, s0 = 32 * (tid >> 7);
      const float gc = s_gC[i];
#pragma unroll 4
      for (int x = 0; x < 32; ++x) {
        const int s = s0 + x;
        const float val = s < nv ? bf_at(sm + OFF_K, s, i) * s_rk[s] *
                                       exp2f(gc - f_at(sm + OFF_G, s, i))
                                 : 0.f;
        const bf16 hi = __float2bfloat16_rn(val);
        const bf16 lo = __float2bfloat16_rn(val - __bfloat162float(hi));
        *reinterpret_cast<bf16 *>(sm + OFF_T + mnmaj_bf16_128(s, i)) = hi;
        *reinterpret_cast<bf16 *>(sm + OFF_A + mnmaj_bf16_128(s, i)) = lo;
      }
    }
    wait(BAR_MMA, mma_par);
    mma_par ^= 1;
    tc_fence_after();
    __syncthreads();
    if (tid == 0 && more) issue((1u << BAR_K) | (1u << BAR_G), c + 1);

    // ---- P8: u = U - W S (fp32 in T1[0,64), tf32 in T1[64,128), bf16 hi/lo in X);
    //      decay S^T by Gamma_C ------------------------------------------------------------
    if (half == 0) {
#pragma unroll 1
      for (int g32 = 0; g32 < 2; ++g32) {
        float ws[32], u[32];
        tmem_ld32(tm + lane_off + TM_3 + 32 * g32, ws);
        tmem_ld32(tm + lane_off + TM_1 + 32 * g32, u);
        tmem_wait_ld();
#pragma unroll
        for (int x = 0; x < 32; ++x) u[x] -= ws[x];
        tmem_st32(tm + lane_off + TM_1 + 32 * g32, u);
#pragma unroll
        for (int x = 0; x < 32; ++x) ws[x] = to_tf32(u[x]);
        tmem_st32(tm + lane_off + TM_1 + 64 + 32 * g32, ws);
#pragma unroll
        for (int c8 = 0; c8 < 4; ++c8) {
          uint32_t hw[4], lw[4];
#pragma unroll
          for (int y = 0; y < 4; ++y) {
            const float a0 = u[8 * c8 + 2 * y], a1 = u[8 * c8 + 2 * y + 1];
            hw[y] = pack_bf2(a0, a1);
            lw[y] = pack_bf2(a0 - bf_lo(hw[y]), a1 - bf_hi(hw[y]));
          }
          const uint32_t off = kmaj_bf16_64(j, 32 * g32 + 8 * c8);
          *reinterpret_cast<uint4 *>(sm + OFF_X + off) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
          *reinterpret_cast<uint4 *>(sm + OFF_X + 16384 + off) =
              make_uint4(lw[0], lw[1], lw[2], lw[3]);
        }
      }
    } else {
#pragma unroll 1
      for (int g32 = 0; g32 < 4; ++g32) {
        float v[32];
        tmem_ld32(tm + lane_off + TM_S + 32 * g32, v);
        tmem_wait_ld();
#pragma unroll
        for (int x = 0; x < 32; ++x) v[x] *= s_GC[32 * g32 + x];
        tmem_st32(tm + lane_off + TM_S + 32 * g32, v);
      }
    }
    tmem_wait_st();
    fence_proxy_async();
    if (!(ok = sync())) break;

    // ---- P9: O += P' u (tf32); S^T += u^T Kbar as hi*hi + hi*lo + lo*hi (bf16) ---------
    if (tid == 0) {
      for (int ks = 0; ks < 8; ++ks) {
        const uint64_t bd = sdesc_sw128(sb + OFF_P + (ks >> 2) * 8192 + (ks & 3) * 32, 16, 1024);
        mma_tf32_ts(tm + TM_3 + 64, tm + TM_1 + 64 + 8 * ks, bd, ID_AP, 1);
      }
      for (int term = 0; term < 3; ++term) {
        const uint32_t a_off = OFF_X + (term == 2 ? 16384 : 0);
        const uint32_t b_off = term == 1 ? OFF_A : OFF_T;
        for (int ks = 0; ks < 4; ++ks) {
          const uint64_t ad = sdesc_sw128(sb + a_off + ks * 32, 16, 1024);
          const uint64_t bd = sdesc_sw128(sb + b_off + ks * 4096, 1024, 2048);
          mma_bf16_ss(tm + TM_S, ad, bd, ID_UPD, 1);
        }
      }
      commit(mma_par);
    }
    wait(BAR_MMA, mma_par);
    mma_par ^= 1;
    tc_fence_after();
    if (GATE) wait(BAR_GATE, par);

    // ---- P10: outputs o_r = scale (O'_r + (q_r.k_r) u_r), norm and gate, store ----------
    {
      float o[32], u[32];
      tmem_ld32(tm + lane_off + TM_3 + 64 + 32 * half, o);
      tmem_ld32(tm + lane_off + TM_1 + 32 * half, u);
      tmem_wait_ld();
#pragma unroll
      for (int x = 0; x < 32; ++x) o[x] = a.scale * fmaf(s_pd[32 * half + x], u[x], o[x]);
      if (GATE) {
        float sq[32];
#pragma unroll
        for (int x = 0; x < 32; ++x) sq[x] = o[x] * o[x];
        // transpose-reduce over the 32 lanes: afterwards sq[0] holds row (32 half + lane)
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) {
          const bool up = (lane & off) != 0;
#pragma unroll
          for (int x = 0; x < off; ++x) {
            const float send = up ? sq[x] : sq[x + off];
            const float recv = __shfl_xor_sync(0xffffffffu, send, off);
            sq[x] = (up ? sq[x + off] : sq[x]) + recv;
          }
        }
        s_red[quarter][32 * half + lane] = sq[0];
      }
      __syncthreads();
      const float w = GATE ? (a.norm_w ? a.norm_w[j] : 1.f) : 1.f;
      bf16 *out = reinterpret_cast<bf16 *>(a.out);
#pragma unroll
      for (int x = 0; x < 32; ++x) {
        const int r = 32 * half + x;
        if (r >= nv) continue;
        float val = o[x];
        if (GATE) {
          const float ss = s_red[0][r] + s_red[1][r] + s_red[2][r] + s_red[3][r];
          val = val * rsqrtf(ss * (1.f / D) + a.norm_eps) * w *
                sigmoidf_(bf_at(sm + OFF_GATE, r, j));
        }
        out[((size_t)(t0 + r) * H + h) * D + j] = __float2bfloat16_rn(val);
      }
    }
    if (!(ok = sync())) break;
    if (GATE && tid == 0 && more) issue(1u << BAR_GATE, c + 1);
  }

  // ---- final state: S[i][j] = S^T[j][i] ------------------------------------------------
  if (ok && a.final_state) {
    ST *dst = reinterpret_cast<ST *>(a.final_state) + ((size_t)n * H + h) * D * D;
#pragma unroll 1
    for (int g32 = 0; g32 < 2; ++g32) {
      float v[32];
      const int i0 = 64 * half + 32 * g32;
      tmem_ld32(tm + lane_off + TM_S + i0, v);
      tmem_wait_ld();
#pragma unroll
      for (int x = 0; x < 32; ++x) dst[(size_t)(i0 + x) * D + j] = from_f<ST>(v[x]);
    }
  }
  if (!ok && tid == 0) {
    // drain: let loads and MMAs still in flight land (bounded) before the CTA exits
    for (int b = 0; b < NBAR; ++b)
      if (s_pend & (1u << b)) mbar_wait(bar(b), s_ppar[b]);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tm, TM_COLS);
}

// ---- host side --------------------------------------------------------------------------

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static bool tried = false;
  if (!tried) {
    tried = true;
    cudaDriverEntryPointQueryResult q;
    void *p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

bool make_map(CUtensorMap *m, const void *ptr, bool f32, int64_t T, int H) {
  const int esz = f32 ? 4 : 2;
  cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)T};
  cuuint64_t strides[2] = {(cuuint64_t)D * esz, (cuuint64_t)H * D * esz};
  cuuint32_t box[3] = {(cuuint32_t)(128 / esz), 1, (cuuint32_t)C};
  cuuint32_t es[3] = {1, 1, 1};
  auto fn = encode_fn();
  if (!fn) return false;
  return fn(m, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
            const_cast<void *>(ptr), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <typename ST, bool GATE>
cudaError_t launch_typed(const TcArgs &a, const Maps &maps, cudaStream_t s) {
  static bool attr_set[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !attr_set[dev]) {
    cudaError_t e = cudaFuncSetAttribute(prefill_tc_kernel<ST, GATE>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  prefill_tc_kernel<ST, GATE><<<dim3(a.H, a.n_seqs), NT, SMEM_BYTES, s>>>(a, maps);
  return cudaGetLastError();
}

}  // namespace

bool prefill_tc_supported(int d, bool io_bf16) {
  if (d != D || !io_bf16) return false;
  int dev = 0, major = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess)
    return false;
  return major == 10 && encode_fn() != nullptr;
}

cudaError_t launch_prefill_tc(const TcArgs &a, int64_t total_tokens, bool st_bf16,
                              cudaStream_t s) {
  if (a.n_seqs == 0) return cudaSuccess;
  Maps maps;
  memset(&maps, 0, sizeof maps);
  if (total_tokens > 0) {
    if (total_tokens >= ((int64_t)1 << 31)) return cudaErrorInvalidValue;
    if (!make_map(&maps.q, a.q, false, total_tokens, a.H) ||
        !make_map(&maps.k, a.k, false, total_tokens, a.H) ||
        !make_map(&maps.v, a.v, false, total_tokens, a.H) ||
        !make_map(&maps.g, a.g, true, total_tokens, a.H) ||
        (a.gate && !make_map(&maps.gate, a.gate, false, total_tokens, a.H)))
      return cudaErrorInvalidValue;
  }
  const bool gate = a.gate != nullptr;
  if (st_bf16)
    return gate ? launch_typed<bf16, true>(a, maps, s) : launch_typed<bf16, false>(a, maps, s);
  return gate ? launch_typed<float, true>(a, maps, s) : launch_typed<float, false>(a, maps, s);
}

}  // namespace kda

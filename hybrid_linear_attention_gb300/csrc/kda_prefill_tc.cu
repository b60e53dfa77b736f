// kda_prefill_tc.cu -- chunked KDA prefill on the 5th-generation tensor cores (sm_103a).
//
// What it computes is the per-head recurrence of the KDA token mixer ("Ling-3.1-flash: a
// 560B hybrid-attention MoE, counted from its safetensors headers", section "How KDA and MLA
// split the work", the state equation; delta-rule write and the -5 log-retention bound from
// "Ling-3.1-flash: Grouped Routing and Two Different MLA Caches", section "KDA replaces a
// token list with a recurrent matrix").  Chunks of C = 64 tokens are processed in the WY/UT
// form of the delta rule, which reaches the token recurrence exactly in exact arithmetic.
// With per-channel cumulative log-retention gam_r (inclusive of token r), Gamma_r =
// exp(gam_r), and the chunk's incoming state S (d_k x d_v):
//     A[r,s] = beta_r sum_i k_ri k_si exp(gam_ri - gam_si)   (s < r)
//     P[r,s] = sum_i q_ri k_si exp(gam_ri - gam_si)          (s < r; diagonal q_r.k_r)
//     T      = (I + A)^-1
//     X      = [K*Gamma ; Q*Gamma] S                         (what S predicts / reads)
//     u      = T beta (V - (K*Gamma) S)                      (the corrected writes)
//     O      = (Q*Gamma) S + P u
//     S     <- Diag(Gamma_C) S + (K * Gamma_C/Gamma)^T u
// The pairwise decay exp(gam_r - gam_s) spans up to 64 * 5 = 320 nats, beyond fp32's range
// as a product of two factors, so A and P are built per 16-token row block R with the
// block start gam_R0 as reference: k_r exp(gam_r - gam_R0) in [e^-80, 1] against
// k_s exp(gam_R0 - gam_s), which is <= 1 for s before the block and <= e^80 inside it.
//
// Work layout: one CTA (384 threads, one CTA per SM) per (head, sequence); chunks walked in
// order.  The fp32 state lives in tensor memory, transposed (lane = value channel j,
// column = key channel i), and is fed to the tensor core directly as the A operand.
//   TMEM columns   [0,128) S^T   [128,256) TA   [256,384) TB   [384,512) TC
// The read of the state by the query rows, O = (Q Gamma) S + P u, can nearly cancel, so a
// tf32 rounding of either factor (the tensor core also truncates a tf32 operand it reads from
// tensor memory) would show in the output after its norm: the state read X = [K Gamma;
// Q Gamma] S is three bf16 products (hi*hi + hi*lo + lo*hi) of [K Gamma; Q Gamma] and of the
// state split into bf16 hi + lo (the split state kept in TA while TA is otherwise idle), good
// to ~2^-16, one product of N = 128 for the key and the query rows together.
// A and P (64 x 64 each, K = 128) come from one product on the tensor core:
// [Ktil; Qtil] (128 rows, bf16 hi + lo in tensor memory) times the stacked Khat^(R) rows
// (160, bf16 in shared memory), hi*hi everywhere and hi*lo + lo*hi on the band (a 16-token
// block and the one before it), where q_r.k_s can nearly cancel with little decay.
// MMA precision elsewhere: tf32 (operands rounded to nearest; beta(V - KGS) split into tf32
// hi + lo); the state update S += Kbar^T u as three bf16 products
// (hi*hi + hi*lo + lo*hi), which keeps the state at fp32-level accuracy.  Inputs arrive by
// TMA in 128-byte-swizzled tiles; every operand is built with 16-byte vector accesses.
#include <cuda.h>
#include <atomic>
#include <cstdlib>
#include <cstring>
#include <cudaTypedefs.h>

#include "kda_common.cuh"
#include "kda_prefill_tc.h"
#include "kda_tc_ptx.cuh"

extern __shared__ uint8_t prefill_dyn_smem[];  // the dynamic shared memory base

namespace kda {
namespace {

using namespace tc;

constexpr int C = 64, D = 128, NT = 384;
constexpr float LOG2E = 1.4426950408889634f;

// Dynamic shared memory map (bytes from a 1024-aligned base).
constexpr uint32_t OFF_Q = 0;        // q bf16 [64][128], two 128B-swizzled boxes of 64 channels
constexpr uint32_t OFF_K = 16384;    // k
constexpr uint32_t OFF_V = 32768;    // v
constexpr uint32_t OFF_G = 49152;    // g -> cumulative log2-retention, fp32, 4 boxes of 32
constexpr uint32_t OFF_X = 81920;    // 64 KB: [K Gamma; Q Gamma] bf16 hi | lo -> Kbar hi | Kbar lo |
                                     //        u hi | u lo
constexpr uint32_t OFF_T = 147456;   // 16 KB: T fp32 (plain) -> T tf32 (K-major)
constexpr uint32_t OFF_P = 163840;   // 16 KB: P' tf32 (K-major)
constexpr uint32_t OFF_A = 180224;   // 17 KB: A fp32, rows of LDA floats
constexpr int LDA = 68;              // A row stride: rows 16 bytes apart in the bank map
// the one-CTA inverse's scratch, four 16 x 16 fp32 blocks past A, over the band lo rows of the
// A/P product's B operand (dead once that product is done)
constexpr uint32_t OFF_SCR = OFF_A + 64 * LDA * 4;
// B operand of the A/P product (bf16, K-major), live until that product completes, over
// T, P' and A: Khat^(R) rows, 48 far then 112 band (hi), and the band rows' lo parts
constexpr uint32_t OFF_BH = 147456;  // 160 rows x 128 channels x 2 B = 40 KB
constexpr uint32_t OFF_BL = 188416;  // 112 rows: 28 KB
constexpr uint32_t SMEM_BYTES = 217088 + 1024;

constexpr uint32_t TM_S = 0, TM_A = 128, TM_B = 256, TM_C = 384, TM_COLS = 512;
// during the A/P product: [Ktil; Qtil] bf16 hi and lo (64 columns each), result 160 columns
constexpr uint32_t TM_AH = 128, TM_AL = 192, TM_D = 256;

// TMA loads and tensor-core completion; in a cluster pair, the consumer's FULL (landing
// buffer 0 / 1 holds T and P') and the producer's EMPTY (buffer 0 / 1 may be rewritten)
// (a cluster-pair consumer commits its state read on BAR_X: it issues that product from another
// thread than the rest, and a commit tracks only the products of the thread that issues it)
enum { BAR_Q = 0, BAR_K, BAR_V, BAR_G, BAR_MMA, BAR_F0, BAR_F1, BAR_E0, BAR_E1, BAR_GT, BAR_X,
       NBAR };
// consumer landing buffers b = 0, 1: T then P' (16 KB each, tf32 K-major); buffer 0 is the
// fused kernel's own T and P' region
__host__ __device__ constexpr uint32_t off_lt(int b) { return 147456u + 32768u * (uint32_t)b; }
__host__ __device__ constexpr uint32_t off_lp(int b) { return off_lt(b) + 16384u; }
static_assert(off_lt(0) == OFF_T && off_lp(0) == OFF_P, "landing buffer 0 = T, P' regions");
static_assert(off_lp(1) + 16384u <= 217088u, "landing buffers inside the shared memory map");
static_assert(OFF_SCR % 16 == 0 && OFF_SCR + 4 * 256 * 4 <= 217088u, "inverse scratch inside the map");

// K-major 128B-swizzled tf32 operand with NR rows: panels of 32 channels, NR*128 bytes each
template <int NR>
__device__ __forceinline__ uint32_t kmaj_f32(int row, int ch) {
  const uint32_t b = (uint32_t)((ch & 31) * 4);
  return (uint32_t)(ch >> 5) * (NR * 128u) + (uint32_t)row * 128u +
         ((((b >> 4) ^ (row & 7))) << 4) + (b & 15u);
}
// K-major 128B-swizzled bf16 operand with NR rows and 128 channels: two panels of 64
template <int NR>
__device__ __forceinline__ uint32_t kmaj_bf16(int row, int ch) {
  const uint32_t b = (uint32_t)((ch & 63) * 2);
  return (uint32_t)(ch >> 6) * (NR * 128u) + (uint32_t)row * 128u +
         ((((b >> 4) ^ (row & 7))) << 4) + (b & 15u);
}
// row of Khat^(R)_s in the B operand: far rows first (R = 2: s < 16; R = 3: s < 32), then
// the band (R = 0: s < 16 at 48; R = 1: s < 32 at 64; R = 2: s in [16, 48) at 96; R = 3:
// s in [32, 64) at 128)
__device__ __forceinline__ int brow(int R, int s) {
  if (R == 0) return 48 + s;
  if (R == 1) return 64 + s;
  if (R == 2) return s < 16 ? s : 80 + s;
  return s < 32 ? 16 + s : 96 + s;
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
// TMA tiles: byte offset of (row, channel) for element size E
template <int E>
__device__ __forceinline__ uint32_t swz(int row, int ch) {
  constexpr int PER = 128 / E;
  const uint32_t b = (uint32_t)((ch % PER) * E);
  return (uint32_t)(ch / PER) * 8192u + (uint32_t)row * 128u + ((((b >> 4) ^ (row & 7))) << 4) +
         (b & 15u);
}
// eight bf16 (channels 8c8..8c8+7) / four fp32 (channels 4c4..4c4+3) of one tile row
__device__ __forceinline__ void bf_row8(const uint8_t *tile, int row, int c8, float (&o)[8]) {
  const uint32_t off = (uint32_t)(c8 >> 3) * 8192u + (uint32_t)row * 128u +
                       ((uint32_t)((c8 & 7) ^ (row & 7)) << 4);
  const uint4 u = *reinterpret_cast<const uint4 *>(tile + off);
  o[0] = __uint_as_float(u.x << 16), o[1] = __uint_as_float(u.x & 0xffff0000u);
  o[2] = __uint_as_float(u.y << 16), o[3] = __uint_as_float(u.y & 0xffff0000u);
  o[4] = __uint_as_float(u.z << 16), o[5] = __uint_as_float(u.z & 0xffff0000u);
  o[6] = __uint_as_float(u.w << 16), o[7] = __uint_as_float(u.w & 0xffff0000u);
}
__device__ __forceinline__ void f_row8(const uint8_t *tile, int row, int c8, float (&o)[8]) {
  const float4 a = *reinterpret_cast<const float4 *>(
      tile + (uint32_t)(c8 >> 2) * 8192u + (uint32_t)row * 128u +
      ((uint32_t)(((2 * c8) & 7) ^ (row & 7)) << 4));
  const float4 b = *reinterpret_cast<const float4 *>(
      tile + (uint32_t)(c8 >> 2) * 8192u + (uint32_t)row * 128u +
      ((uint32_t)(((2 * c8 + 1) & 7) ^ (row & 7)) << 4));
  o[0] = a.x, o[1] = a.y, o[2] = a.z, o[3] = a.w, o[4] = b.x, o[5] = b.y, o[6] = b.z, o[7] = b.w;
}
// two fp32 -> packed bf16 pair (round to nearest even), low half = first
__device__ __forceinline__ uint32_t pack_bf2(float a, float b) {
  uint32_t d;  // one conversion for the pair: the first source lands in the upper half
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(b), "f"(a));
  return d;
}
__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }
// 2^x on the special-function unit (relative error ~2^-22)
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
// sigmoid(x) = 1 / (1 + 2^(-x log2 e)) with the special-function unit's 2^x and reciprocal:
// branch-free (relative error ~1e-7, far below the bf16 output's rounding)
__device__ __forceinline__ float sigmoid_sfu(float x) {
  float r;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(1.f + ex2(-1.4426950408889634f * x)));
  return r;
}

// D(16x16) += A(16 x 8kk) B(8kk x 16) for row-major fp32 blocks in shared memory (row
// strides la, lb), on the warp-level tensor-core MMA (m16n8k8, tf32 inputs, fp32
// accumulate).  Accumulator fragment: d[nt][0..3] = rows g, g, g+8, g+8 and columns
// 8nt + 2t, +1, 2t, +1 (g = lane / 4, t = lane % 4).
__device__ __forceinline__ void warp_mma16(float (&d)[2][4], const float *A, int la,
                                           const float *B, int lb, int ksteps, int lane) {
  const int g = lane >> 2, t = lane & 3;
  for (int kk = 0; kk < ksteps; ++kk) {
    const float *a = A + 8 * kk;
    const uint32_t a0 = __float_as_uint(to_tf32(a[g * la + t]));
    const uint32_t a1 = __float_as_uint(to_tf32(a[(g + 8) * la + t]));
    const uint32_t a2 = __float_as_uint(to_tf32(a[g * la + t + 4]));
    const uint32_t a3 = __float_as_uint(to_tf32(a[(g + 8) * la + t + 4]));
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      const float *b = B + (8 * kk) * lb + 8 * nt;
      const uint32_t b0 = __float_as_uint(to_tf32(b[t * lb + g]));
      const uint32_t b1 = __float_as_uint(to_tf32(b[(t + 4) * lb + g]));
      asm volatile(
          "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
          "{%8,%9}, {%0,%1,%2,%3};"
          : "+f"(d[nt][0]), "+f"(d[nt][1]), "+f"(d[nt][2]), "+f"(d[nt][3])
          : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
    }
  }
}
__device__ __forceinline__ void warp_store16(float *D, int ld, const float (&d)[2][4], int lane,
                                             float sign) {
  const int g = lane >> 2, t = lane & 3;
#pragma unroll
  for (int nt = 0; nt < 2; ++nt) {
    *reinterpret_cast<float2 *>(&D[g * ld + 8 * nt + 2 * t]) =
        make_float2(sign * d[nt][0], sign * d[nt][1]);
    *reinterpret_cast<float2 *>(&D[(g + 8) * ld + 8 * nt + 2 * t]) =
        make_float2(sign * d[nt][2], sign * d[nt][3]);
  }
}

struct Maps {
  CUtensorMap q, k, v, g, out, gate;
};

// 32 fp32 state values of one lane (key channels 32 g32 .. 32 g32 + 31) split into bf16 hi +
// lo, stored as packed pairs (low half = the even channel) in TA: hi at columns 16 g32 ..,
// lo 64 columns further (the A operand of the state read)
__device__ __forceinline__ void split_state_block(uint32_t t_lane, int g32, const float (&v)[32]) {
  float hw[16], lw[16];
#pragma unroll
  for (int y = 0; y < 16; ++y) {
    const uint32_t h = pack_bf2(v[2 * y], v[2 * y + 1]);
    hw[y] = __uint_as_float(h);
    lw[y] = __uint_as_float(pack_bf2(v[2 * y] - bf_lo(h), v[2 * y + 1] - bf_hi(h)));
  }
  tmem_st16(t_lane + TM_A + 16u * (uint32_t)g32, hw);
  tmem_st16(t_lane + TM_A + 64u + 16u * (uint32_t)g32, lw);
}

// Per-CTA shared state that P1 (out of line, below) shares with the kernel
__shared__ float s_beta[2][C], s_rq[C], s_rk[C], s_pd[2][C];  // beta, s_pd by chunk parity
__shared__ __align__(16) float s_g0[4][D];  // log2-retention just before each 16-block
__shared__ __align__(16) float s_gC[D];     // log2-retention at the chunk's last token
__shared__ float s_GC[D];                   // Gamma_C
__shared__ __align__(16) float s_M[3 * 256];  // inverse scratch; block decays P1 -> P2
__shared__ __align__(8) uint64_t s_bar[NBAR];
__shared__ uint32_t s_abort;

// ---- P1 of chunk cc, by a warp group (128 threads): beta; row norms and q.k (two threads
//      per row); per channel (one thread each) the prefix sums of the clamped
//      log2-retention, written back over g, with its value before each 16-token block,
//      at the chunk end and Gamma_C; and per channel the decay between block starts
//      2^(gam_R0 - gam_R'0) for the pairs (1,0) (2,1) (3,2) (2,0) (3,1) (3,0).
//      It runs before the walk for chunk 0 and during the output phase of chunk cc - 1
//      (t: the thread's index in the 128 running it).  part 1: beta and the row norms;
//      part 2: the prefix sums; part 3: both (two groups of 128 may split it).  beta is
//      stored last, so the global load's latency stalls nothing.  One out-of-line copy
//      serves every call site: the kernel is larger than the instruction cache, and code
//      size costs time.
__device__ __noinline__ void p1_run(const float *beta, int64_t bos, int64_t eos, int h, int H,
                                    bool l2norm, float l2_eps, float g_min, uint32_t pad,
                                    int cc, int t, int part) {
  uint8_t *sm = prefill_dyn_smem + pad;
  auto wait = [&](int b, uint32_t parity) {
    if (!mbar_wait(smem_u32(&s_bar[b]), parity)) s_abort = 1;
  };
  const int64_t tc = bos + (int64_t)cc * C;
  const int nvc = (int)((eos - tc) < C ? (eos - tc) : C);
  const uint32_t pc = (uint32_t)(cc & 1);
  float bv = 0.f;
  if ((part & 1) && t < nvc) bv = beta[(size_t)(tc + t) * H + h];
  wait(BAR_Q, pc);
  wait(BAR_K, pc);
  wait(BAR_G, pc);
  if (part & 1) {
    const int r = t >> 1, hf = t & 1;
    float sq = 0.f, sk = 0.f, sqk = 0.f;
    if (r < nvc) {
#pragma unroll 2
      for (int c8 = 0; c8 < 8; ++c8) {  // two at a time: p1 is inlined at three places
        float qv[8], kv[8];
        bf_row8(sm + OFF_Q, r, 8 * hf + c8, qv);
        bf_row8(sm + OFF_K, r, 8 * hf + c8, kv);
#pragma unroll
        for (int y = 0; y < 8; ++y)
          sq = fmaf(qv[y], qv[y], sq), sk = fmaf(kv[y], kv[y], sk), sqk = fmaf(qv[y], kv[y], sqk);
      }
    }
    sq += __shfl_xor_sync(0xffffffffu, sq, 1);
    sk += __shfl_xor_sync(0xffffffffu, sk, 1);
    sqk += __shfl_xor_sync(0xffffffffu, sqk, 1);
    if (hf == 0) {
      const float rq = r < nvc ? (l2norm ? rsqrtf(sq + l2_eps) : 1.f) : 0.f;
      const float rk = r < nvc ? (l2norm ? rsqrtf(sk + l2_eps) : 1.f) : 0.f;
      s_rq[r] = rq, s_rk[r] = rk, s_pd[pc][r] = sqk * rq * rk;
    }
    if (t < C) s_beta[pc][t] = bv;
  }
  if (part & 2) {
    const int i = t;
    // the swizzle repeats every 8 rows: row 8m + x of channel i sits at 1024 m + off[x]
    uint32_t off[8];
#pragma unroll
    for (int x = 0; x < 8; ++x) off[x] = OFF_G + swz<4>(x, i);
    float run = 0.f;
#pragma unroll 1
    for (int blk = 0; blk < 4; ++blk) {  // 16 rows at a time, running sum carried over
      s_g0[blk][i] = run;
#pragma unroll 1
      for (int x0 = 0; x0 < 16; x0 += 8) {  // 8 loads in flight, then the 8 sums
        const int r0 = 16 * blk + x0;
        uint8_t *rows = sm + (uint32_t)r0 * 128u;
        float v[8];
#pragma unroll
        for (int x = 0; x < 8; ++x)
          v[x] = fmaxf(*reinterpret_cast<const float *>(rows + off[x]), g_min);
        if (nvc == C) {  // a full chunk: every row counts
#pragma unroll
          for (int x = 0; x < 8; ++x) {
            run = fmaf(v[x], LOG2E, run);
            *reinterpret_cast<float *>(rows + off[x]) = run;
          }
        } else {
#pragma unroll
          for (int x = 0; x < 8; ++x) {
            if (r0 + x < nvc) run = fmaf(v[x], LOG2E, run);
            *reinterpret_cast<float *>(rows + off[x]) = run;
          }
        }
      }
    }
    float g0[4];
#pragma unroll
    for (int R = 0; R < 4; ++R) g0[R] = s_g0[R][i];
    s_gC[i] = run;
    s_GC[i] = ex2(run);
    s_M[0 * D + i] = ex2(g0[1] - g0[0]);
    s_M[1 * D + i] = ex2(g0[2] - g0[1]);
    s_M[2 * D + i] = ex2(g0[3] - g0[2]);
    s_M[3 * D + i] = ex2(g0[2] - g0[0]);
    s_M[4 * D + i] = ex2(g0[3] - g0[1]);
    s_M[5 * D + i] = ex2(g0[3] - g0[0]);
  }
}


// PAIR: a cluster of two CTAs per (head, sequence), rank 0 the consumer (state walk), rank 1
// the producer (A, P', T); otherwise one CTA does both.
template <typename ST, bool GATE, bool PAIR, bool QUANT>
__global__ void __launch_bounds__(NT, 1)
    prefill_tc_kernel(const TcArgs a, const __grid_constant__ Maps maps) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ float s_red[4][C];
  __shared__ float s_amx[4][C];  // FP8 output: each row's amax by TMEM lane quarter
  __shared__ float s_inv[C];     // FP8 output: each row's 448 / amax
  __shared__ float s_nrm[C];     // gated output: each row's 1 / RMS
  __shared__ uint32_t s_tmem, s_pend, s_ppar[NBAR];

  const uint32_t raw_u32 = smem_u32(smem_raw);
  const uint32_t pad = (1024u - (raw_u32 & 1023u)) & 1023u;
  uint8_t *sm = smem_raw + pad;
  const uint32_t sb = raw_u32 + pad;

  const int h = PAIR ? (int)(blockIdx.x >> 1) : (int)blockIdx.x, n = blockIdx.y;
  const bool producer = PAIR && cluster_rank() == 1;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int H = a.H;
  int64_t bos = a.cu_seqlens[n];
  int64_t eos = a.cu_seqlens[n + 1];
  if (bos < 0 || eos > a.total || eos < bos) {  // offsets outside the rows: flagged, empty
    if (threadIdx.x == 0 && a.err) atomicOr(a.err, ERR_BAD_SEQLEN);
    bos = eos = 0;
  }
  const int nchunks = (int)((eos - bos + C - 1) / C);
  const int quarter = warp & 3, grp = warp >> 2;   // TMEM lane quarter; warp group 0..2
  const int j = 32 * quarter + lane;               // this thread's TMEM lane
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
  if (PAIR) cluster_sync();  // both CTAs' barriers initialised before any remote arrive
  const uint32_t tm = s_tmem;

  // thread 0: TMA loads of chunk c into the buffers in `mask`
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
    if (mask & (1u << BAR_GT)) {  // gate logits [64 tokens][128] bf16, plain, into V's region
      mbar_expect_tx(bar(BAR_GT), 16384);
      tma_load_3d(sb + OFF_V, &maps.gate, 0, h, t0, bar(BAR_GT));
    }
    for (int b = 0; b < NBAR; ++b)
      if (mask & (1u << b)) s_ppar[b] = (uint32_t)(c & 1);
    atomicOr(&s_pend, mask);
  };
  auto commit_on = [&](int b, uint32_t parity) {
    mma_commit(bar(b));
    s_ppar[b] = parity;
    atomicOr(&s_pend, 1u << b);
  };
  auto commit = [&](uint32_t parity) { commit_on(BAR_MMA, parity); };
  // a bounded wait; one that runs out only raises the CTA's abort flag (reported once, at
  // exit): waits are inlined at every phase boundary, and the chunk loop's code size costs time
  auto wait = [&](int b, uint32_t parity) {
    if (!mbar_wait(bar(b), parity)) s_abort = 1;
  };
  auto sync = [&]() {
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    return s_abort == 0;
  };

  // ---- initial state: S^T[j][i] = S0[i][j] (warp groups 0 and 1: 64 key channels each)
  if (grp < 2 && !producer) {
    const ST *s0 = a.init_state
                       ? reinterpret_cast<const ST *>(a.init_state) + ((size_t)n * H + h) * D * D
                       : nullptr;
#pragma unroll 1
    for (int g32 = 0; g32 < 2; ++g32) {
      float v[32];
      const int i0 = 64 * grp + 32 * g32;
#pragma unroll
      for (int x = 0; x < 32; ++x) v[x] = s0 ? to_f(s0[(size_t)(i0 + x) * D + j]) : 0.f;
      tmem_st32(tm + lane_off + TM_S + i0, v);
      split_state_block(tm + lane_off, i0 >> 5, v);
    }
    tmem_wait_st();
  }
  if (tid == 0 && nchunks > 0)
    issue((1u << BAR_Q) | (1u << BAR_K) | (producer ? 0u : (1u << BAR_V)) | (1u << BAR_G), 0);
  bool ok = sync();

  auto p1 = [&](int cc, int t, int part) {
    p1_run(a.beta, bos, eos, h, H, a.qk_l2norm, a.l2_eps, a.g_min, pad, cc, t, part);
  };

  const uint32_t ID_64 = idesc(2, 128, 64, 0, 0);
  const uint32_t ID_X = idesc(1, 128, 128, 0, 0);
  const uint32_t ID_UPD = idesc(1, 128, 128, 0, 1);
  const uint32_t ID_AP160 = idesc(1, 128, 160, 0, 0);
  const uint32_t ID_AP112 = idesc(1, 128, 112, 0, 0);
  uint32_t mma_par = 0;
  int full_seen = 0;  // consumer thread 0: chunks whose T and P' it has waited for
  if (ok && nchunks > 0 && grp == 2) p1(0, tid - 256, 3);
  ok = sync();

  // ---- prefix-state checkpoints: after chunk c (cnt tokens of the sequence done), warp group
  //      2 writes S for every checkpoint placed there ("Ling-3.1-flash: What 63 Linear-
  //      Attention Layers Do to the KV Budget", section "Where the hybrid makes serving
  //      harder": a recurrent state can only be reused where a snapshot was saved).  A
  //      checkpoint passed over (not on a chunk edge or the sequence end) is flagged. ------
  int kc = a.ckpt_cu ? a.ckpt_cu[n] : 0;
  int kend = a.ckpt_cu ? a.ckpt_cu[n + 1] : 0;
  if (kc < 0 || kend > a.n_ckpt || kend < kc) {  // a range outside the checkpoints: flagged
    if (tid == 0 && a.err) atomicOr(a.err, ERR_BAD_INDEX);
    kc = kend = 0;
  }
  auto ckpt_write = [&](int64_t cnt) {
    for (; kc < kend && a.ckpt_pos[kc] <= cnt; ++kc) {
      if (a.ckpt_pos[kc] < cnt) {
        if (tid == 256 && a.err) atomicOr(a.err, ERR_BAD_INDEX);
        continue;
      }
      if (grp != 2) continue;
      ST *dst = reinterpret_cast<ST *>(a.ckpt_states) + ((size_t)kc * H + h) * D * D;
#pragma unroll 1
      for (int g32 = 0; g32 < 4; ++g32) {
        float v[32];
        tmem_ld32(tm + lane_off + TM_S + 32 * g32, v);
        tmem_wait_ld();
#pragma unroll
        for (int x = 0; x < 32; ++x) dst[(size_t)(32 * g32 + x) * D + j] = from_f<ST>(v[x]);
      }
    }
  };

  // ---- phases of one chunk (t0: first token, nv: valid tokens, par: chunk parity) -----
  auto ap_operands = [&](int nv, int nthr) {
    // ---- P2: operands of A and P, and X = [K Gamma; Q Gamma].  Rows relative to their own
    //      16-token block R = r/16 (gam_R0 = the log2-retention just before the block; q, k
    //      L2-normalised): Ktil_r = k_r 2^(gam_r - gam_R0), Qtil_r = q_r 2^(gam_r - gam_R0)
    //      (<= 1) form the tensor-memory A operand (lanes 0-63 and 64-127) as bf16 hi + lo;
    //      then the
    //      B operand, columns Khat^(R)_s = k_s 2^(gam_R0 - gam_s) for s <= 16R + 15, from
    //      Khat^(R(s))_s times the decay between block starts: bf16 hi for all 160 rows, lo
    //      for the 112 band rows.  All three warp groups share both. -----------------------
    {  // tensor-memory A operand and X: lane j's row, 16-channel pieces 3 grp .. (3, 3, 2)
      const int L = j, r = L & 63, R = r >> 4;
      const bool isq = L >= 64, live = r < nv;
      const uint8_t *src = sm + (isq ? OFF_Q : OFF_K);
      const float rn = isq ? s_rq[r] : s_rk[r];
      const int pbeg = nthr == NT ? 3 * grp : 4 * grp;
      const int pend = nthr == NT ? (grp == 2 ? 8 : 3 * grp + 3) : (tid < nthr ? 4 * grp + 4 : 0);
#pragma unroll 1
      for (int pc = pbeg; pc < pend; ++pc) {
        float hw[8], lw[8];  // packed bf16 pairs, low half = even channel
#pragma unroll
        for (int c2 = 0; c2 < 2; ++c2) {
          const int c8 = 2 * pc + c2, ch = 8 * c8;
          float x[8];
          if (live) {
            float vv[8], gg[8];
            bf_row8(src, r, c8, vv);
            f_row8(sm + OFF_G, r, c8, gg);
            const float4 r0 = *reinterpret_cast<const float4 *>(&s_g0[R][ch]);
            const float4 r1 = *reinterpret_cast<const float4 *>(&s_g0[R][ch + 4]);
            const float rr[8] = {r0.x, r0.y, r0.z, r0.w, r1.x, r1.y, r1.z, r1.w};
#pragma unroll
            for (int y = 0; y < 8; ++y) x[y] = vv[y] * rn * ex2(gg[y] - rr[y]);
          } else {
#pragma unroll
            for (int y = 0; y < 8; ++y) x[y] = 0.f;
          }
#pragma unroll
          for (int y = 0; y < 4; ++y) {
            const uint32_t hv = pack_bf2(x[2 * y], x[2 * y + 1]);
            hw[4 * c2 + y] = __uint_as_float(hv);
            lw[4 * c2 + y] =
                __uint_as_float(pack_bf2(x[2 * y] - bf_lo(hv), x[2 * y + 1] - bf_hi(hv)));
          }
        }
        tmem_st8(tm + lane_off + TM_AH + 8 * pc, hw);
        tmem_st8(tm + lane_off + TM_AL + 8 * pc, lw);
      }
      tmem_wait_st();
    }
    for (int it = tid; it < C * 16 && tid < nthr; it += nthr) {  // B: (token s, 8-channel group)
      const int sr = it >> 4, c8 = it & 15, Rs = sr >> 4;
      float kh[8];
      if (sr < nv) {
        float kv[8], gg[8];
        bf_row8(sm + OFF_K, sr, c8, kv);
        f_row8(sm + OFF_G, sr, c8, gg);
        const float4 r0 = *reinterpret_cast<const float4 *>(&s_g0[Rs][8 * c8]);
        const float4 r1 = *reinterpret_cast<const float4 *>(&s_g0[Rs][8 * c8 + 4]);
        const float rr[8] = {r0.x, r0.y, r0.z, r0.w, r1.x, r1.y, r1.z, r1.w};
        const float rk = s_rk[sr];
#pragma unroll
        for (int y = 0; y < 8; ++y) kh[y] = kv[y] * rk * ex2(rr[y] - gg[y]);
      } else {
#pragma unroll
        for (int y = 0; y < 8; ++y) kh[y] = 0.f;
      }
#pragma unroll
      for (int R = 0; R < 4; ++R) {
        if (R < Rs) continue;
        float val[8];
        if (R == Rs) {
#pragma unroll
          for (int y = 0; y < 8; ++y) val[y] = kh[y];
        } else {
          const int pr = R - Rs == 1 ? Rs : (R - Rs == 2 ? 3 + Rs : 5);
          const float4 d0 = *reinterpret_cast<const float4 *>(&s_M[pr * D + 8 * c8]);
          const float4 d1 = *reinterpret_cast<const float4 *>(&s_M[pr * D + 8 * c8 + 4]);
          val[0] = kh[0] * d0.x, val[1] = kh[1] * d0.y, val[2] = kh[2] * d0.z;
          val[3] = kh[3] * d0.w, val[4] = kh[4] * d1.x, val[5] = kh[5] * d1.y;
          val[6] = kh[6] * d1.z, val[7] = kh[7] * d1.w;
        }
        uint32_t hv[4], lv[4];
#pragma unroll
        for (int y = 0; y < 4; ++y) {
          hv[y] = pack_bf2(val[2 * y], val[2 * y + 1]);
          lv[y] = pack_bf2(val[2 * y] - bf_lo(hv[y]), val[2 * y + 1] - bf_hi(hv[y]));
        }
        const int n = brow(R, sr);
        *reinterpret_cast<uint4 *>(sm + OFF_BH + kmaj_bf16<160>(n, 8 * c8)) =
            make_uint4(hv[0], hv[1], hv[2], hv[3]);
        if (R - Rs <= 1)
          *reinterpret_cast<uint4 *>(sm + OFF_BL + kmaj_bf16<112>(n - 48, 8 * c8)) =
              make_uint4(lv[0], lv[1], lv[2], lv[3]);
      }
    }
  };
  // thread 0: D = [Ktil; Qtil] Khat^T: hi*hi over all 160 columns, hi*lo and lo*hi over
  // the band
  auto ap_issue = [&]() {
      for (int ks = 0; ks < 8; ++ks) {
        const uint32_t ko = (uint32_t)(ks >> 2) * (160 * 128) + (ks & 3) * 32;
        mma_bf16_ts(tm + TM_D, tm + TM_AH + 8 * ks, sdesc_sw128(sb + OFF_BH + ko, 16, 1024),
                    ID_AP160, ks > 0);
      }
      for (int ks = 0; ks < 8; ++ks) {
        const uint32_t ko = (uint32_t)(ks >> 2) * (112 * 128) + (ks & 3) * 32;
        mma_bf16_ts(tm + TM_D + 48, tm + TM_AH + 8 * ks, sdesc_sw128(sb + OFF_BL + ko, 16, 1024),
                    ID_AP112, 1);
      }
      for (int ks = 0; ks < 8; ++ks) {
        const uint32_t ko = (uint32_t)(ks >> 2) * (160 * 128) + 48 * 128 + (ks & 3) * 32;
        mma_bf16_ts(tm + TM_D + 48, tm + TM_AL + 8 * ks, sdesc_sw128(sb + OFF_BH + ko, 16, 1024),
                    ID_AP112, 1);
      }
      commit(mma_par);
  };
  // [K Gamma; Q Gamma] as bf16 hi | lo, K-major 128 rows (K rows 0-63, Q rows 64-127), at
  // X[0, 32K) | X[32K, 64K)
  auto x_rows = [&](int nv) {
    for (int it = tid; it < C * 16; it += NT) {  // (token, 8-channel group): rows r, 64 + r
      const int r = it >> 4, c8 = it & 15;
      uint32_t kh[4], kl[4], qh[4], ql[4];
      if (r < nv) {
        float kv[8], qv[8], gg[8];
        bf_row8(sm + OFF_K, r, c8, kv);
        bf_row8(sm + OFF_Q, r, c8, qv);
        f_row8(sm + OFF_G, r, c8, gg);
        const float rk = s_rk[r], rq = s_rq[r];
#pragma unroll
        for (int y = 0; y < 8; ++y) {
          const float G = ex2(gg[y]);
          kv[y] = kv[y] * rk * G;
          qv[y] = qv[y] * rq * G;
        }
#pragma unroll
        for (int y = 0; y < 4; ++y) {
          kh[y] = pack_bf2(kv[2 * y], kv[2 * y + 1]);
          kl[y] = pack_bf2(kv[2 * y] - bf_lo(kh[y]), kv[2 * y + 1] - bf_hi(kh[y]));
          qh[y] = pack_bf2(qv[2 * y], qv[2 * y + 1]);
          ql[y] = pack_bf2(qv[2 * y] - bf_lo(qh[y]), qv[2 * y + 1] - bf_hi(qh[y]));
        }
      } else {
#pragma unroll
        for (int y = 0; y < 4; ++y) kh[y] = kl[y] = qh[y] = ql[y] = 0u;
      }
      const uint32_t ko = kmaj_bf16<128>(r, 8 * c8), qo = kmaj_bf16<128>(64 + r, 8 * c8);
      *reinterpret_cast<uint4 *>(sm + OFF_X + ko) = make_uint4(kh[0], kh[1], kh[2], kh[3]);
      *reinterpret_cast<uint4 *>(sm + OFF_X + 32768 + ko) = make_uint4(kl[0], kl[1], kl[2], kl[3]);
      *reinterpret_cast<uint4 *>(sm + OFF_X + qo) = make_uint4(qh[0], qh[1], qh[2], qh[3]);
      *reinterpret_cast<uint4 *>(sm + OFF_X + 32768 + qo) = make_uint4(ql[0], ql[1], ql[2], ql[3]);
    }
  };
  // P' rows go to pbase (this CTA's shared memory) or, with rbase != 0, into the consumer's
  // shared memory at shared::cluster address rbase by asynchronous stores completing on the
  // consumer's barrier rbar
  auto extract = [&](int nv, uint8_t *pbase, uint32_t rbase, uint32_t rbar, float *Am,
                     uint32_t par) {
    auto put_p = [&](uint32_t off, float4 val) {
      if (rbase) st_async_v4(rbase + off, val, rbar);
      else *reinterpret_cast<float4 *>(pbase + off) = val;
    };
    // ---- P3: A (beta-scaled, strict lower, fp32 rows of LDA) and P' (strict lower, tf32,
    //      K-major) from the product, one tensor-memory lane per row (lanes 0-63: A, 64-127:
    //      P), in 16-column pieces that each hold one block R and 16 consecutive s; zeros in
    //      the blocks of P' above the diagonal. ----------------------------------------------
    {
      const int L = j, r = L & 63, R = r >> 4;
      const bool isp = L >= 64;
      // pieces of this warp: rows 0-31 (R = 0, 1): piece 3 + grp; rows 32-63 (R = 2, 3):
      // group 2 pieces 0-2 (it inverts next, after every piece is in), group 0 pieces 6-7,
      // group 1 pieces 8-9
      const bool lo_rows = (quarter & 1) == 0;
      const int p0 = lo_rows ? 3 + grp : (grp == 2 ? 0 : 6 + 2 * grp);
      const int np = lo_rows ? 1 : (grp == 2 ? 3 : 2);
      const float br = s_beta[par][r];
      for (int pc = p0; pc < p0 + np; ++pc) {
        float v[16];
        tmem_ld16(tm + lane_off + TM_D + 16 * pc, v);
        tmem_wait_ld();
        // piece -> (block, first s)
        const int Rn = pc == 0 ? 2 : pc <= 2 ? 3 : pc == 3 ? 0 : pc <= 5 ? 1 : pc <= 7 ? 2 : 3;
        const int s0 = pc == 0 ? 0 : pc == 1 ? 0 : pc == 2 ? 16 : pc == 3 ? 0 : pc == 4 ? 0
                     : pc == 5 ? 16 : pc == 6 ? 16 : pc == 7 ? 32 : pc == 8 ? 32 : 48;
        if (Rn != R) continue;
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          const int s = s0 + 4 * q4;
          if (!isp) {
            *reinterpret_cast<float4 *>(&Am[r * LDA + s]) =
                make_float4(s < r ? br * v[4 * q4] : 0.f, s + 1 < r ? br * v[4 * q4 + 1] : 0.f,
                            s + 2 < r ? br * v[4 * q4 + 2] : 0.f,
                            s + 3 < r ? br * v[4 * q4 + 3] : 0.f);
          } else {
            put_p(kmaj_f32<64>(r, s),
                  make_float4(s < r ? to_tf32(v[4 * q4]) : 0.f,
                              s + 1 < r ? to_tf32(v[4 * q4 + 1]) : 0.f,
                              s + 2 < r ? to_tf32(v[4 * q4 + 2]) : 0.f,
                              s + 3 < r ? to_tf32(v[4 * q4 + 3]) : 0.f));
          }
        }
      }
      {  // P' blocks (R, R') with R' > R: pairs (0,1) (0,2) (0,3) (1,2) (1,3) (2,3)
        const int pr = tid >> 6, rr16 = (tid >> 2) & 15, c4 = tid & 3;
        const int Rz = pr < 3 ? 0 : pr < 5 ? 1 : 2;
        const int Rpz = pr < 3 ? pr + 1 : pr < 5 ? pr - 1 : 3;
        put_p(kmaj_f32<64>(16 * Rz + rr16, 16 * Rpz + 4 * c4), make_float4(0.f, 0.f, 0.f, 0.f));
      }
    }
  };
  // ---- MMA1: X^T = S^T [K Gamma; Q Gamma]^T -> TC (N = 128: key rows in TC[0, 64), query
  //      rows in TC[64, 128)) as bf16 hi*hi + hi*lo + lo*hi with the split state from TA.
  //      One CTA: issued by thread 0, committed on BAR_MMA; cluster-pair consumer: issued by
  //      thread 256 and committed on BAR_X (phase = chunk parity), since a commit tracks only
  //      the products of the thread that issues it
  auto mma1_issue = [&](bool own_bar, uint32_t par) {
      for (int term = 0; term < 3; ++term) {
        const uint32_t a_col = TM_A + (term == 2 ? 64 : 0);              // S hi | S lo
        const uint32_t b_off = OFF_X + (term == 1 ? 32768 : 0);          // hi | lo rows
        for (int ks = 0; ks < 8; ++ks) {
          const uint64_t bd = sdesc_sw128(sb + b_off + (ks >> 2) * 16384 + (ks & 3) * 32, 16, 1024);
          mma_bf16_ts(tm + TM_C, tm + a_col + 8 * ks, bd, ID_X, term > 0 || ks > 0);
        }
      }
      if (own_bar) commit_on(BAR_X, par);
      else commit(mma_par);
  };
  // the state split into bf16 hi | lo (packed pairs) in TA, 32-column blocks first ..
  // first+n-1 of this thread's lane quarter (the state's final value for the next MMA1)
  auto s_split = [&](int first, int nblk) {
#pragma unroll 1
      for (int g32 = first; g32 < first + nblk; ++g32) {
        float v[32];
        tmem_ld32(tm + lane_off + TM_S + 32 * g32, v);
        tmem_wait_ld();
        split_state_block(tm + lane_off, g32, v);
      }
      tmem_wait_st();
  };
  // ---- T = (I + A)^-1 by 16x16 blocks on warp group 2, fp32, then tf32 K-major [r][s]
  //      at tbase
  auto inverse = [&](uint8_t *tbase, const float *Am, float *Tm, float *scr) {
      const int t = tid - 256, wg = t >> 5;
      if (t < 64) {  // diagonal blocks: right-looking substitution, one column per thread
        const int R = t >> 4, cc = t & 15, b0 = 16 * R;
        float x[16], pacc[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) pacc[i] = 0.f;
#pragma unroll
        for (int k = 0; k < 16; ++k) {
          x[k] = k < cc ? 0.f : (k == cc ? 1.f : -pacc[k]);
#pragma unroll
          for (int i = k + 1; i < 16; ++i) pacc[i] = fmaf(Am[(b0 + i) * LDA + b0 + k], x[k], pacc[i]);
        }
#pragma unroll
        for (int i = 0; i < 16; ++i) Tm[(b0 + i) * 64 + b0 + cc] = x[i];
      }
      asm volatile("bar.sync 3, 128;" ::: "memory");
      if (PAIR) {  // the producer of a pair: by distance (beside its P1 and operand build, the
                   // fewer warps of the last levels measured faster)
        // off-diagonal blocks by distance, one warp per block: M = sum_Q A_RQ T_QS (the A
        // blocks of row R are contiguous in Q), then T_RS = -T_RR M
        for (int dist = 1; dist <= 3; ++dist) {
          if (wg < 4 - dist) {
            const int R = dist + wg, S = R - dist;
            float dacc[2][4] = {};
            for (int Q = S; Q < R; ++Q)
              warp_mma16(dacc, Am + (16 * R) * LDA + 16 * Q, LDA, Tm + (16 * Q) * 64 + 16 * S, 64,
                         2, lane);
            warp_store16(scr + wg * 256, 16, dacc, lane, 1.f);
            __syncwarp();
            float tacc[2][4] = {};
            warp_mma16(tacc, Tm + (16 * R) * 64 + 16 * R, 64, scr + wg * 256, 16, 2, lane);
            warp_store16(Tm + (16 * R) * 64 + 16 * S, 64, tacc, lane, -1.f);
          }
          asm volatile("bar.sync 3, 128;" ::: "memory");
        }
      } else {
        // off-diagonal blocks as a 2 x 2 block inverse of 32 x 32 halves, whose diagonal halves
        // are themselves 2 x 2 block inverses: three levels of at most two 16 x 16 products
        // each (against three by distance, the last of four on one warp).
        // level 1 (warps 0, 1): T_10 = -T_11 (A_10 T_00), T_32 = -T_33 (A_32 T_22)
        if (wg < 2) {
          const int R = 1 + 2 * wg, S = R - 1;
          float dacc[2][4] = {};
          warp_mma16(dacc, Am + (16 * R) * LDA + 16 * S, LDA, Tm + (16 * S) * 64 + 16 * S, 64, 2,
                     lane);
          warp_store16(scr + wg * 256, 16, dacc, lane, 1.f);
          __syncwarp();
          float tacc[2][4] = {};
          warp_mma16(tacc, Tm + (16 * R) * 64 + 16 * R, 64, scr + wg * 256, 16, 2, lane);
          warp_store16(Tm + (16 * R) * 64 + 16 * S, 64, tacc, lane, -1.f);
        }
        asm volatile("bar.sync 3, 128;" ::: "memory");
        // level 2 (warp wg: R = 2 + wg / 2, S = wg % 2): X_RS = sum_{Q = S..1} A_RQ T_QS, the
        // lower-left half's product with the inverse of the upper-left one, into scratch block wg
        {
          const int R = 2 + (wg >> 1), S = wg & 1;
          float dacc[2][4] = {};
          for (int Q = S; Q < 2; ++Q)
            warp_mma16(dacc, Am + (16 * R) * LDA + 16 * Q, LDA, Tm + (16 * Q) * 64 + 16 * S, 64,
                       2, lane);
          warp_store16(scr + wg * 256, 16, dacc, lane, 1.f);
        }
        asm volatile("bar.sync 3, 128;" ::: "memory");
        // level 3: T_RS = -sum_{Q = 2..R} T_RQ X_QS (the inverse of the lower-right half times X)
        {
          const int R = 2 + (wg >> 1), S = wg & 1;
          float tacc[2][4] = {};
          for (int Q = 2; Q <= R; ++Q)
            warp_mma16(tacc, Tm + (16 * R) * 64 + 16 * Q, 64, scr + (2 * (Q - 2) + S) * 256, 16, 2,
                       lane);
          warp_store16(Tm + (16 * R) * 64 + 16 * S, 64, tacc, lane, -1.f);
        }
        asm volatile("bar.sync 3, 128;" ::: "memory");
      }
      // T (lower triangle incl. the unit diagonal) -> tf32, K-major [r][s], in place, four
      // consecutive s at a time (16-byte loads and stores: the swizzle moves whole 16-byte
      // chunks)
      float4 tv[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const int e = 4 * (t + 128 * q), r = e >> 6, s0 = e & 63;
        const float4 v = *reinterpret_cast<const float4 *>(Tm + e);
        tv[q] = make_float4(s0 <= r ? to_tf32(v.x) : 0.f, s0 + 1 <= r ? to_tf32(v.y) : 0.f,
                            s0 + 2 <= r ? to_tf32(v.z) : 0.f, s0 + 3 <= r ? to_tf32(v.w) : 0.f);
      }
      asm volatile("bar.sync 3, 128;" ::: "memory");
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const int e = 4 * (t + 128 * q);
        *reinterpret_cast<float4 *>(tbase + kmaj_f32<64>(e >> 6, e & 63)) = tv[q];
      }
  };
  // ---- S^T *= Gamma_C on 32-column blocks first .. first + nblk - 1 of this warp's lane
  //      quarter (the cluster-pair consumer hands the whole decay to warp group 2, which is
  //      free while groups 0 and 1 form Y)
  auto decay = [&](int first, int nblk) {
#pragma unroll 1
      for (int g32 = first; g32 < first + nblk; ++g32) {
        float v[32];
        const int i0 = 32 * g32;
        tmem_ld32(tm + lane_off + TM_S + i0, v);
        tmem_wait_ld();
#pragma unroll
        for (int x = 0; x < 32; ++x) v[x] *= s_GC[i0 + x];
        tmem_st32(tm + lane_off + TM_S + i0, v);
      }
      tmem_wait_st();
  };
  // ---- groups 0 and 1: (one CTA) decay this group's 64 key channels of S^T while MMA1
  //      runs, since MMA1 reads the split state in TA, not S; then wait for MMA1 and form
  //      Y^T = beta (V - K Gamma S)^T (tf32 hi + lo in TB)
  auto y_decay = [&](int nv, uint32_t par, bool with_decay, bool own_bars) {
      if (with_decay) decay(2 * grp, 2);
      if (own_bars) wait(BAR_X, par);  // MMA1 done
      else wait(BAR_MMA, mma_par);
      tc_fence_after();
      wait(BAR_V, par);
      {
        float xk[32], hi[32];
        tmem_ld32(tm + lane_off + TM_C + 32 * grp, xk);
        // v[s][j] of rows s = 32 grp + x: the tile's 128-byte swizzle depends on x mod 8 only,
        // so eight base addresses serve all 32 rows (row x at + 128 x)
        const uint8_t *vb = sm + OFF_V + (j >> 6) * 8192 + ((2 * j) & 15) + 32 * grp * 128;
        const int jc = (j & 63) >> 3;
        const uint8_t *vp[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) vp[k] = vb + ((jc ^ k) << 4);
        tmem_wait_ld();
#pragma unroll
        for (int x = 0; x < 32; ++x) {
          const int s = 32 * grp + x;
          const float vv = __bfloat162float(*reinterpret_cast<const bf16 *>(vp[x & 7] + 128 * x));
          const float y = s < nv ? s_beta[par][s] * (vv - xk[x]) : 0.f;
          hi[x] = to_tf32(y);
          xk[x] = to_tf32(y - hi[x]);
        }
        tmem_st32(tm + lane_off + TM_B + 32 * grp, hi);
        tmem_st32(tm + lane_off + TM_B + 64 + 32 * grp, xk);
      }
      tmem_wait_st();
  };
  // thread 0: u^T = Y^T T^T, hi then lo (T at shared offset t_off), into TC[0, 64) (X_k has
  // been read by the Y pass)
  auto mmau_issue = [&](uint32_t t_off) {
      for (int ks = 0; ks < 16; ++ks) {
        const int k8 = ks & 7;
        const uint64_t bd = sdesc_sw128(sb + t_off + (k8 >> 2) * 8192 + (k8 & 3) * 32, 16, 1024);
        mma_tf32_ts(tm + TM_C, tm + TM_B + 64 * (ks >> 3) + 8 * k8, bd, ID_64, ks > 0);
      }
      commit(mma_par);
  };
  // Kbar = k Gamma_C / Gamma (bf16 hi | lo, MN-major) into X[0, 32K), items [i0, i1) of the
  // (token, 8-channel group) list by thread t of nt; once all of it is built, k and g of the
  // next chunk may be loaded
  auto kbar_items = [&](int nv, int i0, int i1, int t, int nt) {
    for (int it = i0 + t; it < i1; it += nt) {  // Kbar hi | lo
      const int s = it >> 4, c8 = it & 15;
      uint32_t hw[4], lw[4];
      if (s < nv) {
        float kv[8], gg[8];
        bf_row8(sm + OFF_K, s, c8, kv);
        f_row8(sm + OFF_G, s, c8, gg);
        const float4 c0v = *reinterpret_cast<const float4 *>(&s_gC[8 * c8]);
        const float4 c1v = *reinterpret_cast<const float4 *>(&s_gC[8 * c8 + 4]);
        const float gc[8] = {c0v.x, c0v.y, c0v.z, c0v.w, c1v.x, c1v.y, c1v.z, c1v.w};
        const float rk = s_rk[s];
#pragma unroll
        for (int y = 0; y < 4; ++y) {
          const float a0 = kv[2 * y] * rk * ex2(gc[2 * y] - gg[2 * y]);
          const float a1 = kv[2 * y + 1] * rk * ex2(gc[2 * y + 1] - gg[2 * y + 1]);
          hw[y] = pack_bf2(a0, a1);
          lw[y] = pack_bf2(a0 - bf_lo(hw[y]), a1 - bf_hi(hw[y]));
        }
      } else {
#pragma unroll
        for (int y = 0; y < 4; ++y) hw[y] = lw[y] = 0u;
      }
      const uint32_t off = mnmaj_bf16_128(s, 8 * c8);
      *reinterpret_cast<uint4 *>(sm + OFF_X + off) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
      *reinterpret_cast<uint4 *>(sm + OFF_X + 16384 + off) =
          make_uint4(lw[0], lw[1], lw[2], lw[3]);
    }
  };
  // cluster-pair consumer: warp group 2 builds the first KB2 items once the state read is done
  // (it frees X), in the Y phase it would otherwise idle through; the rest while u is formed
  constexpr int KB2 = 256;
  auto p6 = [&]() {
    // ---- P6: u from TC[0, 64) (fp32 -> TB[0,64) for the output, tf32 -> TB[64,128) for
    //      P'u) and u hi | lo (bf16, K-major [j][s]) into X[32K, 64K) -----------------------
    if (grp < 2) {
      float u[32], t[32];
      tmem_ld32(tm + lane_off + TM_C + 32 * grp, u);
      tmem_wait_ld();
      tmem_st32(tm + lane_off + TM_B + 32 * grp, u);
#pragma unroll
      for (int x = 0; x < 32; ++x) t[x] = to_tf32(u[x]);
      tmem_st32(tm + lane_off + TM_B + 64 + 32 * grp, t);
#pragma unroll
      for (int c8 = 0; c8 < 4; ++c8) {
        uint32_t hw[4], lw[4];
#pragma unroll
        for (int y = 0; y < 4; ++y) {
          const float a0 = u[8 * c8 + 2 * y], a1 = u[8 * c8 + 2 * y + 1];
          hw[y] = pack_bf2(a0, a1);
          lw[y] = pack_bf2(a0 - bf_lo(hw[y]), a1 - bf_hi(hw[y]));
        }
        const uint32_t off = kmaj_bf16_64(j, 32 * grp + 8 * c8);
        *reinterpret_cast<uint4 *>(sm + OFF_X + 32768 + off) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
        *reinterpret_cast<uint4 *>(sm + OFF_X + 49152 + off) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
      }
      tmem_wait_st();
    }
  };
  auto p6_spread = [&]() {
    // ---- the same in 8-column slices spread over the three warp groups (3, 3, 2): the
    //      one-CTA form, whose group 2 is otherwise idle here (the pair's group 2 gains
    //      nothing from it: it is the next chunk's P1 that waits) ----------------------------
    float u[3][8];
#pragma unroll
    for (int q = 0; q < 3; ++q)
      if (grp + 3 * q < 8) tmem_ld8(tm + lane_off + TM_C + 8 * (grp + 3 * q), u[q]);
    tmem_wait_ld();
#pragma unroll
    for (int q = 0; q < 3; ++q) {
      const int s8 = grp + 3 * q;
      if (s8 < 8) {
        float t[8];
        tmem_st8(tm + lane_off + TM_B + 8 * s8, u[q]);
#pragma unroll
        for (int x = 0; x < 8; ++x) t[x] = to_tf32(u[q][x]);
        tmem_st8(tm + lane_off + TM_B + 64 + 8 * s8, t);
        uint32_t hw[4], lw[4];
#pragma unroll
        for (int y = 0; y < 4; ++y) {
          const float a0 = u[q][2 * y], a1 = u[q][2 * y + 1];
          hw[y] = pack_bf2(a0, a1);
          lw[y] = pack_bf2(a0 - bf_lo(hw[y]), a1 - bf_hi(hw[y]));
        }
        const uint32_t off = kmaj_bf16_64(j, 8 * s8);
        *reinterpret_cast<uint4 *>(sm + OFF_X + 32768 + off) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
        *reinterpret_cast<uint4 *>(sm + OFF_X + 49152 + off) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
      }
    }
    tmem_wait_st();
  };
  // ---- P7 (thread 0): O += P' u (tf32, P' at shared offset p_off); S^T += u^T Kbar as
  //      hi*hi + hi*lo + lo*hi (bf16)
  auto p7_issue = [&](uint32_t p_off) {
      for (int ks = 0; ks < 8; ++ks) {
        const uint64_t bd = sdesc_sw128(sb + p_off + (ks >> 2) * 8192 + (ks & 3) * 32, 16, 1024);
        mma_tf32_ts(tm + TM_C + 64, tm + TM_B + 64 + 8 * ks, bd, ID_64, 1);
      }
      for (int term = 0; term < 3; ++term) {
        const uint32_t a_off = OFF_X + (term == 2 ? 49152 : 32768);
        const uint32_t b_off = OFF_X + (term == 1 ? 16384 : 0);
        for (int ks = 0; ks < 4; ++ks) {
          const uint64_t ad = sdesc_sw128(sb + a_off + ks * 32, 16, 1024);
          const uint64_t bd = sdesc_sw128(sb + b_off + ks * 4096, 1024, 2048);
          mma_bf16_ss(tm + TM_S, ad, bd, ID_UPD, 1);
        }
      }
      commit(mma_par);
  };
  auto p8 = [&](int nv, int64_t t0, uint32_t par) {
    // ---- P8: outputs o_r = scale (O'_r + (q_r.k_r) u_r), norm and gate, store.  A full
    //      chunk goes out as one bulk tensor store of the [64 tokens][128] bf16 tile, staged
    //      in the V region (free since the Y pass; the next V load waits for the store to
    //      have read it); a partial last chunk, whose box would run into the next sequence,
    //      is stored element by element.  Meanwhile warp group 2 runs P1 of the next chunk. ----
    if (grp < 2) {
      const bool tile = nv == C;
      bf16 *stage = reinterpret_cast<bf16 *>(sm + OFF_V);  // V was consumed by the Y pass
      bf16 *out = reinterpret_cast<bf16 *>(a.out);
      // Per-row statistics (sum of squares for the norm, amax for FP8) need all 128 values of
      // a row: this thread holds its channel's 32 rows at once and a transpose-reduce over the
      // warp leaves row 32 grp + lane in each lane (31 shuffles for 32 rows); the four lane
      // quarters meet in shared memory, and one lane per row turns them into factors.  Values
      // are then written 8 rows at a time, o re-read from tensor memory, so the unrolled code
      // stays short: the whole kernel is larger than the instruction cache, and unrolled
      // length costs time (measured).
      auto transpose_reduce = [&](float (&v)[32], bool is_max) {
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) {
          const bool up = (lane & off) != 0;
#pragma unroll
          for (int x = 0; x < off; ++x) {
            const float send = up ? v[x] : v[x + off];
            const float recv = __shfl_xor_sync(0xffffffffu, send, off);
            const float keep = up ? v[x + off] : v[x];
            v[x] = is_max ? fmaxf(keep, recv) : keep + recv;
          }
        }
      };
      auto load_o = [&](float (&o)[32]) {  // o of rows 32 grp + x, this thread's channel
        float u[32];
        tmem_ld32(tm + lane_off + TM_C + 64 + 32 * grp, o);
        tmem_ld32(tm + lane_off + TM_B + 32 * grp, u);
        tmem_wait_ld();
#pragma unroll
        for (int x = 0; x < 32; ++x) o[x] = a.scale * fmaf(s_pd[par][32 * grp + x], u[x], o[x]);
      };
      auto o_slice = [&](int sl, float (&v)[8]) {  // o of rows 32 grp + 8 sl + y, this channel
        float u8[8];
        tmem_ld8(tm + lane_off + TM_C + 64 + 32 * grp + 8 * sl, v);
        tmem_ld8(tm + lane_off + TM_B + 32 * grp + 8 * sl, u8);
        tmem_wait_ld();
#pragma unroll
        for (int y = 0; y < 8; ++y) v[y] = a.scale * fmaf(s_pd[par][32 * grp + 8 * sl + y], u8[y], v[y]);
      };
      const float w = GATE ? (a.norm_w ? a.norm_w[j] : 1.f) : 1.f;
      float ov[32];  // o of this thread's 32 rows: one tensor-memory round trip
      if (GATE && !QUANT) load_o(ov);
      if (GATE) {
        wait(BAR_GT, par);  // the gate tile, loaded into the stage region after the Y pass
        {
          float sq[32];
          if (QUANT) load_o(sq);
#pragma unroll
          for (int x = 0; x < 32; ++x) sq[x] = QUANT ? sq[x] * sq[x] : ov[x] * ov[x];
          transpose_reduce(sq, false);
          s_red[quarter][32 * grp + lane] = sq[0];
        }
        asm volatile("bar.sync 1, 256;" ::: "memory");
        if (quarter == 0) {  // the row's norm factor
          const int r = 32 * grp + lane;
          s_nrm[r] = rsqrtf((s_red[0][r] + s_red[1][r] + s_red[2][r] + s_red[3][r]) * (1.f / D) +
                            a.norm_eps);
        }
        asm volatile("bar.sync 1, 256;" ::: "memory");
      }
      if (QUANT) {
        // FP8 output (E4M3 codes, one fp32 scale per token): each row's amax of its final
        // values, then one lane per row computes the scale (to HBM) and 448 / amax (to all)
        auto row_factors = [&]() {
          asm volatile("bar.sync 1, 256;" ::: "memory");
          if (quarter == 0) {
            const int r = 32 * grp + lane;
            const float amax =
                fmaxf(fmaxf(s_amx[0][r], s_amx[1][r]), fmaxf(s_amx[2][r], s_amx[3][r]));
            s_inv[r] = fp8_inv_scale(amax);
            if (r < nv) a.out_scale[(size_t)(t0 + r) * H + h] = fp8_scale(amax);
          }
          asm volatile("bar.sync 1, 256;" ::: "memory");
        };
        uint8_t *stage8 = sm + OFF_V;
        if (!GATE) {
          {
            float mx[32];
            load_o(mx);
#pragma unroll
            for (int x = 0; x < 32; ++x) mx[x] = 32 * grp + x < nv ? fabsf(mx[x]) : 0.f;
            transpose_reduce(mx, true);
            s_amx[quarter][32 * grp + lane] = mx[0];
          }
          row_factors();
#pragma unroll 1
          for (int sl = 0; sl < 4; ++sl) {  // codes, 8 rows at a time
            float v[8];
            o_slice(sl, v);
#pragma unroll
            for (int y = 0; y < 8; ++y) {
              const int r = 32 * grp + 8 * sl + y;
              const uint8_t code = fp8_code(v[y], s_inv[r]);
              if (tile) stage8[r * D + j] = code;
              else if (r < nv) a.out_q[((size_t)(t0 + r) * H + h) * D + j] = code;
            }
          }
        } else {
          // the codes overwrite gate logits of other rows (one byte per value in the same
          // region), so every logit is read first: the 32 gated values stay in registers
          float o[32];
#pragma unroll
          for (int sl = 0; sl < 4; ++sl) {
            float v[8];
            o_slice(sl, v);
#pragma unroll
            for (int y = 0; y < 8; ++y) {
              const int r = 32 * grp + 8 * sl + y;
              o[8 * sl + y] = v[y] * s_nrm[r] * w * sigmoid_sfu(__bfloat162float(stage[r * D + j]));
            }
          }
          {
            float mx[32];
#pragma unroll
            for (int x = 0; x < 32; ++x) mx[x] = 32 * grp + x < nv ? fabsf(o[x]) : 0.f;
            transpose_reduce(mx, true);
            s_amx[quarter][32 * grp + lane] = mx[0];
          }
          row_factors();  // its first barrier: every gate logit has been read
#pragma unroll
          for (int x = 0; x < 32; ++x) {
            const int r = 32 * grp + x;
            const uint8_t code = fp8_code(o[x], s_inv[r]);
            if (tile) stage8[r * D + j] = code;
            else if (r < nv) a.out_q[((size_t)(t0 + r) * H + h) * D + j] = code;
          }
        }
      } else if (GATE) {
        // sigma(gate) of the 32 rows first (every logit read before the outputs overwrite the
        // stage region), then the outputs two rows per packed conversion from o in registers
        float sg[32];
#pragma unroll
        for (int x = 0; x < 32; ++x) sg[x] = sigmoid_sfu(__bfloat162float(stage[(32 * grp + x) * D + j]));
#pragma unroll
        for (int x = 0; x < 32; x += 2) {
          const int r = 32 * grp + x;
          const uint32_t pr = pack_bf2(ov[x] * s_nrm[r] * w * sg[x], ov[x + 1] * s_nrm[r + 1] * w * sg[x + 1]);
          const uint16_t v0 = (uint16_t)(pr & 0xffffu), v1 = (uint16_t)(pr >> 16);
          if (tile) {
            reinterpret_cast<uint16_t *>(stage)[r * D + j] = v0;
            reinterpret_cast<uint16_t *>(stage)[(r + 1) * D + j] = v1;
          } else {
            uint16_t *o16 = reinterpret_cast<uint16_t *>(out);
            if (r < nv) o16[((size_t)(t0 + r) * H + h) * D + j] = v0;
            if (r + 1 < nv) o16[((size_t)(t0 + r + 1) * H + h) * D + j] = v1;
          }
        }
      } else {
#pragma unroll 1
        for (int sl = 0; sl < 4; ++sl) {  // 8 rows at a time: a short loop body
          float o8[8], u8[8];
          tmem_ld8(tm + lane_off + TM_C + 64 + 32 * grp + 8 * sl, o8);
          tmem_ld8(tm + lane_off + TM_B + 32 * grp + 8 * sl, u8);
          tmem_wait_ld();
#pragma unroll
          for (int y = 0; y < 8; y += 2) {  // two rows per packed conversion
            const int r = 32 * grp + 8 * sl + y;
            const uint32_t pr = pack_bf2(a.scale * fmaf(s_pd[par][r], u8[y], o8[y]),
                                         a.scale * fmaf(s_pd[par][r + 1], u8[y + 1], o8[y + 1]));
            const uint16_t v0 = (uint16_t)(pr & 0xffffu), v1 = (uint16_t)(pr >> 16);
            if (tile) {
              reinterpret_cast<uint16_t *>(stage)[r * D + j] = v0;
              reinterpret_cast<uint16_t *>(stage)[(r + 1) * D + j] = v1;
            } else {
              uint16_t *o16 = reinterpret_cast<uint16_t *>(out);
              if (r < nv) o16[((size_t)(t0 + r) * H + h) * D + j] = v0;
              if (r + 1 < nv) o16[((size_t)(t0 + r + 1) * H + h) * D + j] = v1;
            }
          }
        }
      }
      if (tile) {
        fence_proxy_async();
        asm volatile("bar.sync 1, 256;" ::: "memory");
        if (tid == 0) {
          tma_store_3d(&maps.out, 0, h, (int)t0, sb + OFF_V);
          bulk_commit();
        }
      }
    }
  };

  if (!PAIR) {
    for (int c = 0; c < nchunks && ok; ++c) {
      const int64_t t0 = bos + (int64_t)c * C;
      const int nv = (int)((eos - t0) < C ? (eos - t0) : C);
      const uint32_t par = (uint32_t)(c & 1);
      const bool more = c + 1 < nchunks;
      ap_operands(nv, NT);
      fence_proxy_async();
      if (!(ok = sync())) break;
      if (tid == 0) {
        if (c > 0) {  // V is free once the previous output tile has been read out of it
          bulk_wait_read0();
          issue(1u << BAR_V, c);
        }
        ap_issue();
      }
      x_rows(nv);  // while the product runs
      wait(BAR_MMA, mma_par);
      mma_par ^= 1;
      tc_fence_after();
      extract(nv, sm + OFF_P, 0u, 0u, reinterpret_cast<float *>(sm + OFF_A), par);
      if (grp < 2) s_split(2 * grp, 2);  // TA is free once the A/P product is done
      fence_proxy_async();
      if (!(ok = sync())) break;
      if (tid == 0) {
        if (more) issue(1u << BAR_Q, c + 1);  // q is consumed
        mma1_issue(false, 0);
      }
      if (grp == 2) {  // in flight with MMA1 and the Y / decay work
        inverse(sm + OFF_T, reinterpret_cast<const float *>(sm + OFF_A),
                reinterpret_cast<float *>(sm + OFF_T), reinterpret_cast<float *>(sm + OFF_SCR));
      } else {  // then Kbar (X is free once MMA1 is done) while group 2 still inverts
        y_decay(nv, par, true, false);
        kbar_items(nv, 0, C * 16, tid, 256);
      }
      mma_par ^= 1;  // MMA1's phase (waited by groups 0 and 1)
      fence_proxy_async();
      if (!(ok = sync())) break;
      if (tid == 0) {
        mmau_issue(OFF_T);
        if (GATE) issue(1u << BAR_GT, c);  // V is consumed: the gate tile takes its place
        if (more) issue((1u << BAR_K) | (1u << BAR_G), c + 1);  // k and g are consumed
      }
      wait(BAR_MMA, mma_par);  // u ready
      mma_par ^= 1;
      tc_fence_after();
      p6_spread();
      fence_proxy_async();
      if (!(ok = sync())) break;
      if (tid == 0) p7_issue(OFF_P);
      if (grp == 2 && more) p1(c + 1, tid - 256, 3);  // overlapped with the update and the output phase
      wait(BAR_MMA, mma_par);
      mma_par ^= 1;
      tc_fence_after();
      p8(nv, t0, par);
      ckpt_write((int64_t)c * C + nv);
      if (!(ok = sync())) break;
    }
  } else if (!producer) {
    // ---- consumer of a cluster pair: the state walk; T and P' of chunk c arrive from the
    //      producer in landing buffer c & 1 (FULL), which is handed back after the update
    //      (EMPTY) ---------------------------------------------------------------------------
    for (int c = 0; c < nchunks && ok; ++c) {
      const int64_t t0 = bos + (int64_t)c * C;
      const int nv = (int)((eos - t0) < C ? (eos - t0) : C);
      const uint32_t par = (uint32_t)(c & 1);
      const bool more = c + 1 < nchunks;
      const int b = c & 1;
      if (tid == 0 && c > 0) {  // V is free once the previous output tile has been read
        bulk_wait_read0();
        issue(1u << BAR_V, c);
      }
      x_rows(nv);
      fence_proxy_async();
      if (!(ok = sync())) break;
      if (tid == 0 && more) issue(1u << BAR_Q, c + 1);  // q is consumed
      if (tid == 256) mma1_issue(true, par);  // group 2 only decays in this phase
      if (grp < 2) {
        y_decay(nv, par, false, true);
      } else {  // S^T *= Gamma_C: MMA1 reads the split state in TA, not S
        decay(0, 4);
        wait(BAR_X, par);  // the state read is done: X may be rewritten
        kbar_items(nv, 0, KB2, tid - 256, 128);
      }
      fence_proxy_async();
      if (!(ok = sync())) break;
      if (tid == 0) {
        if (GATE) issue(1u << BAR_GT, c);  // V is consumed: the gate tile takes its place
        if (mbar_wait_cluster(bar(BAR_F0 + b), (uint32_t)((c >> 1) & 1))) {
          full_seen = c + 1;
          fence_proxy_async();
          mmau_issue(off_lt(b));
        } else {
          s_abort = 1;
        }
      }
      kbar_items(nv, KB2, C * 16, tid, NT);
      fence_proxy_async();
      if (!(ok = sync())) break;
      if (tid == 0 && more) issue((1u << BAR_K) | (1u << BAR_G), c + 1);
      wait(BAR_MMA, mma_par);  // u ready
      mma_par ^= 1;
      tc_fence_after();
      p6();
      fence_proxy_async();
      if (!(ok = sync())) break;
      if (tid == 0) p7_issue(off_lp(b));
      if (grp == 2 && more) p1(c + 1, tid - 256, 3);
      wait(BAR_MMA, mma_par);
      mma_par ^= 1;
      tc_fence_after();
      if (tid == 0) mbar_arrive_remote(bar(BAR_E0 + b), 1);  // landing buffer b is free
      // TA is free once the state read is done; groups 0 and 1 split the state while
      // group 2 is still in P1
      if (grp < 2 && more) s_split(2 * grp, 2);
      p8(nv, t0, par);
      ckpt_write((int64_t)c * C + nv);
      if (!(ok = sync())) break;
    }
  } else {
    // ---- producer of a cluster pair: A and P' of each chunk, the inverse T, written into the
    //      consumer's landing buffer c & 1 -------------------------------------------------
    // the producer loads no v and builds no X: A, the fp32 T and the inverse's block scratch
    // live there, clear of the operand regions, so the next chunk's operands can be built
    // while the inverse runs
    float *pA = reinterpret_cast<float *>(sm + OFF_X);
    float *pS = reinterpret_cast<float *>(sm + OFF_X + 20480);
    float *pT = reinterpret_cast<float *>(sm + OFF_V);
    // the tf32 T of chunk c is staged here (by chunk parity: buffer b is rewritten only after
    // the consumer has handed landing buffer b back, so its copy has been read) and sent by one
    // bulk copy that completes on the consumer's FULL barrier: no cluster fence on the remote
    // stores of 16 KB
    auto off_st = [](int b) { return OFF_X + 32768u + 16384u * (uint32_t)b; };
    if (ok && nchunks > 0) {
      ap_operands((int)((eos - bos) < C ? (eos - bos) : C), NT);
      fence_proxy_async();
    }
    ok = sync() && ok;
    for (int c = 0; c < nchunks && ok; ++c) {
      const int64_t t0 = bos + (int64_t)c * C;
      const int nv = (int)((eos - t0) < C ? (eos - t0) : C);
      const bool more = c + 1 < nchunks;
      const int b = c & 1;
      if (tid == 0) {
        if (more) issue((1u << BAR_Q) | (1u << BAR_K) | (1u << BAR_G), c + 1);
        ap_issue();
      }
      wait(BAR_MMA, mma_par);
      mma_par ^= 1;
      tc_fence_after();
      if (c >= 2 && !mbar_wait_cluster(bar(BAR_E0 + b), (uint32_t)(((c - 2) >> 1) & 1)))
        s_abort = 1;
      if (!(ok = sync())) break;
      // FULL of landing buffer b completes once P' (16 KB of asynchronous stores from every
      // warp) and T (one 16 KB bulk copy after the inverse) have landed
      if (tid == 256) mbar_arrive_expect_tx_remote(bar(BAR_F0 + b), 0, 32768);
      extract(nv, nullptr, map_shared_rank(sb + off_lp(b), 0), map_shared_rank(bar(BAR_F0 + b), 0),
              pA, (uint32_t)(c & 1));
      fence_proxy_async();
      // only the inverting group waits for every warp's rows of A; groups 0 and 1 go on to P1
      if (grp == 2) {  // FULL once T has landed: the consumer does not wait for P1 below
        asm volatile("bar.sync 6, 384;" ::: "memory");
        inverse(sm + off_st(b), pA, pT, pS);
        fence_proxy_async();
        asm volatile("bar.sync 3, 128;" ::: "memory");
        if (tid == 256) bulk_copy_to_peer(sb + off_lt(b), sb + off_st(b), 16384, bar(BAR_F0 + b), 0);
      } else {
        asm volatile("bar.arrive 6, 384;" ::: "memory");
        if (more) {  // P1 of chunk c + 1 on groups 0 and 1
          p1(c + 1, tid & 127, grp == 0 ? 2 : 1);  // prefix sums | beta and norms
          asm volatile("bar.sync 1, 256;" ::: "memory");
          asm volatile("bar.arrive 5, 384;" ::: "memory");  // P1 done: group 2 may join
        }
      }
      if (more) {  // the operands of chunk c + 1 on all three groups (group 2 after the inverse)
        if (grp == 2) asm volatile("bar.sync 5, 384;" ::: "memory");
        const int64_t t1 = t0 + C;
        ap_operands((int)((eos - t1) < C ? (eos - t1) : C), NT);
      }
      fence_proxy_async();
      if (!(ok = sync())) break;
    }
  }

  if (ok && !producer && kc < kend && tid == 0 && a.err) atomicOr(a.err, ERR_BAD_INDEX);
  if (tid == 0) bulk_wait0();  // output tiles written before the shared memory is released

  // ---- final state: S[i][j] = S^T[j][i] ------------------------------------------------
  if (ok && a.final_state && grp < 2 && !producer) {
    ST *dst = reinterpret_cast<ST *>(a.final_state) + ((size_t)n * H + h) * D * D;
#pragma unroll 1
    for (int g32 = 0; g32 < 2; ++g32) {
      float v[32];
      const int i0 = 64 * grp + 32 * g32;
      tmem_ld32(tm + lane_off + TM_S + i0, v);
      tmem_wait_ld();
#pragma unroll
      for (int x = 0; x < 32; ++x) dst[(size_t)(i0 + x) * D + j] = from_f<ST>(v[x]);
    }
  }
  if (!ok && tid == 0) {
    if (s_abort && a.err) atomicOr(a.err, ERR_MBAR_TIMEOUT);  // a bounded wait ran out
    // drain: let loads and MMAs still in flight land (bounded) before the CTA exits.  s_pend
    // marks every barrier that was ever armed and s_ppar the parity of its latest phase, whose
    // wait returns at once when that phase has completed
    for (int b = 0; b < NBAR; ++b)
      if (s_pend & (1u << b)) mbar_wait(bar(b), s_ppar[b]);
    // a consumer that stops early: the producer's bulk copies of T for the next two chunks
    // may be in flight into this CTA's shared memory; let them land (bounded) before it goes
    if (PAIR && !producer)
      for (int k = full_seen; k < full_seen + 2 && k < nchunks; ++k)
        mbar_wait_cluster(bar(BAR_F0 + (k & 1)), (uint32_t)((k >> 1) & 1));
  }
  tc_fence_before();
  __syncthreads();
  if (PAIR) cluster_sync();  // neither CTA leaves while the other may still write to it
  if (warp == 0) tmem_dealloc(tm, TM_COLS);
}

// ---- host side --------------------------------------------------------------------------


bool make_map(CUtensorMap *m, const void *ptr, bool f32, int64_t T, int H) {
  const int esz = f32 ? 4 : 2;
  cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)T};
  cuuint64_t strides[2] = {(cuuint64_t)D * esz, (cuuint64_t)H * D * esz};
  cuuint32_t box[3] = {(cuuint32_t)(128 / esz), 1, (cuuint32_t)C};
  cuuint32_t es[3] = {1, 1, 1};
  auto fn = tensor_map_encoder();
  if (!fn) return false;
  return fn(m, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
            const_cast<void *>(ptr), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// output [T, H, 128] bf16 (or FP8 codes, one byte each): plain (unswizzled) boxes of 64
// tokens x 128 channels
bool make_out_map(CUtensorMap *m, void *ptr, int64_t T, int H, bool fp8) {
  const int esz = fp8 ? 1 : 2;
  cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)T};
  cuuint64_t strides[2] = {(cuuint64_t)D * esz, (cuuint64_t)H * D * esz};
  cuuint32_t box[3] = {(cuuint32_t)D, 1, (cuuint32_t)C};
  cuuint32_t es[3] = {1, 1, 1};
  auto fn = tensor_map_encoder();
  if (!fn) return false;
  return fn(m, fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, ptr,
            dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <typename ST, bool GATE, bool PAIR, bool QUANT>
cudaError_t launch_typed(const TcArgs &a, const Maps &maps, cudaStream_t s) {
  static std::atomic<bool> attr_set[64];  // the opt-in done, per device (idempotent if raced)
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !attr_set[dev].load()) {
    cudaError_t e = cudaFuncSetAttribute(prefill_tc_kernel<ST, GATE, PAIR, QUANT>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    if (e != cudaSuccess) return e;
    attr_set[dev].store(true);
  }
  if (!PAIR) {
    prefill_tc_kernel<ST, GATE, PAIR, QUANT><<<dim3(a.H, a.n_seqs), NT, SMEM_BYTES, s>>>(a, maps);
    return cudaGetLastError();
  }
  cudaLaunchConfig_t cfg;
  memset(&cfg, 0, sizeof cfg);
  cfg.gridDim = dim3(2 * a.H, a.n_seqs);
  cfg.blockDim = dim3(NT);
  cfg.dynamicSmemBytes = SMEM_BYTES;
  cfg.stream = s;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = 2;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, prefill_tc_kernel<ST, GATE, PAIR, QUANT>, a, maps);
}

// A cluster pair per (head, sequence) when the pairs fit on the device at once (small
// batches: otherwise the SMs are better spent on more units), unless the caller chose a form.
bool use_pair(const TcArgs &a) {
  if (a.form == 1) return false;
  if (a.form == 2) return true;
  int dev = 0, nsm = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  if (cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return false;
  return (int64_t)a.n_seqs * a.H * 2 <= nsm;
}

template <bool QUANT>
cudaError_t dispatch(const TcArgs &a, const Maps &maps, bool st_bf16, bool gate, bool pair,
                     cudaStream_t s) {
  if (pair) {
    if (st_bf16)
      return gate ? launch_typed<bf16, true, true, QUANT>(a, maps, s)
                  : launch_typed<bf16, false, true, QUANT>(a, maps, s);
    return gate ? launch_typed<float, true, true, QUANT>(a, maps, s)
                : launch_typed<float, false, true, QUANT>(a, maps, s);
  }
  if (st_bf16)
    return gate ? launch_typed<bf16, true, false, QUANT>(a, maps, s)
                : launch_typed<bf16, false, false, QUANT>(a, maps, s);
  return gate ? launch_typed<float, true, false, QUANT>(a, maps, s)
              : launch_typed<float, false, false, QUANT>(a, maps, s);
}

}  // namespace

bool prefill_tc_supported(int d, bool io_bf16) {
  if (d != D || !io_bf16) return false;
  int dev = 0, major = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess)
    return false;
  return major == 10 && tensor_map_encoder() != nullptr;
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
        !make_out_map(&maps.out, a.out_q ? static_cast<void *>(a.out_q) : a.out, total_tokens,
                      a.H, a.out_q != nullptr))
      return cudaErrorInvalidValue;
    // gate logits [T, H, 128] bf16: the same plain boxes as the output
    if (a.gate && !make_out_map(&maps.gate, const_cast<void *>(a.gate), total_tokens, a.H, false))
      return cudaErrorInvalidValue;
  }
  const bool gate = a.gate != nullptr, pair = use_pair(a);
  if (a.out_q) return dispatch<true>(a, maps, st_bf16, gate, pair, s);
  return dispatch<false>(a, maps, st_bf16, gate, pair, s);
}

}  // namespace kda

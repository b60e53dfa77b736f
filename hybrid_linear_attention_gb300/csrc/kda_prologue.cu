// kda_prologue.cu -- the short convolution in front of the KDA recurrence.
//
// "Each projection passes through its own causal short convolution of width four with SiLU
// activation ... The KDA kernel normalizes queries and keys" ("Ling-3.1-flash: Grouped
// Routing and Two Different MLA Caches", section "KDA replaces a token list with a recurrent
// matrix").  Per channel c: y[t,c] = SiLU(sum_j w[c][j] x[t-3+j, c]); taps before a
// sequence's first token read that sequence's conv tail (three raw inputs, oldest first).
//
// Kernels:
//   prologue_kernel     packed prefill: conv + SiLU (+ per-head L2 of q, k) for a share of
//                       the tokens x (stream, head) rows, 16-byte vectors, one read per
//                       input, the next tokens' inputs always in flight.
//                       The gate activations beta = sigmoid(logit), g = max(g_raw, g_min)
//                       are spread over the same CTAs after their tokens.
//   conv_tail_kernel    afterwards, the new tail of every sequence (separate launch, so the
//                       in-place update never races with the reads of the old tail).
//   conv_update_kernel  decode: one new token per sequence, tail shifted in place.
#include "kda_common.cuh"
#include "kda_internal.h"

namespace kda {
namespace {

constexpr int PNT = 256;     // threads per prologue CTA
constexpr int MIN_TOK = 16;  // fewest tokens a prologue CTA walks

// eight consecutive channels as fp32 (16-byte bf16 vector, or two fp32 vectors)
__device__ __forceinline__ void load8(const bf16 *p, float (&v)[8]) {
  const uint4 u = *reinterpret_cast<const uint4 *>(p);
  v[0] = __uint_as_float(u.x << 16), v[1] = __uint_as_float(u.x & 0xffff0000u);
  v[2] = __uint_as_float(u.y << 16), v[3] = __uint_as_float(u.y & 0xffff0000u);
  v[4] = __uint_as_float(u.z << 16), v[5] = __uint_as_float(u.z & 0xffff0000u);
  v[6] = __uint_as_float(u.w << 16), v[7] = __uint_as_float(u.w & 0xffff0000u);
}
__device__ __forceinline__ void load8(const float *p, float (&v)[8]) {
  const float4 a = *reinterpret_cast<const float4 *>(p);
  const float4 b = *reinterpret_cast<const float4 *>(p + 4);
  v[0] = a.x, v[1] = a.y, v[2] = a.z, v[3] = a.w, v[4] = b.x, v[5] = b.y, v[6] = b.z, v[7] = b.w;
}
// x * sigmoid(x) with the special-function unit's 2^x and reciprocal (relative error ~1e-7)
__device__ __forceinline__ float silu_fast(float x) {
  float e, r;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e) : "f"(-1.4426950408889634f * x));
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(1.f + e));
  return x * r;
}
__device__ __forceinline__ uint32_t bf2(float a, float b) {
  uint32_t d;  // round to nearest even; the first source lands in the upper half
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(b), "f"(a));
  return d;
}
__device__ __forceinline__ void store8(bf16 *p, const float (&v)[8]) {
  *reinterpret_cast<uint4 *>(p) =
      make_uint4(bf2(v[0], v[1]), bf2(v[2], v[3]), bf2(v[4], v[5]), bf2(v[6], v[7]));
}
__device__ __forceinline__ void store8(float *p, const float (&v)[8]) {
  *reinterpret_cast<float4 *>(p) = make_float4(v[0], v[1], v[2], v[3]);
  *reinterpret_cast<float4 *>(p + 4) = make_float4(v[4], v[5], v[6], v[7]);
}
// eight consecutive channels as loaded, converted to fp32 only when used (a bf16 vector is
// four registers, so a deep prefetch ring stays small)
template <typename IO> struct Raw;
template <> struct Raw<bf16> { uint4 u; };
template <> struct Raw<float> { float4 a, b; };
__device__ __forceinline__ Raw<bf16> load_raw(const bf16 *p) {
  return Raw<bf16>{*reinterpret_cast<const uint4 *>(p)};
}
__device__ __forceinline__ Raw<float> load_raw(const float *p) {
  return Raw<float>{*reinterpret_cast<const float4 *>(p), *reinterpret_cast<const float4 *>(p + 4)};
}
__device__ __forceinline__ void unpack8(const Raw<bf16> &r, float (&v)[8]) {
  v[0] = __uint_as_float(r.u.x << 16), v[1] = __uint_as_float(r.u.x & 0xffff0000u);
  v[2] = __uint_as_float(r.u.y << 16), v[3] = __uint_as_float(r.u.y & 0xffff0000u);
  v[4] = __uint_as_float(r.u.z << 16), v[5] = __uint_as_float(r.u.z & 0xffff0000u);
  v[6] = __uint_as_float(r.u.w << 16), v[7] = __uint_as_float(r.u.w & 0xffff0000u);
}
__device__ __forceinline__ void unpack8(const Raw<float> &r, float (&v)[8]) {
  v[0] = r.a.x, v[1] = r.a.y, v[2] = r.a.z, v[3] = r.a.w;
  v[4] = r.b.x, v[5] = r.b.y, v[6] = r.b.z, v[7] = r.b.w;
}

// Conv weights of eight consecutive channels (channel e, tap j at 4e + j), widened to fp32 once
// (kept packed, they cost an unpack per tap and token: measured slower).
template <typename IO> struct ConvW;
template <> struct ConvW<bf16> {
  float w[8][4];
  __device__ __forceinline__ void load(const bf16 *cw, bool act) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint4 u = act ? *reinterpret_cast<const uint4 *>(cw + 8 * q) : make_uint4(0, 0, 0, 0);
      const uint32_t p[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        w[2 * q + (e >> 1)][2 * (e & 1)] = __uint_as_float(p[e] << 16);
        w[2 * q + (e >> 1)][2 * (e & 1) + 1] = __uint_as_float(p[e] & 0xffff0000u);
      }
    }
  }
  __device__ __forceinline__ float tap(int y, int j) const { return w[y][j]; }
};
template <> struct ConvW<float> {
  float w[8][4];
  __device__ __forceinline__ void load(const float *cw, bool act) {
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const float4 u = act ? *reinterpret_cast<const float4 *>(cw + 4 * q)
                           : make_float4(0.f, 0.f, 0.f, 0.f);
      w[q][0] = u.x, w[q][1] = u.y, w[q][2] = u.z, w[q][3] = u.w;
    }
  }
  __device__ __forceinline__ float tap(int y, int j) const { return w[y][j]; }
};

// Gate activations, elementwise: g = max(g_raw, g_min) (four at a time), beta = sigmoid;
// thread e0 of nthr takes elements e0, e0 + nthr, ...  (without g_raw only the T * H gates)
template <int D>
__device__ __forceinline__ void gate_act(const ProArgs &a, int64_t e0, int64_t nthr) {
  const int64_t n4 = a.g_raw ? a.T * a.H * (int64_t)D / 4 : 0, nb = a.T * a.H;
  for (int64_t e = e0; e < n4; e += nthr) {
    const float4 v = reinterpret_cast<const float4 *>(a.g_raw)[e];
    reinterpret_cast<float4 *>(a.g)[e] = make_float4(fmaxf(v.x, a.g_min), fmaxf(v.y, a.g_min),
                                                     fmaxf(v.z, a.g_min), fmaxf(v.w, a.g_min));
    if (a.beta_logit && e < nb) a.beta[e] = sigmoidf_(a.beta_logit[e]);
  }
  if (a.beta_logit)
    for (int64_t e = n4 + e0; e < nb; e += nthr) a.beta[e] = sigmoidf_(a.beta_logit[e]);
}

// One CTA: a share of the tokens x PNT/(D/8) rows of D channels (a row = one head of one of the
// q, k, v streams); D/8 threads per row, eight channels each.  Every thread walks the tile's
// tokens in order with the last three raw inputs of its channels in registers (each input
// is read once); at a sequence start inside the tile the window restarts from that
// sequence's conv tail (zeros without one).  The per-token L2 norm of q and k is a shuffle
// reduction over the row's D/8 lanes.
template <int D, typename IO>
__global__ void __launch_bounds__(PNT, 2) prologue_kernel(const ProArgs a) {
  constexpr int TPH = D / 8;
  constexpr int NU = PNT / TPH;
  const int H = a.H, C = 3 * H * D;
  const int tid = threadIdx.x, sub = tid % TPH;
  const int u = blockIdx.y * NU + tid / TPH;  // stream * H + head
  const bool act = u < 3 * H;
  const int stream = act ? u / H : 0, h = act ? u % H : 0;
  const int64_t c0 = (int64_t)stream * H * D + (int64_t)h * D + 8 * sub;
  // a contiguous, balanced share of the tokens (gridDim.x shares of T)
  const int64_t t0 = a.T * blockIdx.x / gridDim.x;
  const int64_t t1 = a.T * (blockIdx.x + 1) / gridDim.x;
  const IO *x = reinterpret_cast<const IO *>(a.x);
  const IO *cs = reinterpret_cast<const IO *>(a.conv_state);
  IO *dst = reinterpret_cast<IO *>(stream == 0 ? a.q : stream == 1 ? a.k : a.v);
  const bool norm = a.l2norm_qk && stream < 2;

  ConvW<IO> w;  // the four taps of this thread's eight channels
  w.load(reinterpret_cast<const IO *>(a.conv_w) + 4 * c0, act);
  int n = seq_of_token(a.cu_seqlens, a.n_seqs, t0);
  int64_t bos = a.cu_seqlens[n], eos = a.cu_seqlens[n + 1];
  if ((bos > t0 || eos <= t0) && threadIdx.x == 0 && a.err) atomicOr(a.err, ERR_BAD_SEQLEN);
  float win[3][8];
#pragma unroll
  for (int k = 0; k < 3; ++k) {
    const int64_t src = t0 - 3 + k;
    if (act && src >= bos && src >= 0) load8(x + src * C + c0, win[k]);
    else if (act && cs && src >= bos - 3)
      load8(cs + ((int64_t)n * 3 + 3 + (src - bos)) * C + c0, win[k]);
    else
#pragma unroll
      for (int y = 0; y < 8; ++y) win[k][y] = 0.f;
  }

  // rolling prefetch: the raw inputs of the next PF tokens stay in flight while a token is
  // convolved (slot i of the ring holds token tb + i, refilled with token tb + i + PF)
  constexpr int PF = sizeof(IO) == 2 ? 6 : 2;
  Raw<IO> xr[PF];
#pragma unroll
  for (int i = 0; i < PF; ++i)
    if (act && t0 + i < t1) xr[i] = load_raw(x + (t0 + i) * C + c0);
  const IO *xn = x + (t0 + PF) * C + c0;              // token t + PF of this thread's channels
  IO *dp = dst + (t0 * H + h) * (int64_t)D + 8 * sub;  // output row of token t
  for (int64_t tb = t0; tb < t1; tb += PF) {
#pragma unroll
    for (int i = 0; i < PF; ++i) {
      const int64_t t = tb + i;
      if (t >= t1) break;
      float xv[8];
      unpack8(xr[i], xv);
      if (act && t + PF < t1) xr[i] = load_raw(xn);
      xn += C;
      if (t == eos) {  // next non-empty sequence starts here: its conv tail is the history
        do {
          ++n;
          bos = a.cu_seqlens[n];
          eos = a.cu_seqlens[n + 1];
        } while (eos <= t && n + 1 < a.n_seqs);
#pragma unroll
        for (int k = 0; k < 3; ++k) {
          if (act && cs) load8(cs + ((int64_t)n * 3 + k) * C + c0, win[k]);
          else
#pragma unroll
            for (int y = 0; y < 8; ++y) win[k][y] = 0.f;
        }
      }
      float yv[8];
#pragma unroll
      for (int y = 0; y < 8; ++y) {
        float acc = w.tap(y, 0) * win[0][y];
        acc = fmaf(w.tap(y, 1), win[1][y], acc);
        acc = fmaf(w.tap(y, 2), win[2][y], acc);
        acc = fmaf(w.tap(y, 3), xv[y], acc);
        yv[y] = silu_fast(acc);
        win[0][y] = win[1][y], win[1][y] = win[2][y], win[2][y] = xv[y];
      }
      if (a.l2norm_qk) {  // the same for the whole grid: every lane of a warp takes part in
                          // the shuffle (a warp may hold rows of different streams)
        float ss = 0.f;
#pragma unroll
        for (int y = 0; y < 8; ++y) ss = fmaf(yv[y], yv[y], ss);
#pragma unroll
        for (int off = TPH / 2; off >= 1; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
        if (norm) {
          const float r = rsqrtf(ss + a.l2_eps);
#pragma unroll
          for (int y = 0; y < 8; ++y) yv[y] *= r;
        }
      }
      if (act) store8(dp, yv);
      dp += (int64_t)H * D;
    }
  }
  // the gate activations ride along: each CTA takes a grid-strided share after its tokens (no
  // launch of their own)
  if (a.beta_logit || a.g_raw)
    gate_act<D>(a, ((int64_t)blockIdx.y * gridDim.x + blockIdx.x) * PNT + tid,
                (int64_t)gridDim.x * gridDim.y * PNT);
}

// New tail of sequence n: the last three raw inputs, reaching into the old tail when the
// sequence is shorter than three; a length-0 sequence keeps its tail.  Raw element copies.
template <typename E>
__global__ void conv_tail_kernel(const E *x, E *cs, const int32_t *cu, int C, int64_t T,
                                 int *err) {
  const int n = blockIdx.y;
  const int c = blockIdx.x * blockDim.x + threadIdx.x;
  if (c >= C) return;
  const int64_t bos = cu[n], eos = cu[n + 1];
  if (bos < 0 || eos > T) {  // offsets outside the rows: flagged, tail kept
    if (c == 0 && err) atomicOr(err, ERR_BAD_SEQLEN);
    return;
  }
  if (eos <= bos) return;
  E *st = cs + (int64_t)n * 3 * C + c;
  E nv[3];
#pragma unroll
  for (int r = 0; r < 3; ++r) {
    const int64_t src = eos - 3 + r;
    nv[r] = src >= bos ? x[src * C + c] : st[(3 + (src - bos)) * C];
  }
#pragma unroll
  for (int r = 0; r < 3; ++r) st[r * C] = nv[r];
}

// Conv tail at checkpoint k of sequence n (pos tokens in): the three raw inputs before it,
// oldest first, reaching into the sequence's prior tail (zeros without one) when pos < 3.
// Raw element copies.  A position outside 1..length is flagged and skipped.
template <typename E>
__global__ void conv_ckpt_kernel(const E *x, const E *cs, const int32_t *cu, int n_seqs,
                                 const int32_t *ckpt_cu, const int32_t *ckpt_pos, int C,
                                 int64_t T, E *out, int *err) {
  const int kk = blockIdx.y;
  const int c = blockIdx.x * blockDim.x + threadIdx.x;
  if (c >= C) return;
  int lo = 0, hi = n_seqs;  // sequence n with ckpt_cu[n] <= kk < ckpt_cu[n + 1]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (ckpt_cu[mid] <= kk) lo = mid; else hi = mid;
  }
  const int n = lo;
  const int64_t bos = cu[n], len = (int64_t)cu[n + 1] - bos, pos = ckpt_pos[kk];
  if (bos < 0 || bos + len > T || pos < 1 || pos > len) {
    if (c == 0 && err) atomicOr(err, ERR_BAD_INDEX);
    return;
  }
#pragma unroll
  for (int r = 0; r < 3; ++r) {
    const int64_t src = pos - 3 + r;  // position within the sequence
    E val;
    if (src >= 0) val = x[(bos + src) * C + c];
    else if (cs) val = cs[((int64_t)n * 3 + 3 + src) * C + c];
    else val = E(0);
    out[((int64_t)kk * 3 + r) * C + c] = val;
  }
}

template <typename IO>
__global__ void conv_update_kernel(const ConvArgs a) {
  const int n = blockIdx.y;
  const int c = blockIdx.x * blockDim.x + threadIdx.x;
  if (c >= a.channels) return;
  const int C = a.channels;
  const int slot = a.slot_idx ? a.slot_idx[n] : n;
  if (slot < 0 || slot >= a.n_slots) {  // an index outside the pool: flagged, skipped
    if (c == 0 && a.err) atomicOr(a.err, ERR_BAD_INDEX);
    return;
  }
  IO *st = reinterpret_cast<IO *>(a.conv_state) + (int64_t)slot * 3 * C + c;
  const IO *cw = reinterpret_cast<const IO *>(a.conv_w) + 4 * (int64_t)c;
  const IO x0 = st[0], x1 = st[C], x2 = st[2 * C];
  const IO xn = reinterpret_cast<const IO *>(a.x_new)[(int64_t)n * C + c];
  const float acc = to_f(cw[0]) * to_f(x0) + to_f(cw[1]) * to_f(x1) + to_f(cw[2]) * to_f(x2) +
                    to_f(cw[3]) * to_f(xn);
  reinterpret_cast<IO *>(a.y)[(int64_t)n * C + c] = from_f<IO>(siluf_(acc));
  st[0] = x1;
  st[C] = x2;
  st[2 * C] = xn;
}

template <int D, typename IO>
cudaError_t launch_pro(const ProArgs &a, cudaStream_t s) {
  if (a.T > 0) {
    int dev = 0, nsm = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    // rows of D channels (one head of one stream) in groups of NU; the tokens are split into
    // as many contiguous shares as fill one wave at two CTAs per SM (at least MIN_TOK tokens
    // a share), so every CTA walks the same number of tokens and no partial wave is left
    constexpr int NU = PNT / (D / 8);
    const int64_t groups = (3 * a.H + NU - 1) / NU;
    int64_t shares = 2 * (int64_t)nsm / groups;
    const int64_t most = (a.T + MIN_TOK - 1) / MIN_TOK;
    if (shares > most) shares = most;
    if (shares < 1) shares = 1;
    const dim3 grid((unsigned)shares, (unsigned)groups);
    prologue_kernel<D, IO><<<grid, PNT, 0, s>>>(a);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  if (a.conv_state && a.n_seqs > 0) {
    const int C = 3 * a.H * D;
    const dim3 grid((C + 255) / 256, a.n_seqs);
    if (sizeof(IO) == 2)
      conv_tail_kernel<uint16_t><<<grid, 256, 0, s>>>(
          reinterpret_cast<const uint16_t *>(a.x), reinterpret_cast<uint16_t *>(a.conv_state),
          a.cu_seqlens, C, a.T, a.err);
    else
      conv_tail_kernel<uint32_t><<<grid, 256, 0, s>>>(
          reinterpret_cast<const uint32_t *>(a.x), reinterpret_cast<uint32_t *>(a.conv_state),
          a.cu_seqlens, C, a.T, a.err);
    return cudaGetLastError();
  }
  return cudaSuccess;
}

}  // namespace

cudaError_t launch_prologue(const ProArgs &a, int D, bool io_bf16, cudaStream_t s) {
  if (D == 128) return io_bf16 ? launch_pro<128, bf16>(a, s) : launch_pro<128, float>(a, s);
  if (D == 16) return io_bf16 ? launch_pro<16, bf16>(a, s) : launch_pro<16, float>(a, s);
  return cudaErrorInvalidValue;
}

cudaError_t launch_conv_ckpt(const void *x, const void *conv_state, const int32_t *cu,
                             int n_seqs, int64_t T, const int32_t *ckpt_cu,
                             const int32_t *ckpt_pos, int n_ckpt, int channels, void *out,
                             bool io_bf16, int *err, cudaStream_t s) {
  if (n_ckpt == 0) return cudaSuccess;
  const dim3 grid((channels + 255) / 256, n_ckpt);
  if (io_bf16)
    conv_ckpt_kernel<uint16_t><<<grid, 256, 0, s>>>(
        reinterpret_cast<const uint16_t *>(x), reinterpret_cast<const uint16_t *>(conv_state),
        cu, n_seqs, ckpt_cu, ckpt_pos, channels, T, reinterpret_cast<uint16_t *>(out), err);
  else
    conv_ckpt_kernel<uint32_t><<<grid, 256, 0, s>>>(
        reinterpret_cast<const uint32_t *>(x), reinterpret_cast<const uint32_t *>(conv_state),
        cu, n_seqs, ckpt_cu, ckpt_pos, channels, T, reinterpret_cast<uint32_t *>(out), err);
  return cudaGetLastError();
}

// The bounded-wait path the tensor-core kernels take when an mbarrier phase never completes:
// one thread waits on a barrier nothing arrives at, gives up after `limit` probes and raises
// the library's sticky flag, as those kernels do (the failure is made on purpose, without a
// GPU fault: the wait ends and the kernel returns).
__global__ void wait_probe_kernel(long limit, int *err) {
  __shared__ __align__(8) uint64_t bar;
  const uint32_t b = (uint32_t)__cvta_generic_to_shared(&bar);
  asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(b));
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  bool done = false;
  for (long it = 0; it < limit && !done; ++it) {
    uint32_t ok;
    asm volatile(
        "{\n.reg .pred p;\nmbarrier.try_wait.parity.shared::cta.b64 p, [%1], 0;\n"
        "selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(b)
        : "memory");
    done = ok != 0;
  }
  if (!done && err) atomicOr(err, ERR_MBAR_TIMEOUT);
}

cudaError_t launch_wait_probe(long limit, int *err, cudaStream_t s) {
  wait_probe_kernel<<<1, 1, 0, s>>>(limit, err);
  return cudaGetLastError();
}

cudaError_t launch_conv_update(const ConvArgs &a, bool io_bf16, cudaStream_t s) {
  if (a.n_seqs == 0) return cudaSuccess;
  const dim3 grid((a.channels + 255) / 256, a.n_seqs);
  if (io_bf16) conv_update_kernel<bf16><<<grid, 256, 0, s>>>(a);
  else conv_update_kernel<float><<<grid, 256, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace kda

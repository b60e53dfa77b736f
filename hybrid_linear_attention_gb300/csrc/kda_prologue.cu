// kda_prologue.cu -- the short convolution in front of the KDA recurrence.
//
// "Each projection passes through its own causal short convolution of width four with SiLU
// activation ... The KDA kernel normalizes queries and keys" ("Ling-3.1-flash: Grouped
// Routing and Two Different MLA Caches", section "KDA replaces a token list with a recurrent
// matrix").  Per channel c: y[t,c] = SiLU(sum_j w[c][j] x[t-3+j, c]); taps before a
// sequence's first token read that sequence's conv tail (three raw inputs, oldest first).
//
// Kernels:
//   prologue_kernel     packed prefill: conv + SiLU (+ per-head L2 of q, k) for a tile of
//                       tokens x one (stream, head) group of d channels; also the gate
//                       activations beta = sigmoid(logit), g = max(g_raw, g_min).
//   conv_tail_kernel    afterwards, the new tail of every sequence (separate launch, so the
//                       in-place update never races with the reads of the old tail).
//   conv_update_kernel  decode: one new token per sequence, tail shifted in place.
#include "kda_common.cuh"
#include "kda_internal.h"

namespace kda {
namespace {

constexpr int PT = 16;  // tokens per prologue tile

template <int D, typename IO>
__global__ void __launch_bounds__(D / 2 < 32 ? 32 : D / 2)
    prologue_kernel(const ProArgs a) {
  constexpr int NT = D / 2 < 32 ? 32 : D / 2;
  constexpr int NW = NT / 32;
  __shared__ int64_t s_bos[PT];
  __shared__ int s_seq[PT];
  __shared__ float s_ss[NW][PT];
  __shared__ float s_r[PT];

  const int H = a.H, C = 3 * H * D;
  const int grp = blockIdx.y;                   // stream * H + head
  const int stream = grp / H, h = grp % H;
  const int64_t t0 = (int64_t)blockIdx.x * PT;
  const int nt = (int)((a.T - t0) < PT ? (a.T - t0) : PT);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int c0 = stream * H * D + h * D + 2 * tid;  // this thread's first channel
  const bool act = 2 * tid < D;

  if (tid < nt) {
    const int n = seq_of_token(a.cu_seqlens, a.n_seqs, t0 + tid);
    s_seq[tid] = n;
    s_bos[tid] = a.cu_seqlens[n];
  }
  __syncthreads();

  const IO *x = reinterpret_cast<const IO *>(a.x);
  const IO *cs = reinterpret_cast<const IO *>(a.conv_state);
  float w[2][4];
  if (act) {
    const IO *cw = reinterpret_cast<const IO *>(a.conv_w);
#pragma unroll
    for (int e = 0; e < 2; ++e)
#pragma unroll
      for (int j = 0; j < 4; ++j) w[e][j] = to_f(cw[4 * (c0 + e) + j]);
  }

  float y[PT][2];
#pragma unroll
  for (int tt = 0; tt < PT; ++tt) {
    y[tt][0] = y[tt][1] = 0.f;
    if (tt < nt && act) {
      const int64_t t = t0 + tt, bos = s_bos[tt];
      float acc0 = 0.f, acc1 = 0.f;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int64_t src = t - 3 + j;
        float2 xv = make_float2(0.f, 0.f);
        if (src >= bos) xv = load2(x + src * C + c0);
        else if (cs) xv = load2(cs + ((int64_t)s_seq[tt] * 3 + 3 + (src - bos)) * C + c0);
        acc0 = fmaf(w[0][j], xv.x, acc0);
        acc1 = fmaf(w[1][j], xv.y, acc1);
      }
      y[tt][0] = siluf_(acc0);
      y[tt][1] = siluf_(acc1);
    }
  }

  if (a.l2norm_qk && stream < 2) {  // per-token L2 over the head's D channels
#pragma unroll
    for (int tt = 0; tt < PT; ++tt) {
      const float ss = warp_sum(y[tt][0] * y[tt][0] + y[tt][1] * y[tt][1]);
      if (lane == 0) s_ss[warp][tt] = ss;
    }
    __syncthreads();
    if (tid < PT) {
      float ss = 0.f;
#pragma unroll
      for (int w2 = 0; w2 < NW; ++w2) ss += s_ss[w2][tid];
      s_r[tid] = rsqrtf(ss + a.l2_eps);
    }
    __syncthreads();
#pragma unroll
    for (int tt = 0; tt < PT; ++tt) y[tt][0] *= s_r[tt], y[tt][1] *= s_r[tt];
  }

  IO *dst = reinterpret_cast<IO *>(stream == 0 ? a.q : stream == 1 ? a.k : a.v);
  if (act) {
#pragma unroll
    for (int tt = 0; tt < PT; ++tt)
      if (tt < nt) store2(dst + ((t0 + tt) * H + h) * D + 2 * tid, make_float2(y[tt][0], y[tt][1]));
  }

  if (stream == 0) {  // gate activations for this head's tokens
    if (a.g_raw && act) {
#pragma unroll 4
      for (int tt = 0; tt < nt; ++tt) {
        const size_t row = ((size_t)(t0 + tt) * H + h) * D + 2 * tid;
        const float2 gr = load2(a.g_raw + row);
        store2(a.g + row, make_float2(fmaxf(gr.x, a.g_min), fmaxf(gr.y, a.g_min)));
      }
    }
    if (a.beta_logit && tid < nt) {
      const size_t i = (size_t)(t0 + tid) * H + h;
      a.beta[i] = sigmoidf_(a.beta_logit[i]);
    }
  }
}

// New tail of sequence n: the last three raw inputs, reaching into the old tail when the
// sequence is shorter than three; a length-0 sequence keeps its tail.  Raw element copies.
template <typename E>
__global__ void conv_tail_kernel(const E *x, E *cs, const int32_t *cu, int C) {
  const int n = blockIdx.y;
  const int c = blockIdx.x * blockDim.x + threadIdx.x;
  if (c >= C) return;
  const int64_t bos = cu[n], eos = cu[n + 1];
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

template <typename IO>
__global__ void conv_update_kernel(const ConvArgs a) {
  const int n = blockIdx.y;
  const int c = blockIdx.x * blockDim.x + threadIdx.x;
  if (c >= a.channels) return;
  const int C = a.channels;
  const int slot = a.slot_idx ? a.slot_idx[n] : n;
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
  constexpr int NT = D / 2 < 32 ? 32 : D / 2;
  if (a.T > 0) {
    const dim3 grid((unsigned)((a.T + PT - 1) / PT), 3 * a.H);
    prologue_kernel<D, IO><<<grid, NT, 0, s>>>(a);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  if (a.conv_state && a.n_seqs > 0) {
    const int C = 3 * a.H * D;
    const dim3 grid((C + 255) / 256, a.n_seqs);
    if (sizeof(IO) == 2)
      conv_tail_kernel<uint16_t><<<grid, 256, 0, s>>>(
          reinterpret_cast<const uint16_t *>(a.x), reinterpret_cast<uint16_t *>(a.conv_state),
          a.cu_seqlens, C);
    else
      conv_tail_kernel<uint32_t><<<grid, 256, 0, s>>>(
          reinterpret_cast<const uint32_t *>(a.x), reinterpret_cast<uint32_t *>(a.conv_state),
          a.cu_seqlens, C);
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

cudaError_t launch_conv_update(const ConvArgs &a, bool io_bf16, cudaStream_t s) {
  if (a.n_seqs == 0) return cudaSuccess;
  const dim3 grid((a.channels + 255) / 256, a.n_seqs);
  if (io_bf16) conv_update_kernel<bf16><<<grid, 256, 0, s>>>(a);
  else conv_update_kernel<float><<<grid, 256, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace kda

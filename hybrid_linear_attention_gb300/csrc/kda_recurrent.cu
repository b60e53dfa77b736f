// kda_recurrent.cu -- token-serial KDA recurrence in fp32: the decode step (one token per
// sequence, state streamed from HBM once and written once) and the exact-fp32 prefill path.
//
// Per head and token ("Ling-3.1-flash: a 560B hybrid-attention MoE, counted from its
// safetensors headers", section "How KDA and MLA split the work", the state equation, with
// the delta-rule write of "Ling-3.1-flash: Grouped Routing and Two Different MLA Caches",
// section "KDA replaces a token list with a recurrent matrix"):
//     S' = Diag(exp(max(g, g_min))) S;  u = beta (v - S'^T k);  S = S' + k u^T;
//     o  = scale S^T q = scale (S'^T q + u (k.q))
// so one pass over S gives both column reductions (S'^T k and S'^T q) and the update.
//
// Decode takes one token per sequence, or K tokens (the draft of a speculative step, with the
// state after each token kept for rollback: "Ling-3.1-flash: Grouped Routing and Two
// Different MLA Caches", section "KDA replaces a token list with a recurrent matrix", counts
// speculative rollback state among the per-sequence costs; "Ling-3.1-flash: What 63
// Linear-Attention Layers Do to the KV Budget", section "Where the hybrid makes serving
// harder", reports the MTP acceptance lengths).
//
// Layout of the work: one CTA per (head, sequence) for prefill; for decode a persistent grid
// (as many CTAs as fit on the device) walks the (sequence, head) units in strides and asks L2
// for the next unit's state and inputs before it works on the current one, so the state
// stream stays queued while the CTA computes.  The D x D state is spread over the CTA as
// tiles of RPT rows x 4 columns per thread (float4 along the value dimension, so a warp's
// load covers whole 512-byte rows).  Column reductions over rows go through shared memory.
#include "kda_common.cuh"
#include "kda_internal.h"

namespace kda {
namespace {

constexpr int TT = 8;  // tokens staged per shared-memory fill

__device__ __forceinline__ void prefetch_l2(const void *p) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}
// every 128-byte line of [p, p + bytes), spread over the CTA's threads
__device__ __forceinline__ void prefetch_span(const void *p, size_t bytes, int tid, int nt) {
  const char *c = reinterpret_cast<const char *>(p);
  for (size_t off = (size_t)tid * 128; off < bytes; off += (size_t)nt * 128) prefetch_l2(c + off);
}

template <int D, int NT, typename IO, typename ST, bool CONV, bool GATE, bool QUANT>
__global__ void __launch_bounds__(NT) recurrent_kernel(const RecArgs a) {
  constexpr int CG = D / 4;        // column groups of four
  constexpr int RG = NT / CG;      // row groups
  constexpr int RPT = D / RG;      // rows per thread
  constexpr int NW = NT / 32;
  static_assert(RG * CG == NT && RPT * RG == D, "tile split");
  static_assert(D <= NT, "one thread per value column in the reduction phase");

  __shared__ float s_q[TT][D], s_k[TT][D], s_v[TT][D], s_a[TT][D];
  __shared__ float s_beta[TT], s_rq[TT], s_rk[TT], s_kq[TT];
  __shared__ float s_redp[RG][D], s_redo[RG][D];
  __shared__ float s_u[D];
  __shared__ float s_ss[NW], s_amax[NW];

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int cg = tid % CG, rg = tid / CG;
  const int H = a.H;
  const int64_t units = (int64_t)a.n_seqs * H;
  // prefill: this CTA's (head, sequence) only; decode: units blockIdx.x + k gridDim.x
  const int64_t first = a.cu_seqlens ? (int64_t)blockIdx.y * H + blockIdx.x : blockIdx.x;
  const int64_t stride = a.cu_seqlens ? units : gridDim.x;

  for (int64_t unit = first; unit < units; unit += stride) {
    const int h = (int)(unit % H), n = (int)(unit / H);
    int64_t bos, eos;
    int slot;
    if (a.cu_seqlens) {
      bos = a.cu_seqlens[n];
      eos = a.cu_seqlens[n + 1];
      slot = n;
      if (bos < 0 || eos > a.total || eos < bos) {  // offsets outside the rows: flagged, empty
        if (tid == 0 && a.err) atomicOr(a.err, ERR_BAD_SEQLEN);
        bos = eos = 0;
      }
    } else {
      const int K = a.tokens_per_seq > 0 ? a.tokens_per_seq : 1;
      bos = (int64_t)n * K;
      eos = bos + K;
      slot = a.slot_idx ? a.slot_idx[n] : n;
      const int64_t nx = unit + stride;  // this CTA's next unit: state and inputs into L2
      if (nx < units) {
        const int hn = (int)(nx % H), nn = (int)(nx / H);
        const int sn = a.slot_idx ? a.slot_idx[nn] : nn;
        if (a.state_in && sn >= 0 && sn < a.n_slots)
          prefetch_span(reinterpret_cast<const ST *>(a.state_in) + ((size_t)sn * H + hn) * D * D,
                        sizeof(ST) * D * D, tid, NT);
        if (tid < 3) {
          const size_t C3 = (size_t)3 * H * D, ch = (size_t)tid * H * D + (size_t)hn * D;
          if (CONV && sn >= 0 && sn < a.n_slots) {
            const IO *cs = reinterpret_cast<const IO *>(a.conv_state) + (size_t)sn * 3 * C3 + ch;
            for (int r = 0; r < 3; ++r) prefetch_span(cs + r * C3, sizeof(IO) * D, 0, 1);
            prefetch_span(reinterpret_cast<const IO *>(a.x_raw) + (size_t)nn * C3 + ch,
                          sizeof(IO) * D, 0, 1);
          }
          const size_t row = ((size_t)nn * K * H + hn) * D;
          if (tid == 0) prefetch_span(a.g + row, sizeof(float) * D, 0, 1);
          if (tid == 1 && GATE) prefetch_span(reinterpret_cast<const IO *>(a.gate) + row,
                                              sizeof(IO) * D, 0, 1);
        }
      }
    }
    if (eos < bos) eos = bos;  // a decreasing offset pair processes nothing
    if (slot < 0 || slot >= a.n_slots) {  // an index outside the pool: flagged, unit skipped
      if (tid == 0 && a.err) atomicOr(a.err, ERR_BAD_INDEX);
      continue;
    }

    // ---- load this head's state tile into registers --------------------------------------
    float S[RPT][4];
    const size_t sbase = ((size_t)slot * H + h) * (size_t)D * D;
    if (a.state_in) {
      const ST *src = reinterpret_cast<const ST *>(a.state_in) + sbase;
#pragma unroll
      for (int r = 0; r < RPT; ++r) {
        const float4 x = load4_stream(src + (size_t)(rg * RPT + r) * D + 4 * cg);
        S[r][0] = x.x, S[r][1] = x.y, S[r][2] = x.z, S[r][3] = x.w;
      }
    } else {
#pragma unroll
      for (int r = 0; r < RPT; ++r) S[r][0] = S[r][1] = S[r][2] = S[r][3] = 0.f;
    }

    const IO *q = reinterpret_cast<const IO *>(a.q);
    const IO *k = reinterpret_cast<const IO *>(a.k);
    const IO *v = reinterpret_cast<const IO *>(a.v);
    // prefix-state checkpoints of this sequence (prefill only): next one and the end
    int kc = a.ckpt_cu ? a.ckpt_cu[n] : 0;
    int kend = a.ckpt_cu ? a.ckpt_cu[n + 1] : 0;
    if (kc < 0 || kend > a.n_ckpt || kend < kc) {  // a range outside the checkpoints: flagged
      if (tid == 0 && a.err) atomicOr(a.err, ERR_BAD_INDEX);
      kc = kend = 0;
    }

    for (int64_t t0 = bos; t0 < eos; t0 += TT) {
      const int nt = (int)((eos - t0) < TT ? (eos - t0) : TT);
      __syncthreads();  // staging buffers free
      if (CONV) {
        // decode: one token; q, k, v from the width-4 causal convolution of the raw inputs
        // and the conv tail, then the tail shifts by one (bit-exact copies).
        const int C = 3 * H * D;
        const IO *xr = reinterpret_cast<const IO *>(a.x_raw) + (size_t)n * C;
        const IO *cw = reinterpret_cast<const IO *>(a.conv_w);
        IO *cs = reinterpret_cast<IO *>(a.conv_state) + (size_t)slot * 3 * C;
        if (tid < D) {
#pragma unroll
          for (int st = 0; st < 3; ++st) {
            const int ch = st * H * D + h * D + tid;
            const IO x0 = cs[ch], x1 = cs[C + ch], x2 = cs[2 * C + ch], xn = xr[ch];
            const float acc = to_f(cw[4 * ch + 0]) * to_f(x0) + to_f(cw[4 * ch + 1]) * to_f(x1) +
                              to_f(cw[4 * ch + 2]) * to_f(x2) + to_f(cw[4 * ch + 3]) * to_f(xn);
            const float y = siluf_(acc);
            if (st == 0) s_q[0][tid] = y;
            else if (st == 1) s_k[0][tid] = y;
            else s_v[0][tid] = y;
            cs[ch] = x1;
            cs[C + ch] = x2;
            cs[2 * C + ch] = xn;
          }
          const size_t row = ((size_t)t0 * H + h) * D + tid;
          s_a[0][tid] = expf(fmaxf(a.g[row], a.g_min));
        }
      } else {
        for (int e = tid; e < nt * D; e += NT) {
          const int tt = e / D, i = e % D;
          const size_t row = ((size_t)(t0 + tt) * H + h) * D + i;
          s_q[tt][i] = to_f(q[row]);
          s_k[tt][i] = to_f(k[row]);
          s_v[tt][i] = to_f(v[row]);
          s_a[tt][i] = expf(fmaxf(a.g[row], a.g_min));
        }
      }
      if (tid < nt) s_beta[tid] = a.beta[(size_t)(t0 + tid) * H + h];
      __syncthreads();
      // L2 norms of q and k and their dot product, one warp per token
      for (int tt = warp; tt < nt; tt += NW) {
        float sq = 0.f, sk = 0.f, skq = 0.f;
        for (int i = lane; i < D; i += 32) {
          const float qq = s_q[tt][i], kk = s_k[tt][i];
          sq += qq * qq, sk += kk * kk, skq += qq * kk;
        }
        sq = warp_sum(sq), sk = warp_sum(sk), skq = warp_sum(skq);
        if (lane == 0) {
          const float rq = a.qk_l2norm ? rsqrtf(sq + a.l2_eps) : 1.f;
          const float rk = a.qk_l2norm ? rsqrtf(sk + a.l2_eps) : 1.f;
          s_rq[tt] = rq, s_rk[tt] = rk, s_kq[tt] = skq * rq * rk;
        }
      }
      __syncthreads();

      for (int tt = 0; tt < nt; ++tt) {
        const float rq = s_rq[tt], rk = s_rk[tt];
        float pp[4] = {0.f, 0.f, 0.f, 0.f}, po[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int r = 0; r < RPT; ++r) {
          const int i = rg * RPT + r;
          const float al = s_a[tt][i], kk = s_k[tt][i] * rk, qq = s_q[tt][i] * rq;
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            S[r][c] *= al;
            pp[c] = fmaf(S[r][c], kk, pp[c]);
            po[c] = fmaf(S[r][c], qq, po[c]);
          }
        }
#pragma unroll
        for (int c = 0; c < 4; ++c) s_redp[rg][4 * cg + c] = pp[c], s_redo[rg][4 * cg + c] = po[c];
        __syncthreads();
        float o = 0.f;
        if (tid < D) {
          float p = 0.f, o1 = 0.f;
#pragma unroll
          for (int g2 = 0; g2 < RG; ++g2) p += s_redp[g2][tid], o1 += s_redo[g2][tid];
          const float u = s_beta[tt] * (s_v[tt][tid] - p);
          s_u[tid] = u;
          o = a.scale * fmaf(u, s_kq[tt], o1);
        }
        if (GATE && warp < (D + 31) / 32) {
          const float ss = warp_sum(tid < D ? o * o : 0.f);
          if (lane == 0) s_ss[warp] = ss;
        }
        __syncthreads();
#pragma unroll
        for (int r = 0; r < RPT; ++r) {
          const float kk = s_k[tt][rg * RPT + r] * rk;
#pragma unroll
          for (int c = 0; c < 4; ++c) S[r][c] = fmaf(kk, s_u[4 * cg + c], S[r][c]);
        }
        // checkpoints placed after this token; one placed before (out of order) is flagged
        for (const int64_t done = t0 + tt + 1 - bos; kc < kend && a.ckpt_pos[kc] <= done; ++kc) {
          if (a.ckpt_pos[kc] < done) {
            if (tid == 0 && a.err) atomicOr(a.err, ERR_BAD_INDEX);
            continue;
          }
          ST *dst = reinterpret_cast<ST *>(a.ckpt_states) + ((size_t)kc * H + h) * D * D;
#pragma unroll
          for (int r = 0; r < RPT; ++r)
            store4(dst + (size_t)(rg * RPT + r) * D + 4 * cg,
                   make_float4(S[r][0], S[r][1], S[r][2], S[r][3]));
        }
        if (a.step_states) {  // the state after this token (speculative rollback points)
          ST *dst = reinterpret_cast<ST *>(a.step_states) + ((size_t)(t0 + tt) * H + h) * D * D;
#pragma unroll
          for (int r = 0; r < RPT; ++r)
            store4_stream(dst + (size_t)(rg * RPT + r) * D + 4 * cg,
                   make_float4(S[r][0], S[r][1], S[r][2], S[r][3]));
        }
        const size_t row = ((size_t)(t0 + tt) * H + h) * D + tid;
        if (tid < D) {
          if (GATE) {
            float ss = 0.f;
#pragma unroll
            for (int w = 0; w < (D + 31) / 32; ++w) ss += s_ss[w];
            const float r = rsqrtf(ss / D + a.norm_eps);
            const float w = a.norm_w ? a.norm_w[tid] : 1.f;
            const float z = to_f(reinterpret_cast<const IO *>(a.gate)[row]);
            o = o * r * w * sigmoidf_(z);
          }
          if (!QUANT) reinterpret_cast<IO *>(a.out)[row] = from_f<IO>(o);
        }
        if (QUANT) {
          // FP8 output: the group's amax over its D values (warp max, then across warps)
          const float m = warp_max(tid < D ? fabsf(o) : 0.f);
          if (lane == 0 && warp < (D + 31) / 32) s_amax[warp] = m;
          __syncthreads();
          if (tid < D) {
            float amax = 0.f;
#pragma unroll
            for (int w = 0; w < (D + 31) / 32; ++w) amax = fmaxf(amax, s_amax[w]);
            a.out_q[row] = fp8_code(o, fp8_inv_scale(amax));
            if (tid == 0) a.out_scale[(size_t)(t0 + tt) * H + h] = fp8_scale(amax);
          }
        }
      }
    }

    if (kc < kend && tid == 0 && a.err) atomicOr(a.err, ERR_BAD_INDEX);  // beyond the end
    if (a.state_out) {
      ST *dst = reinterpret_cast<ST *>(a.state_out) + sbase;
#pragma unroll
      for (int r = 0; r < RPT; ++r)
        store4_stream(dst + (size_t)(rg * RPT + r) * D + 4 * cg,
               make_float4(S[r][0], S[r][1], S[r][2], S[r][3]));
    }
  }  // units
}

// prefill: grid (H, N); decode: a persistent grid of the CTAs that fit at once, capped by the
// number of (sequence, head) units
template <typename K>
cudaError_t launch_grid(K kernel, int nt, const RecArgs &a, cudaStream_t s) {
  dim3 grid(a.H, a.n_seqs);
  if (!a.cu_seqlens) {
    int dev = 0, nsm = 0, per_sm = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, nt, 0);
    if (e != cudaSuccess) return e;
    const int64_t units = (int64_t)a.n_seqs * a.H;
    const int64_t fit = (int64_t)nsm * (per_sm > 0 ? per_sm : 1);
    grid = dim3((unsigned)(units < fit ? units : fit), 1);
  }
  kernel<<<grid, nt, 0, s>>>(a);
  return cudaGetLastError();
}

template <int D, int NT, typename IO, typename ST>
cudaError_t launch_typed(const RecArgs &a, cudaStream_t s) {
  const bool conv = a.x_raw != nullptr, gate = a.gate != nullptr;
  if (a.out_q) {  // FP8 output epilogue (its own instantiations: the bf16 path is untouched)
    if (conv && gate) return launch_grid(recurrent_kernel<D, NT, IO, ST, true, true, true>, NT, a, s);
    if (conv) return launch_grid(recurrent_kernel<D, NT, IO, ST, true, false, true>, NT, a, s);
    if (gate) return launch_grid(recurrent_kernel<D, NT, IO, ST, false, true, true>, NT, a, s);
    return launch_grid(recurrent_kernel<D, NT, IO, ST, false, false, true>, NT, a, s);
  }
  if (conv && gate) return launch_grid(recurrent_kernel<D, NT, IO, ST, true, true, false>, NT, a, s);
  if (conv) return launch_grid(recurrent_kernel<D, NT, IO, ST, true, false, false>, NT, a, s);
  if (gate) return launch_grid(recurrent_kernel<D, NT, IO, ST, false, true, false>, NT, a, s);
  return launch_grid(recurrent_kernel<D, NT, IO, ST, false, false, false>, NT, a, s);
}

template <int D, int NT>
cudaError_t launch_d(const RecArgs &a, bool io_bf16, bool st_bf16, cudaStream_t s) {
  if (io_bf16)
    return st_bf16 ? launch_typed<D, NT, bf16, bf16>(a, s) : launch_typed<D, NT, bf16, float>(a, s);
  return st_bf16 ? launch_typed<D, NT, float, bf16>(a, s) : launch_typed<D, NT, float, float>(a, s);
}

// Commit accepted speculative steps: for sequence n and head h, pool[slot(n), h] <-
// step_states[n*K + accept[n] - 1, h] when 1 <= accept[n] <= K; 0 keeps the pool state.
// Raw 16-byte copies (bit-exact).  Indices outside their range are flagged and skipped.
__global__ void state_accept_kernel(const uint4 *step, uint4 *pool, const int32_t *accept,
                                    const int32_t *slot_idx, int n_slots, int K, int H,
                                    int vec_per_head, int *err) {
  const int h = blockIdx.x, n = blockIdx.y;
  const int acc = accept[n];
  const int slot = slot_idx ? slot_idx[n] : n;
  if (acc < 0 || acc > K || slot < 0 || slot >= n_slots) {
    if (threadIdx.x == 0 && err) atomicOr(err, ERR_BAD_INDEX);
    return;
  }
  if (acc == 0) return;
  const uint4 *src = step + (((size_t)n * K + acc - 1) * H + h) * vec_per_head;
  uint4 *dst = pool + ((size_t)slot * H + h) * vec_per_head;
  for (int e = threadIdx.x; e < vec_per_head; e += blockDim.x) dst[e] = src[e];
}

}  // namespace

cudaError_t launch_state_accept(const void *step_states, void *pool, const int32_t *accept,
                                const int32_t *slot_idx, int n_slots, int n_seqs, int K, int H,
                                int D, bool st_bf16, int *err, cudaStream_t s) {
  if (n_seqs == 0) return cudaSuccess;
  const int vec = D * D * (st_bf16 ? 2 : 4) / 16;
  state_accept_kernel<<<dim3(H, n_seqs), 256, 0, s>>>(
      reinterpret_cast<const uint4 *>(step_states), reinterpret_cast<uint4 *>(pool), accept,
      slot_idx, n_slots, K, H, vec, err);
  return cudaGetLastError();
}

cudaError_t launch_recurrent(const RecArgs &a, int D, bool io_bf16, bool st_bf16,
                             cudaStream_t s) {
  if (decode_one_serves(a, D)) return launch_decode_one(a, io_bf16, st_bf16, s);
  if (D == 128) return launch_d<128, 256>(a, io_bf16, st_bf16, s);
  if (D == 16) return launch_d<16, 64>(a, io_bf16, st_bf16, s);
  return cudaErrorInvalidValue;
}

}  // namespace kda

// kda_decode.cu -- the one-token decode step at d = 128: the state of every (sequence, head)
// read from HBM once and written once, with as few block barriers as the recurrence allows.
//
// The recurrence is the token-serial one of kda_recurrent.cu ("Ling-3.1-flash: a 560B
// hybrid-attention MoE, counted from its safetensors headers", section "How KDA and MLA
// split the work", the state equation; the delta-rule write of "Ling-3.1-flash: Grouped
// Routing and Two Different MLA Caches", section "KDA replaces a token list with a recurrent
// matrix"):  S' = Diag(exp(max(g, g_min))) S;  u = beta (v - S'^T k);  S = S' + k u^T;
// o = scale (S'^T q + u (k.q)).
//
// Work layout: a persistent grid walks the (sequence, head) units, asking L2 for the next
// unit's state and inputs before working on the current one.  Warp w of the CTA owns the 16
// value columns 16 w .. 16 w + 15 of the 128 x 128 state; lane 4 rg + cq holds rows
// 16 rg .. 16 rg + 15 of columns 16 w + 4 cq .. + 3.  A value column's two reductions over
// the 128 key rows (S'^T k and S'^T q) therefore close inside its warp by shuffles, and
// u, the update and the output of a column need nothing from another warp: the only block
// barriers of a unit are the two around the staging of q, k, v and the retention (plus one
// for the output norm's sum of squares and one for the FP8 group's maximum).  Each warp
// recomputes the q, k norms from shared memory instead of waiting for one warp to.  The state
// is loaded and stored with streaming cache hints: it is touched once per step, and evicting
// it first keeps the next units' prefetched state in L2 (0.391 -> 0.362 ms per step at 256
// sequences x 64 heads).
#include "kda_common.cuh"
#include "kda_internal.h"

namespace kda {
namespace {

constexpr int DD = 128, DNT = 256;

__device__ __forceinline__ void prefetch_l2_line(const void *p) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}
__device__ __forceinline__ void prefetch_lines(const void *p, size_t bytes, int tid, int nt) {
  const char *c = reinterpret_cast<const char *>(p);
  for (size_t off = (size_t)tid * 128; off < bytes; off += (size_t)nt * 128) prefetch_l2_line(c + off);
}
__device__ __forceinline__ float dot4(float4 a, float4 b) {
  return fmaf(a.x, b.x, fmaf(a.y, b.y, fmaf(a.z, b.z, a.w * b.w)));
}

template <typename IO, typename ST, bool CONV, bool GATE, bool QUANT>
__global__ void __launch_bounds__(DNT, 2) decode_kernel(const RecArgs a) {
  __shared__ __align__(16) float s_q[DD], s_k[DD], s_v[DD], s_a[DD];
  __shared__ float s_beta;
  __shared__ float s_ss[DNT / 32], s_mx[DNT / 32];

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int cq = lane & 3, rg = lane >> 2;
  const int col = 16 * warp + 4 * cq;  // this thread's four value columns
  const int H = a.H;
  const int64_t units = (int64_t)a.n_seqs * H;

  for (int64_t unit = blockIdx.x; unit < units; unit += gridDim.x) {
    const int h = (int)(unit % H), n = (int)(unit / H);
    const int slot = a.slot_idx ? a.slot_idx[n] : n;
    {  // the next unit of this CTA: its state and inputs into L2
      const int64_t nx = unit + gridDim.x;
      if (nx < units) {
        const int hn = (int)(nx % H), nn = (int)(nx / H);
        const int sn = a.slot_idx ? a.slot_idx[nn] : nn;
        if (a.state_in && sn >= 0 && sn < a.n_slots)
          prefetch_lines(reinterpret_cast<const ST *>(a.state_in) + ((size_t)sn * H + hn) * DD * DD,
                         sizeof(ST) * DD * DD, tid, DNT);
        if (tid < 3) {
          const size_t C3 = (size_t)3 * H * DD, ch = (size_t)tid * H * DD + (size_t)hn * DD;
          if (CONV && sn >= 0 && sn < a.n_slots) {
            const IO *cs = reinterpret_cast<const IO *>(a.conv_state) + (size_t)sn * 3 * C3 + ch;
            for (int r = 0; r < 3; ++r) prefetch_lines(cs + r * C3, sizeof(IO) * DD, 0, 1);
            prefetch_lines(reinterpret_cast<const IO *>(a.x_raw) + (size_t)nn * C3 + ch,
                           sizeof(IO) * DD, 0, 1);
          }
          const size_t row = ((size_t)nn * H + hn) * DD;
          if (tid == 0) prefetch_lines(a.g + row, sizeof(float) * DD, 0, 1);
          if (tid == 1 && GATE) prefetch_lines(reinterpret_cast<const IO *>(a.gate) + row,
                                               sizeof(IO) * DD, 0, 1);
        }
      }
    }
    if (slot < 0 || slot >= a.n_slots) {  // an index outside the pool: flagged, unit skipped
      if (tid == 0 && a.err) atomicOr(a.err, ERR_BAD_INDEX);
      continue;
    }

    // ---- this thread's state: rows 16 rg .. 16 rg + 15, columns col .. col + 3 -------------
    float S[16][4];
    const size_t sbase = ((size_t)slot * H + h) * (size_t)DD * DD;
    if (a.state_in) {
      const ST *src = reinterpret_cast<const ST *>(a.state_in) + sbase + col;
#pragma unroll
      for (int r = 0; r < 16; ++r) {
        const float4 x = load4_stream(src + (size_t)(16 * rg + r) * DD);
        S[r][0] = x.x, S[r][1] = x.y, S[r][2] = x.z, S[r][3] = x.w;
      }
    } else {
#pragma unroll
      for (int r = 0; r < 16; ++r) S[r][0] = S[r][1] = S[r][2] = S[r][3] = 0.f;
    }

    // ---- staging: q, retention (threads 0-127), k, v (128-255) ---------------------------
    __syncthreads();  // the previous unit's staging has been read
    const size_t row = ((size_t)n * H + h) * DD;  // this token's [H, D] row
    {
      const int i = tid & (DD - 1);
      if (CONV) {
        // q, k, v from the width-4 causal convolution of the raw inputs and the conv tail,
        // then the tail shifts by one (bit-exact copies)
        const int C = 3 * H * DD;
        const IO *xr = reinterpret_cast<const IO *>(a.x_raw) + (size_t)n * C;
        const IO *cw = reinterpret_cast<const IO *>(a.conv_w);
        IO *cs = reinterpret_cast<IO *>(a.conv_state) + (size_t)slot * 3 * C;
        auto conv = [&](int st) {
          const int ch = st * H * DD + h * DD + i;
          const IO x0 = cs[ch], x1 = cs[C + ch], x2 = cs[2 * C + ch], xn = xr[ch];
          const float acc = to_f(cw[4 * ch + 0]) * to_f(x0) + to_f(cw[4 * ch + 1]) * to_f(x1) +
                            to_f(cw[4 * ch + 2]) * to_f(x2) + to_f(cw[4 * ch + 3]) * to_f(xn);
          cs[ch] = x1;
          cs[C + ch] = x2;
          cs[2 * C + ch] = xn;
          return siluf_(acc);
        };
        if (tid < DD) {
          s_q[i] = conv(0);
        } else {
          s_k[i] = conv(1);
          s_v[i] = conv(2);
        }
      } else {
        if (tid < DD) {
          s_q[i] = to_f(reinterpret_cast<const IO *>(a.q)[row + i]);
        } else {
          s_k[i] = to_f(reinterpret_cast<const IO *>(a.k)[row + i]);
          s_v[i] = to_f(reinterpret_cast<const IO *>(a.v)[row + i]);
        }
      }
      if (tid < DD) s_a[i] = expf(fmaxf(a.g[row + i], a.g_min));
      if (tid == DD) s_beta = a.beta[(size_t)n * H + h];
    }
    __syncthreads();

    // ---- q, k norms and k.q, in every warp (lane: channels 4 lane .. 4 lane + 3) -----------
    float rq, rk, kq;
    {
      const float4 qv = reinterpret_cast<const float4 *>(s_q)[lane];
      const float4 kv = reinterpret_cast<const float4 *>(s_k)[lane];
      const float sq = warp_sum(dot4(qv, qv)), sk = warp_sum(dot4(kv, kv));
      const float sqk = warp_sum(dot4(qv, kv));
      rq = a.qk_l2norm ? rsqrtf(sq + a.l2_eps) : 1.f;
      rk = a.qk_l2norm ? rsqrtf(sk + a.l2_eps) : 1.f;
      kq = sqk * rq * rk;
    }

    // ---- decay, the two column reductions over this thread's rows, then over the warp ----
    float kk[16], pp[4] = {0.f, 0.f, 0.f, 0.f}, po[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int r4 = 0; r4 < 4; ++r4) {
      const float4 al4 = reinterpret_cast<const float4 *>(s_a)[4 * rg + r4];
      const float4 k4 = reinterpret_cast<const float4 *>(s_k)[4 * rg + r4];
      const float4 q4 = reinterpret_cast<const float4 *>(s_q)[4 * rg + r4];
      const float al[4] = {al4.x, al4.y, al4.z, al4.w};
      const float kr[4] = {k4.x, k4.y, k4.z, k4.w}, qr[4] = {q4.x, q4.y, q4.z, q4.w};
#pragma unroll
      for (int y = 0; y < 4; ++y) {
        const int r = 4 * r4 + y;
        kk[r] = kr[y] * rk;
        const float qq = qr[y] * rq;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          S[r][c] *= al[y];
          pp[c] = fmaf(S[r][c], kk[r], pp[c]);
          po[c] = fmaf(S[r][c], qq, po[c]);
        }
      }
    }
#pragma unroll
    for (int off = 4; off < 32; off <<= 1)  // the eight row groups of these columns
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        pp[c] += __shfl_xor_sync(0xffffffffu, pp[c], off);
        po[c] += __shfl_xor_sync(0xffffffffu, po[c], off);
      }

    // ---- the corrected write, the update and the read ------------------------------------
    const float4 v4 = reinterpret_cast<const float4 *>(s_v)[col >> 2];
    const float vv[4] = {v4.x, v4.y, v4.z, v4.w};
    const float beta = s_beta;
    float u[4], o[4];
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      u[c] = beta * (vv[c] - pp[c]);
      o[c] = a.scale * fmaf(u[c], kq, po[c]);
    }
#pragma unroll
    for (int r = 0; r < 16; ++r)
#pragma unroll
      for (int c = 0; c < 4; ++c) S[r][c] = fmaf(kk[r], u[c], S[r][c]);

    // ---- output: optional RMSNorm x w x sigmoid(gate), optional FP8 codes -----------------
    if (GATE) {
      float ss = o[0] * o[0] + o[1] * o[1] + o[2] * o[2] + o[3] * o[3];
      ss += __shfl_xor_sync(0xffffffffu, ss, 1);
      ss += __shfl_xor_sync(0xffffffffu, ss, 2);
      if (lane == 0) s_ss[warp] = ss;  // the warp's 16 columns
      __syncthreads();
      float tot = 0.f;
#pragma unroll
      for (int w = 0; w < DNT / 32; ++w) tot += s_ss[w];
      const float rn = rsqrtf(tot / DD + a.norm_eps);
      const float4 gl = load4(reinterpret_cast<const IO *>(a.gate) + row + col);
      const float gz[4] = {gl.x, gl.y, gl.z, gl.w};
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const float w = a.norm_w ? a.norm_w[col + c] : 1.f;
        o[c] = o[c] * rn * w * sigmoidf_(gz[c]);
      }
    }
    if (QUANT) {
      float m = fmaxf(fmaxf(fabsf(o[0]), fabsf(o[1])), fmaxf(fabsf(o[2]), fabsf(o[3])));
      m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
      m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
      if (lane == 0) s_mx[warp] = m;
      __syncthreads();
      float amax = 0.f;
#pragma unroll
      for (int w = 0; w < DNT / 32; ++w) amax = fmaxf(amax, s_mx[w]);
      if (rg == 0) {
        const float inv = fp8_inv_scale(amax);
        const uint32_t code = (uint32_t)fp8_code(o[0], inv) | ((uint32_t)fp8_code(o[1], inv) << 8) |
                              ((uint32_t)fp8_code(o[2], inv) << 16) |
                              ((uint32_t)fp8_code(o[3], inv) << 24);
        *reinterpret_cast<uint32_t *>(a.out_q + row + col) = code;
      }
      if (tid == 0) a.out_scale[(size_t)n * H + h] = fp8_scale(amax);
    } else if (rg == 0) {
      store4(reinterpret_cast<IO *>(a.out) + row + col, make_float4(o[0], o[1], o[2], o[3]));
    }

    if (a.state_out) {
      ST *dst = reinterpret_cast<ST *>(a.state_out) + sbase + col;
#pragma unroll
      for (int r = 0; r < 16; ++r)
        store4_stream(dst + (size_t)(16 * rg + r) * DD, make_float4(S[r][0], S[r][1], S[r][2], S[r][3]));
    }
  }  // units
}

template <typename IO, typename ST, bool CONV, bool GATE, bool QUANT>
cudaError_t launch_one(const RecArgs &a, cudaStream_t s) {
  auto kernel = decode_kernel<IO, ST, CONV, GATE, QUANT>;
  int dev = 0, nsm = 0, per_sm = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
  if (e == cudaSuccess) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, DNT, 0);
  if (e != cudaSuccess) return e;
  const int64_t units = (int64_t)a.n_seqs * a.H;
  const int64_t fit = (int64_t)nsm * (per_sm > 0 ? per_sm : 1);
  kernel<<<(unsigned)(units < fit ? units : fit), DNT, 0, s>>>(a);
  return cudaGetLastError();
}

template <typename IO, typename ST>
cudaError_t launch_typed(const RecArgs &a, cudaStream_t s) {
  const bool conv = a.x_raw != nullptr, gate = a.gate != nullptr;
  if (a.out_q) {
    if (conv && gate) return launch_one<IO, ST, true, true, true>(a, s);
    if (conv) return launch_one<IO, ST, true, false, true>(a, s);
    if (gate) return launch_one<IO, ST, false, true, true>(a, s);
    return launch_one<IO, ST, false, false, true>(a, s);
  }
  if (conv && gate) return launch_one<IO, ST, true, true, false>(a, s);
  if (conv) return launch_one<IO, ST, true, false, false>(a, s);
  if (gate) return launch_one<IO, ST, false, true, false>(a, s);
  return launch_one<IO, ST, false, false, false>(a, s);
}

}  // namespace

bool decode_one_serves(const RecArgs &a, int D) {
  return D == DD && !a.cu_seqlens && a.tokens_per_seq <= 1 && !a.step_states && !a.ckpt_cu;
}

cudaError_t launch_decode_one(const RecArgs &a, bool io_bf16, bool st_bf16, cudaStream_t s) {
  if (a.n_seqs == 0) return cudaSuccess;
  if (io_bf16)
    return st_bf16 ? launch_typed<bf16, bf16>(a, s) : launch_typed<bf16, float>(a, s);
  return st_bf16 ? launch_typed<float, bf16>(a, s) : launch_typed<float, float>(a, s);
}

}  // namespace kda

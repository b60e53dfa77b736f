// kda_host_stream.cu -- kda_prefill_host: the prefill hot path (kda_prologue, then kda_prefill)
// for a packed batch held in host memory, streamed through the GPU in token segments so that
// the copies in, the kernels and the copies out of neighbouring segments overlap.
//
// Serving engines already cut a long prompt's prefill into pieces and carry the recurrent
// state from one piece to the next (a chunked-prefill size of 4096 tokens next to the
// recurrent-state cache settings, "Ling-3.1-flash: What 63 Linear-Attention Layers Do to the
// KV Budget", section "Where the hybrid makes serving harder"): the state summarises every
// token before it, so running T1 + T2 tokens equals running T2 from the state that T1 left.
// Here every inner segment boundary falls on a chunk edge of the sequence it cuts (a multiple
// of 64 tokens from that sequence's start), so each sequence is chunked exactly as one
// kda_prefill over the whole batch chunks it and the results are the same bits.  The fp32
// state and the conv tail of a cut sequence wait in device memory for the next segment.
//
// Streams: the caller's stream runs the kernels; two copy streams bring the inputs in (the raw
// projections on one; the log-retention, write-strength logits and gate logits on the other,
// so that two copy engines can work at once) and a third takes the outputs back.  The segment
// buffers are double-buffered in the caller's workspace, and events order each buffer's reuse.
#include "../../include/kda.h"

#include <cstdint>
#include <cstring>
#include <mutex>

#include "kda_trace.h"

namespace kda {
kda_status validate_params(const kda_params *p);
void note_launches(int n);
}  // namespace kda

namespace {

constexpr int kMaxDevices = 64;
constexpr int kChunk = 64;
constexpr int64_t kMaxSegment = (int64_t)1 << 24;

// One table of a segment's sequence offsets, passed by value as a kernel parameter (8 KB,
// within the 32 KB parameter space), so no pageable host copy (and its implicit
// synchronisation) is needed to get it onto the device.
constexpr int kFill = 2048;
struct FillTable {
  int32_t v[kFill];
};

__global__ void fill_i32_kernel(const FillTable t, int n, int32_t *dst) {
  for (int i = threadIdx.x; i < n; i += blockDim.x) dst[i] = t.v[i];
}

// Per-device copy streams and events, created on first use and kept until the process exits.
struct Pipe {
  bool ready = false;
  cudaStream_t in_x = nullptr, in_g = nullptr, out = nullptr;
  cudaEvent_t start = nullptr, end = nullptr, carry_in = nullptr;
  cudaEvent_t in_x_done[2] = {}, in_g_done[2] = {}, used[2] = {}, out_free[2] = {};
  std::mutex mu;  // one enqueue at a time per device: the events are shared
};
Pipe g_pipe[kMaxDevices];
std::mutex g_pipe_init;

Pipe *pipe_for(int dev) {
  if (dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lk(g_pipe_init);
  Pipe &pp = g_pipe[dev];
  if (pp.ready) return &pp;
  auto ev = [](cudaEvent_t *e) {
    return cudaEventCreateWithFlags(e, cudaEventDisableTiming) == cudaSuccess;
  };
  bool ok = cudaStreamCreateWithFlags(&pp.in_x, cudaStreamNonBlocking) == cudaSuccess &&
            cudaStreamCreateWithFlags(&pp.in_g, cudaStreamNonBlocking) == cudaSuccess &&
            cudaStreamCreateWithFlags(&pp.out, cudaStreamNonBlocking) == cudaSuccess &&
            ev(&pp.start) && ev(&pp.end) && ev(&pp.carry_in);
  for (int s = 0; s < 2 && ok; ++s)
    ok = ev(&pp.in_x_done[s]) && ev(&pp.in_g_done[s]) && ev(&pp.used[s]) && ev(&pp.out_free[s]);
  if (!ok) return nullptr;
  pp.ready = true;
  return &pp;
}

size_t up256(size_t b) { return (b + 255) & ~(size_t)255; }

// Workspace map: per slot (two) the segment's raw projections, log-retention, write-strength
// logits, gate logits and output; once the convolved q, k, v, beta and the offsets table; the
// carried states and conv tails of every sequence.
struct Layout {
  size_t x[2], g[2], bl[2], gate[2], out[2], q, k, v, beta, cu, state, conv, total;
};

Layout layout(const kda_params *p, int n_seqs, int64_t S, bool with_gate) {
  const size_t e = p->io_dtype == KDA_BF16 ? 2 : 4, H = (size_t)p->H, d = (size_t)p->d_k;
  const size_t rows = (size_t)S;
  const size_t xb = up256(rows * 3 * H * d * e), gb = up256(rows * H * d * 4),
               blb = up256(rows * H * 4), gateb = with_gate ? up256(rows * H * d * e) : 0,
               outb = up256(rows * H * d * e);
  Layout L;
  size_t o = 0;
  for (int s = 0; s < 2; ++s) {
    L.x[s] = o, o += xb;
    L.g[s] = o, o += gb;
    L.bl[s] = o, o += blb;
    L.gate[s] = o, o += gateb;
    L.out[s] = o, o += outb;
  }
  L.q = o, o += outb;
  L.k = o, o += outb;
  L.v = o, o += outb;
  L.beta = o, o += blb;
  L.cu = o, o += up256(((size_t)n_seqs + 1) * 4);
  L.state = o, o += up256((size_t)n_seqs * H * d * d * 4);
  L.conv = o, o += up256((size_t)n_seqs * 3 * 3 * H * d * e);
  L.total = o;
  return L;
}

// A segment: packed rows [r0, r1), sequences n_a .. n_a + count - 1 (those it cuts, with any
// empty ones between them).
struct Seg {
  int64_t r0, r1;
  int n_a, count;
};

// the sequence n with cu[n] <= r < cu[n + 1] (cu non-decreasing, cu[0] = 0 <= r < cu[n_seqs])
int seq_containing(const int32_t *cu, int n_seqs, int64_t r) {
  int lo = 0, hi = n_seqs;  // answer in [lo, hi): the last n with cu[n] <= r
  while (hi - lo > 1) {
    const int mid = (lo + hi) / 2;
    if ((int64_t)cu[mid] <= r) lo = mid;
    else hi = mid;
  }
  return lo;  // the last such n: cu[n + 1] > r, so sequence n is not empty
}

// Cuts [0, T) into segments of at most S rows whose inner boundaries lie on the chunk grid of
// the sequence they fall in, one segment per call of next() (nothing is stored: a long batch
// cut into short segments costs no host memory).  The last 2S rows are cut in halves (S,
// S/2, ..., 64 rows), so that little of the work is left once the last inputs have arrived:
// the kernels and the copy-out of the last segment are all that does not overlap the copies
// in.
struct Planner {
  const int32_t *cu;
  int n_seqs;
  int64_t T, S, r0 = 0;

  bool next(Seg *sg) {
    if (r0 >= T) return false;
    int64_t want = S;  // a multiple of the chunk, at least one chunk
    if (T - r0 <= 2 * S) {
      want = (T - r0) / 2 / kChunk * kChunk;
      if (want < kChunk) want = kChunk;
    }
    int64_t r1 = r0 + want;
    if (r1 >= T) {
      r1 = T;
    } else {
      const int n = seq_containing(cu, n_seqs, r1);
      // down to the chunk grid of sequence n.  Still > r0: if n also holds r0, r0 is on its
      // grid (a sequence start or an earlier boundary) and `want` is a multiple of the chunk,
      // so nothing is cut; otherwise r1 >= cu[n] > r0.
      r1 = cu[n] + (r1 - cu[n]) / kChunk * kChunk;
    }
    const int a = seq_containing(cu, n_seqs, r0), b = seq_containing(cu, n_seqs, r1 - 1);
    *sg = Seg{r0, r1, a, b - a + 1};
    r0 = r1;
    return true;
  }
};

bool aligned(const void *ptr, uintptr_t a) {
  return (reinterpret_cast<uintptr_t>(ptr) & (a - 1)) == 0;
}

}  // namespace

extern "C" {

size_t kda_prefill_host_workspace_size(const kda_params *p, int n_seqs, int64_t segment_tokens,
                                       int with_gate) {
  if (kda::validate_params(p) != KDA_OK || n_seqs < 1 || n_seqs > 65535 ||
      segment_tokens < kChunk || segment_tokens % kChunk != 0 || segment_tokens > kMaxSegment)
    return 0;
  return layout(p, n_seqs, segment_tokens, with_gate != 0).total;
}

int64_t kda_prefill_host_plan(const int32_t *cu_seqlens, int n_seqs, int64_t total_tokens,
                              int64_t segment_tokens, int64_t *bounds, int64_t max_segments) {
  if (!cu_seqlens || n_seqs < 1 || n_seqs > 65535 || total_tokens < 0 ||
      total_tokens > INT32_MAX || segment_tokens < kChunk || segment_tokens % kChunk != 0 ||
      segment_tokens > kMaxSegment || max_segments < 0 || (max_segments > 0 && !bounds))
    return -1;
  if (cu_seqlens[0] != 0 || (int64_t)cu_seqlens[n_seqs] != total_tokens) return -1;
  for (int n = 0; n < n_seqs; ++n)
    if (cu_seqlens[n + 1] < cu_seqlens[n]) return -1;
  Planner planner{cu_seqlens, n_seqs, total_tokens, segment_tokens};
  Seg sg;
  int64_t k = 0;
  if (max_segments > 0) bounds[0] = 0;
  while (planner.next(&sg)) {
    ++k;
    if (k <= max_segments) bounds[k] = sg.r1;
  }
  return k;
}

kda_status kda_prefill_host(const kda_params *p, const void *x_raw, const void *conv_w,
                            void *conv_state, const int32_t *cu_seqlens, int n_seqs,
                            int64_t total_tokens, const float *beta_logit, const float *g_raw,
                            const void *init_state, const void *gate_logit,
                            const float *norm_w, void *out, void *final_state, void *workspace,
                            size_t ws_bytes, int64_t segment_tokens, cudaStream_t stream) {
  KDA_TRACE(TR_PREFILL_HOST);
  // ---- host-side checks, before any CUDA call
  kda_status st = kda::validate_params(p);
  if (st != KDA_OK) return st;
  if (p->state_dtype != KDA_F32) return KDA_ERR_UNSUPPORTED;
  if (n_seqs < 1 || n_seqs > 65535 || total_tokens < 0) return KDA_ERR_INVALID_ARG;
  if (total_tokens > INT32_MAX) return KDA_ERR_UNSUPPORTED;
  if (segment_tokens < kChunk || segment_tokens % kChunk != 0 || segment_tokens > kMaxSegment)
    return KDA_ERR_INVALID_ARG;
  if (!cu_seqlens || !conv_w) return KDA_ERR_INVALID_ARG;
  if (total_tokens > 0 && (!x_raw || !beta_logit || !g_raw || !out)) return KDA_ERR_INVALID_ARG;
  if (cu_seqlens[0] != 0 || (int64_t)cu_seqlens[n_seqs] != total_tokens) return KDA_ERR_INVALID_ARG;
  for (int n = 0; n < n_seqs; ++n)
    if (cu_seqlens[n + 1] < cu_seqlens[n]) return KDA_ERR_INVALID_ARG;
  if (!aligned(conv_w, 16) || !aligned(norm_w, 16)) return KDA_ERR_INVALID_ARG;
  const bool with_gate = gate_logit != nullptr;
  const Layout L = layout(p, n_seqs, segment_tokens, with_gate);
  if (ws_bytes < L.total) return KDA_ERR_WORKSPACE;
  if (!workspace || !aligned(workspace, 256)) return KDA_ERR_INVALID_ARG;

  const size_t e = p->io_dtype == KDA_BF16 ? 2 : 4, H = (size_t)p->H, d = (size_t)p->d_k;
  const size_t x_row = 3 * H * d * e, g_row = H * d * 4, bl_row = H * 4, o_row = H * d * e;
  const size_t st_seq = H * d * d * 4, conv_seq = 3 * 3 * H * d * e;
  Planner planner{cu_seqlens, n_seqs, total_tokens, segment_tokens};

  // ---- enqueue
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return KDA_ERR_CUDA;
  Pipe *pp = pipe_for(dev);
  if (!pp) return KDA_ERR_CUDA;
  std::lock_guard<std::mutex> lk(pp->mu);
  uint8_t *ws = static_cast<uint8_t *>(workspace);
  const uint8_t *hx = static_cast<const uint8_t *>(x_raw);
  const uint8_t *hg = reinterpret_cast<const uint8_t *>(g_raw);
  const uint8_t *hbl = reinterpret_cast<const uint8_t *>(beta_logit);
  const uint8_t *hgate = static_cast<const uint8_t *>(gate_logit);
  uint8_t *hout = static_cast<uint8_t *>(out);
  bool ok = true;
  auto chk = [&](cudaError_t r) { ok = ok && r == cudaSuccess; };
  auto h2d = [&](void *dst, const void *src, size_t n, cudaStream_t s) {
    if (n) chk(cudaMemcpyAsync(dst, src, n, cudaMemcpyHostToDevice, s));
  };

  // every copy stream starts after the caller's earlier work on its stream (and hence after
  // the previous call of this function on it, which ends by making that stream wait)
  chk(cudaEventRecord(pp->start, stream));
  chk(cudaStreamWaitEvent(pp->in_x, pp->start, 0));
  chk(cudaStreamWaitEvent(pp->in_g, pp->start, 0));
  chk(cudaStreamWaitEvent(pp->out, pp->start, 0));
  // the carried states and conv tails start as the caller's (or zeros)
  if (init_state) h2d(ws + L.state, init_state, (size_t)n_seqs * st_seq, pp->in_g);
  else chk(cudaMemsetAsync(ws + L.state, 0, (size_t)n_seqs * st_seq, pp->in_g));
  if (conv_state) h2d(ws + L.conv, conv_state, (size_t)n_seqs * conv_seq, pp->in_g);
  else chk(cudaMemsetAsync(ws + L.conv, 0, (size_t)n_seqs * conv_seq, pp->in_g));
  chk(cudaEventRecord(pp->carry_in, pp->in_g));

  int fills = 0;
  kda_status fail = KDA_OK;  // a launch that failed part-way
  Seg sg;
  for (int64_t i = 0; ok && fail == KDA_OK && planner.next(&sg); ++i) {
    const int s = (int)(i & 1);
    const size_t rows = (size_t)(sg.r1 - sg.r0), r0 = (size_t)sg.r0;
    // inputs of segment i into slot s, once segment i - 2 has used that slot
    if (i >= 2) {
      chk(cudaStreamWaitEvent(pp->in_x, pp->used[s], 0));
      chk(cudaStreamWaitEvent(pp->in_g, pp->used[s], 0));
    }
    h2d(ws + L.x[s], hx + r0 * x_row, rows * x_row, pp->in_x);
    chk(cudaEventRecord(pp->in_x_done[s], pp->in_x));
    h2d(ws + L.g[s], hg + r0 * g_row, rows * g_row, pp->in_g);
    h2d(ws + L.bl[s], hbl + r0 * bl_row, rows * bl_row, pp->in_g);
    if (with_gate) h2d(ws + L.gate[s], hgate + r0 * o_row, rows * o_row, pp->in_g);
    chk(cudaEventRecord(pp->in_g_done[s], pp->in_g));

    // this segment's sequence offsets: the cut sequences' offsets clamped to [r0, r1)
    int32_t *cu_dev = reinterpret_cast<int32_t *>(ws + L.cu);
    for (int base = 0; base <= sg.count && ok; base += kFill) {
      FillTable t{};
      const int n = sg.count + 1 - base < kFill ? sg.count + 1 - base : kFill;
      for (int j = 0; j < n; ++j) {
        int64_t c = cu_seqlens[sg.n_a + base + j];
        c = c < sg.r0 ? sg.r0 : (c > sg.r1 ? sg.r1 : c);
        t.v[j] = (int32_t)(c - sg.r0);
      }
      fill_i32_kernel<<<1, 256, 0, stream>>>(t, n, cu_dev + base);
      chk(cudaGetLastError());
      ++fills;
    }
    chk(cudaStreamWaitEvent(stream, pp->in_x_done[s], 0));
    chk(cudaStreamWaitEvent(stream, pp->in_g_done[s], 0));
    if (!ok) break;
    uint8_t *conv_c = ws + L.conv + (size_t)sg.n_a * conv_seq;
    uint8_t *state_c = ws + L.state + (size_t)sg.n_a * st_seq;
    st = kda_prologue(p, ws + L.x[s], conv_w, conv_c, cu_dev, sg.count, (int64_t)rows, 0,
                      reinterpret_cast<const float *>(ws + L.bl[s]), nullptr, ws + L.q,
                      ws + L.k, ws + L.v, reinterpret_cast<float *>(ws + L.beta), nullptr,
                      stream);
    if (st != KDA_OK) {
      fail = st;
      break;
    }
    if (i >= 2) chk(cudaStreamWaitEvent(stream, pp->out_free[s], 0));  // output slot copied out
    st = kda_prefill(p, ws + L.q, ws + L.k, ws + L.v,
                     reinterpret_cast<const float *>(ws + L.g[s]),
                     reinterpret_cast<const float *>(ws + L.beta), state_c, cu_dev, sg.count,
                     (int64_t)rows, with_gate ? ws + L.gate[s] : nullptr, norm_w, ws + L.out[s],
                     state_c, nullptr, 0, stream);
    if (st != KDA_OK) {
      fail = st;
      break;
    }
    chk(cudaEventRecord(pp->used[s], stream));

    // outputs of segment i back to the host
    chk(cudaStreamWaitEvent(pp->out, pp->used[s], 0));
    chk(cudaMemcpyAsync(hout + r0 * o_row, ws + L.out[s], rows * o_row, cudaMemcpyDeviceToHost,
                        pp->out));
    chk(cudaEventRecord(pp->out_free[s], pp->out));
  }
  kda::note_launches(fills);
  if (!ok || fail != KDA_OK) {
    // nothing more is enqueued, but `stream` still waits for the copies already on their way,
    // so that none of them runs on once the caller has synchronised it
    cudaEventRecord(pp->in_x_done[0], pp->in_x);
    cudaEventRecord(pp->in_g_done[0], pp->in_g);
    cudaEventRecord(pp->end, pp->out);
    cudaStreamWaitEvent(stream, pp->in_x_done[0], 0);
    cudaStreamWaitEvent(stream, pp->in_g_done[0], 0);
    cudaStreamWaitEvent(stream, pp->end, 0);
    return fail != KDA_OK ? fail : KDA_ERR_CUDA;
  }
  // final states and conv tails (after the last segment's kernels, which the output stream
  // has waited for; with no tokens, after the carries came in)
  chk(cudaStreamWaitEvent(pp->out, pp->carry_in, 0));
  if (final_state)
    chk(cudaMemcpyAsync(final_state, ws + L.state, (size_t)n_seqs * st_seq,
                        cudaMemcpyDeviceToHost, pp->out));
  if (conv_state)
    chk(cudaMemcpyAsync(conv_state, ws + L.conv, (size_t)n_seqs * conv_seq,
                        cudaMemcpyDeviceToHost, pp->out));
  chk(cudaEventRecord(pp->end, pp->out));
  chk(cudaStreamWaitEvent(stream, pp->end, 0));
  return ok ? KDA_OK : KDA_ERR_CUDA;
}

}  // extern "C"

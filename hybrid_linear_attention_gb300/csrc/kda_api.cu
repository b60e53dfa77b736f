// kda_api.cu -- the C ABI (include/kda.h): host-side validation, then kernel launches.
// Nothing here allocates device memory; every buffer belongs to the caller.
#include "../../include/kda.h"
#include "../../include/mla.h"

#include <atomic>
#include <cstdint>
#include <cstring>

#include "kda_internal.h"
#include "kda_prefill_tc.h"
#include "kda_trace.h"

namespace kda {
const char *const kTraceNames[TR_COUNT] = {
    "kda_prologue", "kda_prefill", "kda_prefill_fp8", "kda_prefill_checkpointed",
    "kda_conv_tail_checkpoints", "kda_decode_step", "kda_decode_step_fused",
    "kda_decode_step_fused_fp8", "kda_conv_state_update", "kda_decode_multi", "kda_state_accept",
    "kda_prefill_host", "mla_decode_latent", "mla_decode_latent_noalloc", "mla_decode",
    "kda_check_device_error", "kda_wait_probe"};
}  // namespace kda

namespace {

std::atomic<uint64_t> g_launches{0};

// Sticky error word written by kernels whose bounded waits ran out.
__device__ int g_device_error = 0;

constexpr int kMaxDevices = 64;
int *g_err_ptr[kMaxDevices] = {nullptr};

int *device_error_ptr() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  if (!g_err_ptr[dev]) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_device_error) != cudaSuccess) return nullptr;
    g_err_ptr[dev] = static_cast<int *>(p);
  }
  return g_err_ptr[dev];
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool opt_aligned16(const void *p) { return p == nullptr || aligned16(p); }

kda_status check_params(const kda_params *p) {
  if (!p) return KDA_ERR_INVALID_ARG;
  if (p->H < 1 || p->d_k < 1 || p->d_v < 1) return KDA_ERR_INVALID_ARG;
  if (!(p->l2_eps >= 0.f) || !(p->norm_eps >= 0.f)) return KDA_ERR_INVALID_ARG;
  if (!(p->g_min <= 0.f)) return KDA_ERR_INVALID_ARG;  // also rejects NaN
  if (p->scale != p->scale) return KDA_ERR_INVALID_ARG;
  if ((p->io_dtype != KDA_F32 && p->io_dtype != KDA_BF16) ||
      (p->state_dtype != KDA_F32 && p->state_dtype != KDA_BF16))
    return KDA_ERR_INVALID_ARG;
  if (p->prefill_form < KDA_PREFILL_AUTO || p->prefill_form > KDA_PREFILL_PAIR)
    return KDA_ERR_INVALID_ARG;
  if (p->d_k != p->d_v) return KDA_ERR_UNSUPPORTED;
  if (p->d_k != 16 && p->d_k != 128) return KDA_ERR_UNSUPPORTED;
  if (p->H > 21845) return KDA_ERR_UNSUPPORTED;  // 3*H grid rows of the prologue
  return KDA_OK;
}

kda_status finish(cudaError_t e, int n_launches) {
  g_launches += (uint64_t)n_launches;
  return e == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

kda::RecArgs base_args(const kda_params *p) {
  kda::RecArgs a;
  std::memset(&a, 0, sizeof a);
  a.H = p->H;
  a.scale = p->scale;
  a.l2_eps = p->l2_eps;
  a.norm_eps = p->norm_eps;
  a.g_min = p->g_min;
  a.qk_l2norm = p->qk_l2norm ? 1 : 0;
  a.err = device_error_ptr();
  return a;
}

}  // namespace

namespace kda {
// for the other host-side entry points of the library (kda_host_stream.cu)
kda_status validate_params(const kda_params *p) { return check_params(p); }
void note_launches(int n) { g_launches += (uint64_t)n; }
}  // namespace kda

extern "C" {

void kda_params_default(kda_params *p) {
  if (!p) return;
  p->H = 64;
  p->d_k = p->d_v = 128;
  p->scale = 1.0f;
  p->l2_eps = 1e-6f;
  p->norm_eps = 1e-6f;
  p->g_min = -5.0f;
  p->qk_l2norm = 1;
  p->io_dtype = KDA_BF16;
  p->state_dtype = KDA_F32;
  p->prefill_form = KDA_PREFILL_AUTO;
}

const char *kda_status_string(kda_status s) {
  switch (s) {
    case KDA_OK: return "KDA_OK";
    case KDA_ERR_INVALID_ARG: return "KDA_ERR_INVALID_ARG: invalid argument";
    case KDA_ERR_UNSUPPORTED: return "KDA_ERR_UNSUPPORTED: shape or dtype not supported";
    case KDA_ERR_CUDA: return "KDA_ERR_CUDA: CUDA launch or runtime error";
    case KDA_ERR_WORKSPACE: return "KDA_ERR_WORKSPACE: workspace too small";
    case KDA_ERR_TIMEOUT: return "KDA_ERR_TIMEOUT: a bounded device wait ran out";
    case KDA_ERR_BAD_INDEX: return "KDA_ERR_BAD_INDEX: a device-side index was out of range";
    case KDA_ERR_BAD_SEQLENS:
      return "KDA_ERR_BAD_SEQLENS: device-side sequence offsets outside the token rows";
  }
  return "unknown kda_status";
}

size_t kda_state_bytes(const kda_params *p) {
  if (!p || p->H < 1 || p->d_k < 1 || p->d_v < 1) return 0;
  return (size_t)p->H * p->d_k * p->d_v * (p->state_dtype == KDA_BF16 ? 2 : 4);
}

size_t kda_prefill_workspace_size(const kda_params *p, int n_seqs, int64_t total_tokens) {
  (void)n_seqs;
  (void)total_tokens;
  if (check_params(p) != KDA_OK) return 0;
  return 0;
}

kda_status kda_prologue(const kda_params *p, const void *x_raw, const void *conv_w,
                        void *conv_state, const int32_t *cu_seqlens, int n_seqs,
                        int64_t total_tokens, int l2norm_qk, const float *beta_logit,
                        const float *g_raw, void *q, void *k, void *v, float *beta, float *g,
                        cudaStream_t stream) {
  KDA_TRACE(TR_PROLOGUE);
  kda_status st = check_params(p);
  if (st != KDA_OK) return st;
  if (n_seqs < 0 || total_tokens < 0 || n_seqs > 65535) return KDA_ERR_INVALID_ARG;
  if (n_seqs == 0 && total_tokens > 0) return KDA_ERR_INVALID_ARG;
  if (total_tokens > (int64_t)INT32_MAX * 16) return KDA_ERR_UNSUPPORTED;  // prologue grid
  if (n_seqs == 0) return KDA_OK;
  if (!x_raw || !conv_w || !cu_seqlens || !q || !k || !v) return KDA_ERR_INVALID_ARG;
  if ((beta_logit == nullptr) != (beta == nullptr)) return KDA_ERR_INVALID_ARG;
  if ((g_raw == nullptr) != (g == nullptr)) return KDA_ERR_INVALID_ARG;
  if (!aligned16(x_raw) || !aligned16(conv_w) || !opt_aligned16(conv_state) || !aligned16(q) ||
      !aligned16(k) || !aligned16(v) || !opt_aligned16(beta_logit) || !opt_aligned16(g_raw) ||
      !opt_aligned16(beta) || !opt_aligned16(g) || !aligned16(cu_seqlens))
    return KDA_ERR_INVALID_ARG;
  kda::ProArgs a;
  std::memset(&a, 0, sizeof a);
  a.H = p->H;
  a.n_seqs = n_seqs;
  a.T = total_tokens;
  a.l2_eps = p->l2_eps;
  a.g_min = p->g_min;
  a.l2norm_qk = l2norm_qk ? 1 : 0;
  a.x = x_raw;
  a.conv_w = conv_w;
  a.conv_state = conv_state;
  a.cu_seqlens = cu_seqlens;
  a.beta_logit = beta_logit;
  a.g_raw = g_raw;
  a.q = q, a.k = k, a.v = v;
  a.beta = beta, a.g = g;
  a.err = device_error_ptr();
  const int n_launch = (total_tokens > 0 ? 1 : 0) + (conv_state ? 1 : 0);
  return finish(kda::launch_prologue(a, p->d_k, p->io_dtype == KDA_BF16, stream), n_launch);
}

static kda_status prefill_impl(const kda_params *p, const void *q, const void *k, const void *v,
                               const float *g, const float *beta, const void *init_state,
                               const int32_t *cu_seqlens, int n_seqs, int64_t total_tokens,
                               const void *gate_logit, const float *norm_w, void *out,
                               uint8_t *out_q, float *out_scale, void *final_state,
                               const int32_t *ckpt_cu, const int32_t *ckpt_pos, int n_ckpt,
                               void *ckpt_states, void *workspace, size_t ws_bytes,
                               cudaStream_t stream) {
  kda_status st = check_params(p);
  if (st != KDA_OK) return st;
  if (n_seqs < 0 || total_tokens < 0 || n_seqs > 65535) return KDA_ERR_INVALID_ARG;
  if (n_seqs == 0 && total_tokens > 0) return KDA_ERR_INVALID_ARG;
  if (ws_bytes < kda_prefill_workspace_size(p, n_seqs, total_tokens)) return KDA_ERR_WORKSPACE;
  (void)workspace;
  if (n_seqs == 0) return KDA_OK;
  if (!cu_seqlens) return KDA_ERR_INVALID_ARG;
  if (total_tokens > 0 && (!q || !k || !v || !g || !beta || !(out_q ? out_scale : out)))
    return KDA_ERR_INVALID_ARG;
  if (total_tokens > 0 && out_q && (!aligned16(out_q) || !aligned16(out_scale)))
    return KDA_ERR_INVALID_ARG;
  if (!opt_aligned16(q) || !opt_aligned16(k) || !opt_aligned16(v) || !opt_aligned16(g) ||
      !opt_aligned16(beta) || !opt_aligned16(init_state) || !aligned16(cu_seqlens) ||
      !opt_aligned16(gate_logit) || !opt_aligned16(norm_w) || !opt_aligned16(out) ||
      !opt_aligned16(final_state))
    return KDA_ERR_INVALID_ARG;
  if (n_ckpt < 0) return KDA_ERR_INVALID_ARG;
  if (n_ckpt > 0 && (!ckpt_cu || !ckpt_pos || !ckpt_states || !aligned16(ckpt_states) ||
                     !aligned16(ckpt_cu) || !aligned16(ckpt_pos)))
    return KDA_ERR_INVALID_ARG;
  if (n_ckpt == 0) ckpt_cu = nullptr;

  const bool io_bf16 = p->io_dtype == KDA_BF16, st_bf16 = p->state_dtype == KDA_BF16;
  if (kda::prefill_tc_supported(p->d_k, io_bf16)) {
    kda::TcArgs t;
    std::memset(&t, 0, sizeof t);
    t.H = p->H;
    t.n_seqs = n_seqs;
    t.scale = p->scale;
    t.l2_eps = p->l2_eps;
    t.norm_eps = p->norm_eps;
    t.g_min = p->g_min;
    t.qk_l2norm = p->qk_l2norm ? 1 : 0;
    t.q = q, t.k = k, t.v = v, t.g = g, t.beta = beta;
    t.init_state = init_state;
    t.final_state = final_state;
    t.cu_seqlens = cu_seqlens;
    t.gate = gate_logit;
    t.norm_w = norm_w;
    t.out = out;
    t.ckpt_cu = ckpt_cu, t.ckpt_pos = ckpt_pos, t.ckpt_states = ckpt_states;
    t.out_q = out_q, t.out_scale = out_scale;
    t.total = total_tokens, t.n_ckpt = n_ckpt;
    t.err = device_error_ptr();
    t.form = p->prefill_form;
    return finish(kda::launch_prefill_tc(t, total_tokens, st_bf16, stream), 1);
  }
  kda::RecArgs a = base_args(p);
  a.n_seqs = n_seqs;
  a.n_slots = n_seqs;
  a.q = q, a.k = k, a.v = v, a.g = g, a.beta = beta;
  a.cu_seqlens = cu_seqlens;
  a.state_in = init_state;
  a.state_out = final_state;
  a.gate = gate_logit;
  a.norm_w = norm_w;
  a.out = out;
  a.ckpt_cu = ckpt_cu, a.ckpt_pos = ckpt_pos, a.ckpt_states = ckpt_states;
  a.total = total_tokens, a.n_ckpt = n_ckpt;
  a.out_q = out_q, a.out_scale = out_scale;
  return finish(kda::launch_recurrent(a, p->d_k, io_bf16, st_bf16, stream), 1);
}

kda_status kda_prefill(const kda_params *p, const void *q, const void *k, const void *v,
                       const float *g, const float *beta, const void *init_state,
                       const int32_t *cu_seqlens, int n_seqs, int64_t total_tokens,
                       const void *gate_logit, const float *norm_w, void *out,
                       void *final_state, void *workspace, size_t ws_bytes,
                       cudaStream_t stream) {
  KDA_TRACE(TR_PREFILL);
  return prefill_impl(p, q, k, v, g, beta, init_state, cu_seqlens, n_seqs, total_tokens,
                      gate_logit, norm_w, out, nullptr, nullptr, final_state, nullptr, nullptr, 0,
                      nullptr, workspace, ws_bytes, stream);
}

kda_status kda_prefill_fp8(const kda_params *p, const void *q, const void *k, const void *v,
                           const float *g, const float *beta, const void *init_state,
                           const int32_t *cu_seqlens, int n_seqs, int64_t total_tokens,
                           const void *gate_logit, const float *norm_w, uint8_t *out_q,
                           float *out_scale, void *final_state, void *workspace,
                           size_t ws_bytes, cudaStream_t stream) {
  KDA_TRACE(TR_PREFILL_FP8);
  if (total_tokens > 0 && !out_q) return KDA_ERR_INVALID_ARG;
  return prefill_impl(p, q, k, v, g, beta, init_state, cu_seqlens, n_seqs, total_tokens,
                      gate_logit, norm_w, nullptr, out_q, out_scale, final_state, nullptr,
                      nullptr, 0, nullptr, workspace, ws_bytes, stream);
}

kda_status kda_prefill_checkpointed(const kda_params *p, const void *q, const void *k,
                                    const void *v, const float *g, const float *beta,
                                    const void *init_state, const int32_t *cu_seqlens,
                                    int n_seqs, int64_t total_tokens, const void *gate_logit,
                                    const float *norm_w, void *out, void *final_state,
                                    const int32_t *ckpt_cu, const int32_t *ckpt_pos,
                                    int n_ckpt, void *ckpt_states, void *workspace,
                                    size_t ws_bytes, cudaStream_t stream) {
  KDA_TRACE(TR_PREFILL_CKPT);
  if (n_ckpt < 1) return KDA_ERR_INVALID_ARG;
  return prefill_impl(p, q, k, v, g, beta, init_state, cu_seqlens, n_seqs, total_tokens,
                      gate_logit, norm_w, out, nullptr, nullptr, final_state, ckpt_cu, ckpt_pos,
                      n_ckpt, ckpt_states, workspace, ws_bytes, stream);
}

kda_status kda_conv_tail_checkpoints(const kda_params *p, const void *x_raw,
                                     const void *conv_state, const int32_t *cu_seqlens,
                                     int n_seqs, int64_t total_tokens, const int32_t *ckpt_cu,
                                     const int32_t *ckpt_pos, int n_ckpt, void *conv_ckpt,
                                     cudaStream_t stream) {
  KDA_TRACE(TR_CONV_TAIL_CKPT);
  kda_status st = check_params(p);
  if (st != KDA_OK) return st;
  if (n_seqs < 1 || n_seqs > 65535 || n_ckpt < 0 || n_ckpt > 65535) return KDA_ERR_INVALID_ARG;
  if (n_ckpt == 0) return KDA_OK;
  if (!x_raw || !cu_seqlens || !ckpt_cu || !ckpt_pos || !conv_ckpt) return KDA_ERR_INVALID_ARG;
  if (!aligned16(x_raw) || !opt_aligned16(conv_state) || !aligned16(cu_seqlens) ||
      !aligned16(ckpt_cu) || !aligned16(ckpt_pos) || !aligned16(conv_ckpt))
    return KDA_ERR_INVALID_ARG;
  const int channels = 3 * p->H * p->d_k;
  if (total_tokens < 0) return KDA_ERR_INVALID_ARG;
  return finish(kda::launch_conv_ckpt(x_raw, conv_state, cu_seqlens, n_seqs, total_tokens,
                                      ckpt_cu, ckpt_pos, n_ckpt, channels, conv_ckpt,
                                      p->io_dtype == KDA_BF16, device_error_ptr(), stream),
                1);
}

static kda_status decode_common(const kda_params *p, const float *g, const float *beta,
                                void *state, int n_slots, const int32_t *slot_idx, int n_seqs,
                                const void *gate_logit, const float *norm_w, void *out) {
  kda_status st = check_params(p);
  if (st != KDA_OK) return st;
  if (n_seqs < 0 || n_seqs > 65535 || n_slots < 0) return KDA_ERR_INVALID_ARG;
  if (n_seqs == 0) return KDA_OK;
  if (!g || !beta || !state || !out) return KDA_ERR_INVALID_ARG;
  if (!slot_idx && n_slots < n_seqs) return KDA_ERR_INVALID_ARG;
  if (!aligned16(g) || !aligned16(beta) || !aligned16(state) || !aligned16(out) ||
      !opt_aligned16(slot_idx) || !opt_aligned16(gate_logit) || !opt_aligned16(norm_w))
    return KDA_ERR_INVALID_ARG;
  return KDA_OK;
}

kda_status kda_decode_step(const kda_params *p, const void *q, const void *k, const void *v,
                           const float *g, const float *beta, void *state, int n_slots,
                           const int32_t *slot_idx, int n_seqs, const void *gate_logit,
                           const float *norm_w, void *out, cudaStream_t stream) {
  KDA_TRACE(TR_DECODE);
  kda_status st = decode_common(p, g, beta, state, n_slots, slot_idx, n_seqs, gate_logit,
                                norm_w, out);
  if (st != KDA_OK || n_seqs == 0) return st;
  if (!q || !k || !v || !aligned16(q) || !aligned16(k) || !aligned16(v))
    return KDA_ERR_INVALID_ARG;
  kda::RecArgs a = base_args(p);
  a.n_seqs = n_seqs;
  a.n_slots = n_slots;
  a.q = q, a.k = k, a.v = v, a.g = g, a.beta = beta;
  a.slot_idx = slot_idx;
  a.state_in = state;
  a.state_out = state;
  a.gate = gate_logit;
  a.norm_w = norm_w;
  a.out = out;
  return finish(kda::launch_recurrent(a, p->d_k, p->io_dtype == KDA_BF16,
                                      p->state_dtype == KDA_BF16, stream),
                1);
}

static kda_status decode_fused_impl(const kda_params *p, const void *x_raw, const void *conv_w,
                                    void *conv_state, const float *g, const float *beta,
                                    void *state, int n_slots, const int32_t *slot_idx,
                                    int n_seqs, const void *gate_logit, const float *norm_w,
                                    void *out, uint8_t *out_q, float *out_scale,
                                    cudaStream_t stream) {
  kda_status st = decode_common(p, g, beta, state, n_slots, slot_idx, n_seqs, gate_logit,
                                norm_w, out_q ? static_cast<void *>(out_q) : out);
  if (st != KDA_OK || n_seqs == 0) return st;
  if (out_q && (!out_scale || !aligned16(out_scale))) return KDA_ERR_INVALID_ARG;
  if (!x_raw || !conv_w || !conv_state || !aligned16(x_raw) || !aligned16(conv_w) ||
      !aligned16(conv_state))
    return KDA_ERR_INVALID_ARG;
  kda::RecArgs a = base_args(p);
  a.n_seqs = n_seqs;
  a.n_slots = n_slots;
  a.x_raw = x_raw;
  a.conv_w = conv_w;
  a.conv_state = conv_state;
  a.g = g, a.beta = beta;
  a.slot_idx = slot_idx;
  a.state_in = state;
  a.state_out = state;
  a.gate = gate_logit;
  a.norm_w = norm_w;
  a.out = out;
  a.out_q = out_q, a.out_scale = out_scale;
  return finish(kda::launch_recurrent(a, p->d_k, p->io_dtype == KDA_BF16,
                                      p->state_dtype == KDA_BF16, stream),
                1);
}

kda_status kda_decode_step_fused(const kda_params *p, const void *x_raw, const void *conv_w,
                                 void *conv_state, const float *g, const float *beta,
                                 void *state, int n_slots, const int32_t *slot_idx, int n_seqs,
                                 const void *gate_logit, const float *norm_w, void *out,
                                 cudaStream_t stream) {
  KDA_TRACE(TR_DECODE_FUSED);
  return decode_fused_impl(p, x_raw, conv_w, conv_state, g, beta, state, n_slots, slot_idx,
                           n_seqs, gate_logit, norm_w, out, nullptr, nullptr, stream);
}

kda_status kda_decode_step_fused_fp8(const kda_params *p, const void *x_raw,
                                     const void *conv_w, void *conv_state, const float *g,
                                     const float *beta, void *state, int n_slots,
                                     const int32_t *slot_idx, int n_seqs,
                                     const void *gate_logit, const float *norm_w,
                                     uint8_t *out_q, float *out_scale, cudaStream_t stream) {
  KDA_TRACE(TR_DECODE_FUSED_FP8);
  return decode_fused_impl(p, x_raw, conv_w, conv_state, g, beta, state, n_slots, slot_idx,
                           n_seqs, gate_logit, norm_w, nullptr, out_q, out_scale, stream);
}

kda_status kda_conv_state_update(const kda_params *p, const void *x_new, const void *conv_w,
                                 void *conv_state, int n_slots, const int32_t *slot_idx,
                                 int n_seqs, int channels, void *y, cudaStream_t stream) {
  KDA_TRACE(TR_CONV_UPDATE);
  if (!p) return KDA_ERR_INVALID_ARG;
  if (p->io_dtype != KDA_F32 && p->io_dtype != KDA_BF16) return KDA_ERR_INVALID_ARG;
  if (n_seqs < 0 || n_seqs > 65535 || channels < 1 || n_slots < 0) return KDA_ERR_INVALID_ARG;
  if (n_seqs == 0) return KDA_OK;
  if (!slot_idx && n_slots < n_seqs) return KDA_ERR_INVALID_ARG;
  if (!x_new || !conv_w || !conv_state || !y || !aligned16(x_new) || !aligned16(conv_w) ||
      !aligned16(conv_state) || !aligned16(y) || !opt_aligned16(slot_idx))
    return KDA_ERR_INVALID_ARG;
  kda::ConvArgs a;
  a.n_seqs = n_seqs;
  a.channels = channels;
  a.x_new = x_new;
  a.conv_w = conv_w;
  a.conv_state = conv_state;
  a.slot_idx = slot_idx;
  a.n_slots = n_slots;
  a.err = device_error_ptr();
  a.y = y;
  return finish(kda::launch_conv_update(a, p->io_dtype == KDA_BF16, stream), 1);
}

kda_status kda_decode_multi(const kda_params *p, const void *q, const void *k, const void *v,
                            const float *g, const float *beta, void *state, int n_slots,
                            const int32_t *slot_idx, int n_seqs, int K, const void *gate_logit,
                            const float *norm_w, void *out, void *step_states, int commit_final,
                            cudaStream_t stream) {
  KDA_TRACE(TR_DECODE_MULTI);
  if (K < 1 || K > 64) return KDA_ERR_INVALID_ARG;
  if ((int64_t)n_seqs * K > 65535 * 64) return KDA_ERR_UNSUPPORTED;
  kda_status st = decode_common(p, g, beta, state, n_slots, slot_idx, n_seqs, gate_logit,
                                norm_w, out);
  if (st != KDA_OK || n_seqs == 0) return st;
  if (!q || !k || !v || !aligned16(q) || !aligned16(k) || !aligned16(v) ||
      !opt_aligned16(step_states))
    return KDA_ERR_INVALID_ARG;
  if (!step_states && !commit_final) return KDA_ERR_INVALID_ARG;  // nothing would be kept
  kda::RecArgs a = base_args(p);
  a.n_seqs = n_seqs;
  a.n_slots = n_slots;
  a.tokens_per_seq = K;
  a.total = (int64_t)n_seqs * K;
  a.q = q, a.k = k, a.v = v, a.g = g, a.beta = beta;
  a.slot_idx = slot_idx;
  a.state_in = state;
  a.state_out = commit_final ? state : nullptr;
  a.step_states = step_states;
  a.gate = gate_logit;
  a.norm_w = norm_w;
  a.out = out;
  return finish(kda::launch_recurrent(a, p->d_k, p->io_dtype == KDA_BF16,
                                      p->state_dtype == KDA_BF16, stream),
                1);
}

kda_status kda_state_accept(const kda_params *p, const void *step_states, int n_seqs, int K,
                            const int32_t *accept_len, void *state, int n_slots,
                            const int32_t *slot_idx, cudaStream_t stream) {
  KDA_TRACE(TR_STATE_ACCEPT);
  kda_status st = check_params(p);
  if (st != KDA_OK) return st;
  if (n_seqs < 0 || n_seqs > 65535 || K < 1 || K > 64 || n_slots < 0) return KDA_ERR_INVALID_ARG;
  if (n_seqs == 0) return KDA_OK;
  if (!step_states || !accept_len || !state) return KDA_ERR_INVALID_ARG;
  if (!slot_idx && n_slots < n_seqs) return KDA_ERR_INVALID_ARG;
  if (!aligned16(step_states) || !aligned16(state) || !opt_aligned16(slot_idx))
    return KDA_ERR_INVALID_ARG;
  return finish(kda::launch_state_accept(step_states, state, accept_len, slot_idx, n_slots,
                                         n_seqs, K, p->H, p->d_k, p->state_dtype == KDA_BF16,
                                         device_error_ptr(), stream),
                1);
}

// ---- absorbed gated-MLA decode ----------------------------------------------------------

static kda_status mla_common(const void *cache, int64_t cache_len, const int32_t *lengths,
                             int n_seqs, float scale, float *z) {
  if (n_seqs < 0 || n_seqs > 65535 || !(scale > 0.f) || !(scale < 1e30f))
    return KDA_ERR_INVALID_ARG;
  if (n_seqs == 0) return KDA_OK;
  if (cache_len < 1 || cache_len > (int64_t)1 << 30 || !cache || !lengths || !z)
    return KDA_ERR_INVALID_ARG;
  if (!aligned16(cache) || !aligned16(lengths) || !aligned16(z)) return KDA_ERR_INVALID_ARG;
  return KDA_OK;
}

kda_status mla_set_split_override(int n_split) {
  return kda::mla_set_split(n_split) ? KDA_OK : KDA_ERR_INVALID_ARG;
}

size_t mla_decode_workspace_size(int n_seqs, int64_t cache_len) {
  if (n_seqs < 1 || n_seqs > 65535 || cache_len < 1) return 0;
  return kda::mla_split_bytes(kda::mla_preferred_split(n_seqs, cache_len), n_seqs);
}

// the preferred split of each sequence's positions, lowered to what the workspace holds
static int mla_split_for(int n_seqs, int64_t cache_len, size_t ws_bytes) {
  int ns = kda::mla_preferred_split(n_seqs, cache_len);
  while (ns > 1 && kda::mla_split_bytes(ns, n_seqs) > ws_bytes) --ns;
  return ns;
}

kda_status mla_decode_latent(const void *q_cat, const void *cache, int64_t cache_len,
                             const int32_t *lengths, int n_seqs, float scale, float *z,
                             void *workspace, size_t ws_bytes, cudaStream_t stream) {
  KDA_TRACE(TR_MLA_LATENT);
  kda_status st = mla_common(cache, cache_len, lengths, n_seqs, scale, z);
  if (st != KDA_OK || n_seqs == 0) return st;
  if (!q_cat || !aligned16(q_cat) || !opt_aligned16(workspace)) return KDA_ERR_INVALID_ARG;
  if (!workspace) ws_bytes = 0;
  if (!kda::mla_latent_supported()) return KDA_ERR_UNSUPPORTED;
  kda::MlaArgs a;
  std::memset(&a, 0, sizeof a);
  a.B = n_seqs, a.L_max = cache_len, a.scale_log2 = scale * 1.4426950408889634f;
  a.q_cat = const_cast<void *>(q_cat), a.cache = cache, a.lengths = lengths, a.z = z;
  a.n_split = mla_split_for(n_seqs, cache_len, ws_bytes);
  a.part = static_cast<float *>(workspace);
  a.err = device_error_ptr();
  return finish(kda::launch_mla_latent(a, stream), a.n_split > 1 ? 2 : 1);
}

kda_status mla_decode_latent_noalloc(const void *q_cat, const void *cache, int64_t cache_len,
                                     const int32_t *lengths, int n_seqs, float scale, float *z,
                                     cudaStream_t stream) {
  KDA_TRACE(TR_MLA_LATENT_NOALLOC);
  kda_status st = mla_common(cache, cache_len, lengths, n_seqs, scale, z);
  if (st != KDA_OK || n_seqs == 0) return st;
  if (!q_cat || !aligned16(q_cat)) return KDA_ERR_INVALID_ARG;
  const size_t need = mla_decode_workspace_size(n_seqs, cache_len);
  if (need > kda::mla_static_scratch_bytes()) return KDA_ERR_WORKSPACE;
  if (!kda::mla_latent_supported()) return KDA_ERR_UNSUPPORTED;
  void *scratch = need ? kda::mla_static_scratch() : nullptr;
  if (need && !scratch) return KDA_ERR_CUDA;
  kda::MlaArgs a;
  std::memset(&a, 0, sizeof a);
  a.B = n_seqs, a.L_max = cache_len, a.scale_log2 = scale * 1.4426950408889634f;
  a.q_cat = const_cast<void *>(q_cat), a.cache = cache, a.lengths = lengths, a.z = z;
  a.n_split = mla_split_for(n_seqs, cache_len, need);
  a.part = static_cast<float *>(scratch);
  a.err = device_error_ptr();
  return finish(kda::launch_mla_latent(a, stream), a.n_split > 1 ? 2 : 1);
}

kda_status mla_decode(const void *q_nope, const void *q_rope, const void *w_uk,
                      const void *w_uv, const void *cache, int64_t cache_len,
                      const int32_t *lengths, int n_seqs, const void *gate_logit, float scale,
                      void *q_cat, float *z, void *out, void *workspace, size_t ws_bytes,
                      cudaStream_t stream) {
  KDA_TRACE(TR_MLA_DECODE);
  kda_status st = mla_common(cache, cache_len, lengths, n_seqs, scale, z);
  if (st != KDA_OK || n_seqs == 0) return st;
  if (!q_nope || !q_rope || !w_uk || !w_uv || !gate_logit || !q_cat || !out)
    return KDA_ERR_INVALID_ARG;
  if (!aligned16(q_nope) || !aligned16(q_rope) || !aligned16(w_uk) || !aligned16(w_uv) ||
      !aligned16(gate_logit) || !aligned16(q_cat) || !aligned16(out) ||
      !opt_aligned16(workspace))
    return KDA_ERR_INVALID_ARG;
  if (!workspace) ws_bytes = 0;
  if (!kda::mla_latent_supported()) return KDA_ERR_UNSUPPORTED;
  kda::MlaArgs a;
  std::memset(&a, 0, sizeof a);
  a.B = n_seqs, a.L_max = cache_len, a.scale_log2 = scale * 1.4426950408889634f;
  a.q_nope = q_nope, a.q_rope = q_rope, a.w_uk = w_uk, a.w_uv = w_uv, a.gate = gate_logit;
  a.q_cat = q_cat, a.cache = cache, a.lengths = lengths, a.z = z, a.out = out;
  a.n_split = mla_split_for(n_seqs, cache_len, ws_bytes);
  a.part = static_cast<float *>(workspace);
  a.err = device_error_ptr();
  cudaError_t e = kda::launch_mla_absorb(a, stream);
  if (e == cudaSuccess) e = kda::launch_mla_latent(a, stream);
  if (e == cudaSuccess) e = kda::launch_mla_up_gate(a, stream);
  return finish(e, a.n_split > 1 ? 4 : 3);
}

kda_status kda_check_device_error(cudaStream_t stream) {
  KDA_TRACE(TR_CHECK_ERROR);
  if (cudaStreamSynchronize(stream) != cudaSuccess) return KDA_ERR_CUDA;
  int *ptr = device_error_ptr();
  if (!ptr) return KDA_ERR_CUDA;
  int host = 0;
  if (cudaMemcpy(&host, ptr, sizeof host, cudaMemcpyDeviceToHost) != cudaSuccess)
    return KDA_ERR_CUDA;
  if (host != 0) {
    const int zero = 0;
    if (cudaMemcpy(ptr, &zero, sizeof zero, cudaMemcpyHostToDevice) != cudaSuccess)
      return KDA_ERR_CUDA;
    if (host & kda::ERR_MBAR_TIMEOUT) return KDA_ERR_TIMEOUT;
    return (host & kda::ERR_BAD_INDEX) ? KDA_ERR_BAD_INDEX : KDA_ERR_BAD_SEQLENS;
  }
  return KDA_OK;
}

kda_status kda_wait_probe(int64_t probes, cudaStream_t stream) {
  KDA_TRACE(TR_WAIT_PROBE);
  if (probes < 1 || probes > ((int64_t)1 << 30)) return KDA_ERR_INVALID_ARG;
  return finish(kda::launch_wait_probe((long)probes, device_error_ptr(), stream), 1);
}

uint64_t kda_launch_count(void) { return g_launches.load(); }

int kda_trace_ranges(const char **names, int max_names) {
  for (int i = 0; names && i < max_names && i < kda::TR_COUNT; ++i) names[i] = kda::kTraceNames[i];
  return kda::TR_COUNT;
}

}  // extern "C"

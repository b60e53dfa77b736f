// kda_internal.h -- argument blocks and launchers shared between the ABI layer and kernels.
#pragma once

#include <cuda_runtime.h>

#include <cstdint>

namespace kda {

// bits of the library's sticky device error flag
enum : int { ERR_MBAR_TIMEOUT = 1, ERR_BAD_SEQLEN = 2, ERR_BAD_INDEX = 4 };

// Token-serial recurrence (decode, and the exact-fp32 prefill path).
struct RecArgs {
  int H, n_seqs;
  float scale, l2_eps, norm_eps, g_min;
  int qk_l2norm;
  const void *q, *k, *v;       // [T, H, D] io (unused when x_raw is set)
  const float *g, *beta;       // [T, H, D], [T, H]
  const void *x_raw;           // fused conv (decode): [N, 3HD] io, or nullptr
  const void *conv_w;          // [3HD, 4] io
  void *conv_state;            // [slots, 3, 3HD] io, updated in place
  const int32_t *cu_seqlens;   // prefill: [N + 1]; nullptr for decode (seq n = token n)
  const int32_t *slot_idx;     // decode: state/conv slot of each sequence, or nullptr
  int n_slots;                 // slots in the state pool (slot indices are checked against it)
  int64_t total;               // rows of q, k, v, g, out (sequence offsets are checked against it)
  int n_ckpt;                  // checkpoints (checkpoint ranges are checked against it)
  int tokens_per_seq;          // decode: tokens per sequence (rows n*K .. n*K+K-1); 0 = one
  void *step_states;           // decode: [N*K, H, D, D] state after each token, or nullptr
  const int32_t *ckpt_cu;      // prefill: checkpoints of sequence n are ckpt_cu[n] .. [n+1]
  const int32_t *ckpt_pos;     // tokens of the sequence before each checkpoint
  void *ckpt_states;           // [n_ckpt, H, D, D] state dtype
  const void *state_in;        // [N or slots, H, D, D] state dtype, or nullptr (zeros)
  void *state_out;             // same layout, or nullptr; may equal state_in
  const void *gate;            // [T, H, D] io or nullptr
  const float *norm_w;         // [D] or nullptr
  void *out;                   // [T, H, D] io (unused when out_q is set)
  uint8_t *out_q;              // [T, H, D] FP8 E4M3 codes of the output, or nullptr
  float *out_scale;            // [T, H] fp32 scale of each (token, head) group
  int *err;
};

// Absorbed gated-MLA decode, the pages' shapes: 64 heads, latent 512 + positional key 64,
// 128-wide non-positional query and value per head.
struct MlaArgs {
  int B;                       // sequences (one query token each)
  int64_t L_max;               // cache rows per sequence
  float scale_log2;            // score scale x log2(e)
  const void *q_nope, *q_rope; // [B, 64, 128], [B, 64, 64] bf16
  const void *w_uk, *w_uv;     // [64, 128, 512] bf16 each
  const void *gate;            // [B, 64] bf16 gate logits
  void *q_cat;                 // [B, 64, 576] bf16 absorbed query (written, then read)
  const void *cache;           // [B, L_max, 576] bf16: latent | positional key per row
  const int32_t *lengths;      // [B] cached positions of each sequence
  float *z;                    // [B, 64, 512] fp32 attention output (latent)
  int n_split;                 // splits of each sequence's positions (1: none)
  float *part;                 // split partials: [n_split, B, 64, 512] Z, then [.., 64, 2] (m, l)
  void *out;                   // [B, 64, 128] bf16 gated head outputs
  int *err;
};

struct ProArgs {
  int H, n_seqs;
  int64_t T;
  float l2_eps, g_min;
  int l2norm_qk;
  const void *x;               // [T, 3HD]
  const void *conv_w;          // [3HD, 4]
  void *conv_state;            // [N, 3, 3HD] or nullptr
  const int32_t *cu_seqlens;
  const float *beta_logit;     // [T, H] or nullptr
  const float *g_raw;          // [T, H, D] or nullptr
  void *q, *k, *v;             // [T, H, D]
  float *beta, *g;
  int *err;
};

struct ConvArgs {
  int n_seqs, channels, n_slots;
  int *err;
  const void *x_new;           // [N, C]
  const void *conv_w;          // [C, 4]
  void *conv_state;            // [slots, 3, C]
  const int32_t *slot_idx;
  void *y;                     // [N, C]
};

cudaError_t launch_recurrent(const RecArgs &a, int D, bool io_bf16, bool st_bf16,
                             cudaStream_t s);
// pool[slot(n)] <- step_states[n*K + accept[n] - 1] for accept[n] in 1..K (0: unchanged)
cudaError_t launch_state_accept(const void *step_states, void *pool, const int32_t *accept,
                                const int32_t *slot_idx, int n_slots, int n_seqs, int K, int H,
                                int D, bool st_bf16, int *err, cudaStream_t s);
cudaError_t launch_prologue(const ProArgs &a, int D, bool io_bf16, cudaStream_t s);
// the one-token decode step at d = 128 (kda_decode.cu): serves decode calls without step
// states or checkpoints
bool decode_one_serves(const RecArgs &a, int D);
cudaError_t launch_decode_one(const RecArgs &a, bool io_bf16, bool st_bf16, cudaStream_t s);
// out[k] <- the three raw inputs before checkpoint k (conv tail at that position)
cudaError_t launch_wait_probe(long limit, int *err, cudaStream_t s);
bool mla_latent_supported();
int mla_preferred_split(int n_seqs, int64_t cache_len);
bool mla_set_split(int n);  // 0: the automatic rule; 1..64: that split count
size_t mla_split_bytes(int n_split, int n_seqs);
size_t mla_static_scratch_bytes();
void *mla_static_scratch();  // this device's copy, or nullptr
cudaError_t launch_mla_absorb(const MlaArgs &a, cudaStream_t s);
cudaError_t launch_mla_latent(const MlaArgs &a, cudaStream_t s);
cudaError_t launch_mla_up_gate(const MlaArgs &a, cudaStream_t s);
cudaError_t launch_conv_ckpt(const void *x, const void *conv_state, const int32_t *cu,
                             int n_seqs, int64_t T, const int32_t *ckpt_cu,
                             const int32_t *ckpt_pos, int n_ckpt, int channels, void *out,
                             bool io_bf16, int *err, cudaStream_t s);
cudaError_t launch_conv_update(const ConvArgs &a, bool io_bf16, cudaStream_t s);

}  // namespace kda

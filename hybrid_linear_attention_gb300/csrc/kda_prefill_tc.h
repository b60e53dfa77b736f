// kda_prefill_tc.h -- chunked KDA prefill on the 5th-generation tensor cores (tcgen05).
#pragma once

#include <cuda_runtime.h>

#include <cstdint>

namespace kda {

struct TcArgs {
  int H, n_seqs;
  float scale, l2_eps, norm_eps, g_min;
  int qk_l2norm;
  const void *q, *k, *v;       // [T, H, 128] bf16
  const float *g, *beta;       // [T, H, 128], [T, H]
  const void *init_state;      // [N, H, 128, 128] state dtype or nullptr
  void *final_state;           // same or nullptr (may alias init_state)
  const int32_t *cu_seqlens;   // [N + 1]
  const void *gate;            // [T, H, 128] bf16 or nullptr
  const float *norm_w;         // [128] or nullptr
  void *out;                   // [T, H, 128] bf16
  uint8_t *out_q;              // FP8 E4M3 output codes [T, H, D] (instead of out), or nullptr
  float *out_scale;            // [T, H] fp32 scale of each (token, head) group
  int64_t total;               // rows of q, k, v, g, out (sequence offsets are checked against it)
  int n_ckpt;                  // checkpoints (checkpoint ranges are checked against it)
  const int32_t *ckpt_cu;      // checkpoints of sequence n: ckpt_cu[n] .. ckpt_cu[n+1], or null
  const int32_t *ckpt_pos;     // tokens of the sequence before each checkpoint
  void *ckpt_states;           // [n_ckpt, H, 128, 128] state dtype
  int *err;
  int form;                    // kda_prefill_form: 0 automatic, 1 one CTA, 2 cluster pair
};

// True when the tensor-core path serves this shape (d = 128, bf16 I/O).
bool prefill_tc_supported(int d, bool io_bf16);
cudaError_t launch_prefill_tc(const TcArgs &a, int64_t total_tokens, bool st_bf16, cudaStream_t s);

}  // namespace kda

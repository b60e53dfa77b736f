/*
 * kda.h -- C ABI of the GB300 (sm_103a) Kimi Delta Attention (KDA) token-mixer library.
 *
 * What the layer computes (web pages, cited by title and section):
 *   [Grouped]  "Ling-3.1-flash: Grouped Routing and Two Different MLA Caches",
 *              section "KDA replaces a token list with a recurrent matrix": q, k, v streams of
 *              64 x 128 channels, each through its own causal short convolution of width 4
 *              with SiLU; q and k normalised; channel-dependent retention; a delta-rule
 *              write that corrects the state's prediction for k toward v; the safe forget
 *              gate's log-retention lower bound -5; an output normalisation and sigmoid gate.
 *   [Headers]  "Ling-3.1-flash: a 560B hybrid-attention MoE, counted from its safetensors
 *              headers", section "How KDA and MLA split the work", the state equation:
 *              a 128 x 128 state per head, decayed by Diag(alpha_t), written with strength
 *              beta_t (one scalar per head), read as o_t = S_t^T q_t.
 *   [Budget]   "Ling-3.1-flash: What 63 Linear-Attention Layers Do to the KV Budget",
 *              section "The memory math": fp32 state of 64 x 128 x 128 values per layer and
 *              sequence; the short-convolution tails.
 *
 * Per head and token (state S is d_k x d_v, row i = key channel, column j = value channel):
 *     alpha = exp(max(g, g_min));  S' = Diag(alpha) S;  u = beta (v - S'^T k)
 *     S = S' + k u^T;  o = scale * S^T q
 * with q, k L2-normalised first when params->qk_l2norm is set, and, when gate logits are
 * given, o <- o / sqrt(mean_j o_j^2 + norm_eps) * norm_w * sigmoid(gate).
 *
 * Conventions for every entry point:
 *  - Every pointer is a DEVICE pointer unless stated otherwise; tensors are dense and
 *    row-major in the layouts given.  The caller owns every buffer; the library allocates
 *    no device memory.
 *  - Calls are asynchronous on the given stream; they return after enqueueing.
 *  - Arguments are validated on the host before anything is launched.  Errors are
 *    returned (never thrown, never trapped on the device): KDA_ERR_INVALID_ARG for bad
 *    pointers/sizes, KDA_ERR_UNSUPPORTED for valid but unimplemented shapes or dtypes,
 *    KDA_ERR_CUDA when a launch fails.  Device-side waits are bounded; a wait that runs out
 *    sets a sticky device flag read by kda_check_device_error().
 *  - Packed sequences: token t of the batch lives at row t of every [T_tot, ...] tensor;
 *    sequence n owns rows [cu_seqlens[n], cu_seqlens[n+1]).  cu_seqlens is a device int32
 *    array of n_seqs + 1 non-decreasing offsets starting at 0.  The library does not read
 *    it on the host; the kernels check every sequence's offsets against [0, total_tokens]
 *    and treat one that falls outside (or runs backwards) as empty, setting the sticky flag
 *    (KDA_ERR_BAD_SEQLENS).  Offsets that are in range but not non-decreasing across
 *    sequences give unspecified values for those rows, never an access outside the
 *    buffers.
 *  - Supported: d_k == d_v == d in {16, 128}; any H >= 1; sequences of any length >= 0.
 */
#ifndef KDA_H_
#define KDA_H_

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  KDA_OK = 0,
  KDA_ERR_INVALID_ARG = -1,
  KDA_ERR_UNSUPPORTED = -2,
  KDA_ERR_CUDA = -3,
  KDA_ERR_WORKSPACE = -4,
  KDA_ERR_TIMEOUT = -5,
  KDA_ERR_BAD_INDEX = -6,
  KDA_ERR_BAD_SEQLENS = -7
} kda_status;

typedef enum { KDA_F32 = 0, KDA_BF16 = 1 } kda_dtype;

/* Kernel form of the tensor-core prefill (d = 128, bf16 I/O); other shapes ignore it.  Every
 * form computes the same function; they differ in how the SMs are spent. */
typedef enum {
  KDA_PREFILL_AUTO = 0,  /* the library chooses by the batch's shape and the device's SMs */
  KDA_PREFILL_FUSED = 1, /* one CTA per (head, sequence) walks its chunks                 */
  KDA_PREFILL_PAIR = 2   /* a cluster of two CTAs per (head, sequence): one builds each
                            chunk's intra-chunk products, the other walks the state       */
} kda_prefill_form;

/* Layer configuration.  Defaults in brackets are the pages' configuration. */
typedef struct {
  int H;                 /* heads [64]                                                  */
  int d_k, d_v;          /* head dims, equal, 16 or 128 [128]                           */
  float scale;           /* read scale applied to S^T q [1.0]                           */
  float l2_eps;          /* q/k L2 norm: x / sqrt(sum x^2 + l2_eps) [1e-6]              */
  float norm_eps;        /* output RMS norm epsilon [1e-6]                              */
  float g_min;           /* log-retention lower bound of the safe forget gate [-5]      */
  int qk_l2norm;         /* 1: L2-normalise q and k inside the call [1]                 */
  kda_dtype io_dtype;    /* q, k, v, raw x, conv weights/state, gate logits, out [BF16] */
  kda_dtype state_dtype; /* recurrent state storage [F32]; BF16 = bf16 storage variant   */
  int prefill_form;      /* kda_prefill_form [KDA_PREFILL_AUTO]                          */
} kda_params;

/* Fills *p with the pages' configuration (H 64, d 128, scale 1, eps 1e-6, g_min -5,
 * qk_l2norm 1, bf16 I/O, fp32 state) and the automatic prefill form. */
void kda_params_default(kda_params* p);

/* Human-readable name of a status code (static storage). */
const char* kda_status_string(kda_status s);

/* Bytes of one sequence's recurrent state for one layer: H * d_k * d_v * sizeof(state).
 * [Budget] "The memory math": 64 x 128 x 128 fp32 values = 4 MiB per layer. */
size_t kda_state_bytes(const kda_params* p);

/* Device workspace kda_prefill needs for this batch (0 today; kept so callers can size a
 * buffer once).  Returns 0 for invalid params. */
size_t kda_prefill_workspace_size(const kda_params* p, int n_seqs, int64_t total_tokens);

/*
 * kda_prologue -- short convolution + SiLU (+ optional q/k L2 norm) + gate activations for a
 * packed batch ([Grouped]: "Each projection passes through its own causal short
 * convolution of width four with SiLU activation").
 *
 *   x_raw       [T_tot, 3*H*d] io_dtype: the q, k and v projections side by side
 *               (channels [0,Hd) = q, [Hd,2Hd) = k, [2Hd,3Hd) = v; head h of a stream is
 *               channels h*d .. h*d+d-1 of it).
 *   conv_w      [3*H*d, 4] io_dtype: y[t,c] = SiLU(sum_j conv_w[c][j] * x[t-3+j, c]).
 *   conv_state  [n_seqs, 3, 3*H*d] io_dtype or NULL.  In: the three raw inputs before each
 *               sequence (oldest first); taps before the sequence start read it (zeros if
 *               NULL).  Out (updated in place when non-NULL): the last three raw inputs of
 *               each sequence, reaching into the old tail for sequences shorter than 3;
 *               a length-0 sequence keeps its tail.  Bit-exact copies.
 *   q, k, v     [T_tot, H, d] io_dtype outputs (SiLU(conv) of each stream).
 *   l2norm_qk   1: q and k outputs are L2-normalised per head (eps = p->l2_eps).
 *   beta_logit  [T_tot, H] fp32 or NULL -> beta [T_tot, H] fp32 = sigmoid(beta_logit).
 *   g_raw       [T_tot, H, d] fp32 or NULL -> g [T_tot, H, d] fp32 = max(g_raw, p->g_min).
 */
kda_status kda_prologue(const kda_params* p, const void* x_raw, const void* conv_w,
                        void* conv_state, const int32_t* cu_seqlens, int n_seqs,
                        int64_t total_tokens, int l2norm_qk, const float* beta_logit,
                        const float* g_raw, void* q, void* k, void* v, float* beta, float* g,
                        cudaStream_t stream);

/*
 * kda_prefill -- the recurrence over a packed batch of sequences ([Headers] state equation,
 * [Grouped] delta-rule write), chunk-parallel inside each sequence.
 *
 *   q, k        [T_tot, H, d_k] io_dtype; v [T_tot, H, d_v] io_dtype.
 *   g           [T_tot, H, d_k] fp32 log-retention (clamped at p->g_min inside).
 *   beta        [T_tot, H] fp32 write strength in (0, 1).
 *   init_state  [n_seqs, H, d_k, d_v] state_dtype, or NULL for zeros.
 *   cu_seqlens  [n_seqs + 1] int32 (device): cu_seqlens[0] = 0, non-decreasing,
 *               cu_seqlens[n_seqs] = total_tokens.  A sequence whose offsets fall outside
 *               [0, total_tokens] (or run backwards) is treated as empty and reported by
 *               kda_check_device_error (KDA_ERR_BAD_SEQLENS).
 *   gate_logit  [T_tot, H, d_v] io_dtype, or NULL: no output norm/gate (plain read).
 *   norm_w      [d_v] fp32 output-norm weight, or NULL for ones (used only with a gate).
 *   out         [T_tot, H, d_v] io_dtype.
 *   final_state [n_seqs, H, d_k, d_v] state_dtype, or NULL.  May alias init_state.
 *   workspace / ws_bytes: at least kda_prefill_workspace_size() bytes (may be NULL when 0).
 * A length-0 sequence copies its initial state (or zeros) to final_state.
 */
kda_status kda_prefill(const kda_params* p, const void* q, const void* k, const void* v,
                       const float* g, const float* beta, const void* init_state,
                       const int32_t* cu_seqlens, int n_seqs, int64_t total_tokens,
                       const void* gate_logit, const float* norm_w, void* out,
                       void* final_state, void* workspace, size_t ws_bytes,
                       cudaStream_t stream);

/*
 * kda_prefill_fp8 -- kda_prefill whose output leaves the kernel quantised for a block-FP8
 * o_proj, as kda_decode_step_fused_fp8 does for decode (same pages, same reading): one group
 * per (token, head).
 *
 *   out_q      [T_tot, H, d_v] uint8 E4M3 codes of o * (448 / a) (nearest even, saturated),
 *              a = max(amax, 1e-10) over the group's d_v values (after the output norm and
 *              gate when gate logits are given).
 *   out_scale  [T_tot, H] fp32: a / 448.
 *   Other arguments as kda_prefill.
 */
kda_status kda_prefill_fp8(const kda_params* p, const void* q, const void* k, const void* v,
                           const float* g, const float* beta, const void* init_state,
                           const int32_t* cu_seqlens, int n_seqs, int64_t total_tokens,
                           const void* gate_logit, const float* norm_w, uint8_t* out_q,
                           float* out_scale, void* final_state, void* workspace,
                           size_t ws_bytes, cudaStream_t stream);

/*
 * kda_prefill_checkpointed -- kda_prefill that also saves the state at caller-given token
 * boundaries inside the sequences (prefix-state checkpoints: a recurrent state can be
 * reused only where a snapshot of it was saved, "Ling-3.1-flash: What 63 Linear-Attention
 * Layers Do to the KV Budget", section "Where the hybrid makes serving harder").
 *
 *   ckpt_cu     [n_seqs + 1] int32 (device): checkpoints of sequence n are
 *               ckpt_cu[n] .. ckpt_cu[n+1]-1, non-decreasing, ckpt_cu[n_seqs] = n_ckpt.
 *   ckpt_pos    [n_ckpt] int32 (device): tokens of its sequence before the checkpoint,
 *               strictly increasing within a sequence, each in [1, length] and a multiple
 *               of 64 (the chunk) or the sequence length.  A fork at another position is
 *               taken by ending a sequence there and passing its final state on as the
 *               next part's init_state.
 *   ckpt_states [n_ckpt, H, d_k, d_v] state_dtype: the state after ckpt_pos[j] tokens of
 *               its sequence, the same value a kda_prefill of that prefix leaves in
 *               final_state.
 *   Other arguments as kda_prefill.  n_ckpt >= 1 (KDA_ERR_INVALID_ARG otherwise).  Ranges
 *   or positions that break these rules are skipped and reported by
 *   kda_check_device_error (KDA_ERR_BAD_INDEX); the outputs and final states are unaffected.
 */
kda_status kda_prefill_checkpointed(const kda_params* p, const void* q, const void* k,
                                    const void* v, const float* g, const float* beta,
                                    const void* init_state, const int32_t* cu_seqlens,
                                    int n_seqs, int64_t total_tokens, const void* gate_logit,
                                    const float* norm_w, void* out, void* final_state,
                                    const int32_t* ckpt_cu, const int32_t* ckpt_pos,
                                    int n_ckpt, void* ckpt_states, void* workspace,
                                    size_t ws_bytes, cudaStream_t stream);

/*
 * kda_conv_tail_checkpoints -- the short-convolution half of a prefix checkpoint: for every
 * checkpoint j (ckpt_cu / ckpt_pos as in kda_prefill_checkpointed, any position in
 * [1, length] allowed), the three raw inputs before position ckpt_pos[j] of its sequence,
 * oldest first, i.e. the conv_state a kda_prologue of that prefix would leave.  Reuse at
 * a token boundary needs both halves ("Ling-3.1-flash: Grouped Routing and Two Different
 * MLA Caches", section "Two cache budgets for one checkpoint": prefix reuse restores every
 * recurrent state at the same boundary).
 *
 *   x_raw       [T_tot, 3*H*d] io_dtype, as kda_prologue.
 *   conv_state  [n_seqs, 3, 3*H*d] io_dtype or NULL: the tails before the sequences (the
 *               values kda_prologue reads, so call this first when kda_prologue updates
 *               them in place); taps before a sequence start read it (zeros if NULL).
 *   conv_ckpt   [n_ckpt, 3, 3*H*d] io_dtype output.  Bit-exact copies.
 * n_ckpt = 0 is a no-op.  A position outside [1, length] is skipped and reported
 * (KDA_ERR_BAD_INDEX).
 */
kda_status kda_conv_tail_checkpoints(const kda_params* p, const void* x_raw,
                                     const void* conv_state, const int32_t* cu_seqlens,
                                     int n_seqs, int64_t total_tokens, const int32_t* ckpt_cu,
                                     const int32_t* ckpt_pos, int n_ckpt, void* conv_ckpt,
                                     cudaStream_t stream);

/*
 * kda_decode_step -- one token for each of n_seqs sequences, state updated in place.
 *
 *   q, k, v     [n_seqs, H, d] io_dtype (post-convolution streams).
 *   g           [n_seqs, H, d] fp32 log-retention; beta [n_seqs, H] fp32.
 *   state       [n_slots, H, d, d] state_dtype pool, updated in place.
 *   slot_idx    [n_seqs] int32 (device): sequence n uses state slot slot_idx[n]; NULL means
 *               slot n.  Slots must be distinct; a slot outside [0, n_slots) is skipped and
 *               reported by kda_check_device_error (KDA_ERR_BAD_INDEX).
 *   gate_logit  [n_seqs, H, d] io_dtype or NULL; norm_w [d] fp32 or NULL.
 *   out         [n_seqs, H, d] io_dtype.
 * Each head's state is read from HBM once and written once.
 */
kda_status kda_decode_step(const kda_params* p, const void* q, const void* k, const void* v,
                           const float* g, const float* beta, void* state, int n_slots,
                           const int32_t* slot_idx, int n_seqs, const void* gate_logit,
                           const float* norm_w, void* out, cudaStream_t stream);

/*
 * kda_conv_state_update -- decode-time short convolution: for each sequence n and channel c,
 * y[n,c] = SiLU(sum_{j<3} conv_w[c][j] * conv_state[s][j][c] + conv_w[c][3] * x_new[n,c]),
 * then conv_state[s] <- (conv_state[s][1], conv_state[s][2], x_new[n]) in place, where
 * s = slot_idx[n] (or n when slot_idx is NULL).
 *   x_new [n_seqs, channels], conv_w [channels, 4], conv_state [n_slots, 3, channels],
 *   y [n_seqs, channels]; all io_dtype.  The state shift is bit-exact.
 */
kda_status kda_conv_state_update(const kda_params* p, const void* x_new, const void* conv_w,
                                 void* conv_state, int n_slots, const int32_t* slot_idx,
                                 int n_seqs, int channels, void* y, cudaStream_t stream);

/*
 * kda_decode_step_fused -- kda_conv_state_update and kda_decode_step in one launch, from
 * the raw projections: x_raw [n_seqs, 3*H*d] (q|k|v as in kda_prologue), conv_w
 * [3*H*d, 4], conv_state [n_slots, 3, 3*H*d] updated in place; the convolved q, k, v stay
 * in fp32 on chip.  Other arguments as in kda_decode_step.
 */
kda_status kda_decode_step_fused(const kda_params* p, const void* x_raw, const void* conv_w,
                                 void* conv_state, const float* g, const float* beta,
                                 void* state, int n_slots, const int32_t* slot_idx, int n_seqs,
                                 const void* gate_logit, const float* norm_w, void* out,
                                 cudaStream_t stream);

/*
 * kda_decode_step_fused_fp8 -- kda_decode_step_fused whose output leaves the kernel already
 * quantised for a block-FP8 o_proj.  The checkpoint's weights are E4M3 in 128 x 128 scaling
 * blocks with dynamic activation quantisation ("Ling-3.1-flash: Grouped Routing and Two
 * Different MLA Caches", section "Production boundaries"), and the serving setup fuses this
 * quantisation into the KDA kernel for decode ("Ling-3.1-flash: What 63 Linear-Attention
 * Layers Do to the KV Budget", section "Fitting it on a node").  One group = the d values of
 * one (sequence, head): the 128 input channels that meet one weight block.
 *
 *   out_q      [n_seqs, H, d] uint8: E4M3 codes (1 sign, 4 exponent bits with bias 7,
 *              3 mantissa bits, no infinities) of o * (448 / a), rounded to nearest even
 *              and saturated at +-448; a = max(amax, 1e-10), amax = max |o| over the group
 *              (o after the output norm and gate when gate logits are given).
 *   out_scale  [n_seqs, H] fp32: scale = a / 448 (value = code * scale).
 *   The divisions and the product are IEEE fp32 round-to-nearest.  Other arguments as
 *   kda_decode_step_fused.
 */
kda_status kda_decode_step_fused_fp8(const kda_params* p, const void* x_raw,
                                     const void* conv_w, void* conv_state, const float* g,
                                     const float* beta, void* state, int n_slots,
                                     const int32_t* slot_idx, int n_seqs,
                                     const void* gate_logit, const float* norm_w,
                                     uint8_t* out_q, float* out_scale, cudaStream_t stream);

/*
 * kda_decode_multi -- K tokens for each of n_seqs sequences (a speculative draft), from the
 * state in its pool slot, keeping the state after every token for rollback.  The pages
 * count speculative rollback state among the per-sequence costs of a KDA layer
 * ("Ling-3.1-flash: Grouped Routing and Two Different MLA Caches", section "KDA replaces a
 * token list with a recurrent matrix") and report MTP acceptance lengths of 2.1-2.6 tokens
 * ("Ling-3.1-flash: What 63 Linear-Attention Layers Do to the KV Budget", section "Where the
 * hybrid makes serving harder").  No counterpart interface is printed on the pages.
 *
 *   q, k, v, gate_logit, out [n_seqs * K, H, d] io_dtype, sequence-major (row n*K + i is
 *               token i of sequence n); g [n_seqs * K, H, d] fp32; beta [n_seqs * K, H] fp32.
 *   state       [n_slots, H, d, d] state_dtype pool: read; written with the state after all
 *               K tokens only when commit_final is nonzero.
 *   slot_idx    as in kda_decode_step.
 *   K           1..64.
 *   step_states [n_seqs * K, H, d, d] state_dtype or NULL: the state after token i of
 *               sequence n at row n*K + i.  At least one of step_states / commit_final.
 * Token by token the result equals K calls of kda_decode_step.  Slot indices outside
 * [0, n_slots) are skipped and reported by kda_check_device_error (KDA_ERR_BAD_INDEX).
 */
kda_status kda_decode_multi(const kda_params* p, const void* q, const void* k, const void* v,
                            const float* g, const float* beta, void* state, int n_slots,
                            const int32_t* slot_idx, int n_seqs, int K, const void* gate_logit,
                            const float* norm_w, void* out, void* step_states, int commit_final,
                            cudaStream_t stream);

/*
 * kda_state_accept -- commit the accepted part of a speculative step: for every sequence n
 * and head, state[slot(n)] <- step_states[n*K + accept_len[n] - 1] when
 * 1 <= accept_len[n] <= K; accept_len[n] == 0 leaves the pool state as it was.  Bit-exact
 * copies.
 *   step_states [n_seqs * K, H, d, d] from kda_decode_multi; accept_len [n_seqs] int32
 *   (device); state, n_slots, slot_idx as in kda_decode_step.  Out-of-range accept lengths
 *   or slots are skipped and reported by kda_check_device_error (KDA_ERR_BAD_INDEX).
 * No counterpart interface is printed on the pages.
 */
kda_status kda_state_accept(const kda_params* p, const void* step_states, int n_seqs, int K,
                            const int32_t* accept_len, void* state, int n_slots,
                            const int32_t* slot_idx, cudaStream_t stream);

/*
 * kda_prefill_host_workspace_size -- device bytes kda_prefill_host needs for n_seqs sequences
 * cut into segments of at most segment_tokens rows (a positive multiple of 64, at most 2^24),
 * with gate logits when with_gate is nonzero: two sets of segment buffers (raw projections,
 * log-retention, write-strength logits, gate logits, output), one set of convolved q, k, v
 * and beta, and every sequence's carried fp32 state and conv tail: at H = 64, d = 128 with
 * bf16 I/O about 241 KB per segment row (273 KB with gate logits) plus 4.3 MB per sequence.
 * Returns 0 for invalid arguments.
 */
size_t kda_prefill_host_workspace_size(const kda_params* p, int n_seqs, int64_t segment_tokens,
                                       int with_gate);

/*
 * kda_prefill_host -- the prefill hot path (kda_prologue: short convolution, SiLU and
 * beta = sigmoid(logit); then kda_prefill: q/k L2 norm, the clamp of g at p->g_min, the
 * chunked recurrence and the optional output norm and gate) for a packed batch whose inputs
 * and outputs are in HOST memory.  The batch is streamed through the GPU in segments of at
 * most segment_tokens rows (the last ones halving down to 64 rows, so that little work is left
 * once the last inputs are in): while the kernels run on one segment, the next segment's inputs
 * are copied in and the previous segment's output is copied out.  Every inner segment
 * boundary falls on a chunk edge (a multiple of 64 tokens from the start of the sequence it
 * cuts), and the state and conv tail of a cut sequence are carried on the device to the next
 * segment -- the way a serving engine runs a long prompt's prefill in pieces ("Ling-3.1-flash:
 * What 63 Linear-Attention Layers Do to the KV Budget", section "Where the hybrid makes
 * serving harder": a recurrent state summarises everything before it).  The results are the
 * same bits as kda_prologue (conv_state in place, l2norm_qk = 0, no g output) followed by one
 * kda_prefill over the whole batch on device copies of these buffers, when both runs choose
 * the same kernel form (as they do for batches of up to SM count / (2 H) sequences).
 *
 * HOST pointers (page-locked memory lets the copies overlap the kernels; pageable memory
 * works but serialises them):
 *   x_raw       [T_tot, 3*H*d] io_dtype raw q|k|v projections, as in kda_prologue.
 *   conv_state  [n_seqs, 3, 3*H*d] io_dtype, in/out (the conv tails, updated as kda_prologue
 *               updates them), or NULL: zeros in, nothing written back.
 *   cu_seqlens  [n_seqs + 1] int32: 0, non-decreasing, ending at total_tokens (checked here,
 *               KDA_ERR_INVALID_ARG otherwise).
 *   beta_logit  [T_tot, H] fp32 write-strength logits; g_raw [T_tot, H, d] fp32 raw
 *               log-retention (clamped inside).
 *   init_state  [n_seqs, H, d, d] fp32 or NULL (zeros).
 *   gate_logit  [T_tot, H, d] io_dtype or NULL (no output norm/gate).
 *   out         [T_tot, H, d] io_dtype.
 *   final_state [n_seqs, H, d, d] fp32 or NULL; may alias init_state.
 * DEVICE pointers: conv_w [3*H*d, 4] io_dtype and norm_w [d] fp32 or NULL (layer weights,
 * resident on the GPU); workspace: kda_prefill_host_workspace_size() bytes, 256-byte aligned,
 * owned by the caller and not to be touched until the call's work has finished.
 *
 * Only fp32 state storage (p->state_dtype == KDA_F32; KDA_ERR_UNSUPPORTED otherwise): a bf16
 * state would be rounded at every segment boundary.  The call enqueues its work and returns;
 * the kernels run on `stream`, the copies on three copy streams of the library (created on the
 * first call on each device and kept until the process exits) that start after the work
 * already on `stream`, and `stream` is made to wait for all of it: synchronising `stream`
 * (or kda_check_device_error(stream)) means the outputs are in host memory.  Calls are
 * serialised per device while they enqueue.  Not meant for CUDA-graph capture.  Arguments are
 * checked on the host before any CUDA call.  A launch or copy that fails part-way returns its
 * error (KDA_ERR_CUDA) after making `stream` wait for the copies already issued; the outputs
 * are then undefined.
 */
kda_status kda_prefill_host(const kda_params* p, const void* x_raw, const void* conv_w,
                            void* conv_state, const int32_t* cu_seqlens, int n_seqs,
                            int64_t total_tokens, const float* beta_logit, const float* g_raw,
                            const void* init_state, const void* gate_logit,
                            const float* norm_w, void* out, void* final_state, void* workspace,
                            size_t ws_bytes, int64_t segment_tokens, cudaStream_t stream);

/*
 * kda_prefill_host_plan -- the segments kda_prefill_host cuts a batch into (host only, no CUDA
 * call): with cu_seqlens a HOST array as in kda_prefill_host, writes the row boundaries
 * 0 = b_0 < b_1 < ... < b_k = total_tokens to bounds[0 .. min(k, max_segments)] and returns
 * k, the number of segments (0 for an empty batch); -1 for invalid arguments (the checks of
 * kda_prefill_host).  Every segment holds at most segment_tokens rows; every inner boundary
 * lies a multiple of 64 tokens after the start of the sequence it falls in; the last
 * 2 * segment_tokens rows are cut in halves down to 64 rows.
 */
int64_t kda_prefill_host_plan(const int32_t* cu_seqlens, int n_seqs, int64_t total_tokens,
                              int64_t segment_tokens, int64_t* bounds, int64_t max_segments);

/* Synchronises `stream`, then reads and clears the library's sticky device error flag
 * (set when a bounded device wait ran out, a device-side index was out of range, or a
 * sequence's offsets fell outside the token rows).  Returns KDA_OK, KDA_ERR_TIMEOUT,
 * KDA_ERR_BAD_INDEX, KDA_ERR_BAD_SEQLENS (in that order of precedence) or KDA_ERR_CUDA. */
kda_status kda_check_device_error(cudaStream_t stream);

/* Failure detection without a GPU fault: launches a one-thread kernel that waits, with the
 * same bounded mbarrier wait the tensor-core kernels use, on a barrier nothing ever arrives
 * at; after `probes` (1 .. 2^30) unsuccessful probes it gives up and raises the sticky flag,
 * exactly as a kernel whose copy or product never completed would, and returns.  A following
 * kda_check_device_error then reports KDA_ERR_TIMEOUT and the context stays usable.  No
 * counterpart interface is printed on the pages. */
kda_status kda_wait_probe(int64_t probes, cudaStream_t stream);

/* Number of kernels the library launched since load (host-side counter, for benchmarks). */
uint64_t kda_launch_count(void);

/* Names of the NVTX ranges the library opens around its calls (one per traced entry point:
 * the compute calls, kda_prefill_host, kda_check_device_error and kda_wait_probe; each range
 * spans the call's host-side work and names the kernels it enqueues on a timeline).  Writes up
 * to max_names pointers to static strings into names (may be NULL) and returns the count. */
int kda_trace_ranges(const char** names, int max_names);

#ifdef __cplusplus
}
#endif

#endif /* KDA_H_ */

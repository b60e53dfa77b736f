/*
 * mla.h -- C ABI of the absorbed gated-MLA decode (the hybrid's other token mixer) in the
 * same GB300 (sm_103a) library as kda.h; conventions as kda.h (device pointers, caller-owned
 * buffers, asynchronous on the stream, host validation with status codes, 16-byte alignment,
 * device-side index checks reported by kda_check_device_error).
 *
 * What it computes ("Ling-3.1-flash: Grouped Routing and Two Different MLA Caches",
 * sections "MLA's expanded reference path" and "Why weight absorption keeps the same
 * attention function"): each cached position t of a sequence keeps the normalised latent
 * c_t (512) and the rotated positional key r_t (64) shared by the 64 heads.  For the query
 * token, head i has non-positional part q_i^N (128) and rotated positional part q_i^R (64);
 * the key and value up-projections W_K,i, W_V,i are 128 x 512.  Absorbed execution:
 *     q~_i = W_K,i^T q_i^N                             (512)
 *     s_t  = scale * ([q~_i ; q_i^R] . [c_t ; r_t])      over t < length
 *     z_i  = sum_t softmax_t(s)_t c_t                  (512: the latent is the value)
 *     o_i  = W_V,i z_i * sigmoid(gate_i)               (128; one gate logit per head)
 * the same attention function as expanding every cached position into 64 heads of 192-wide
 * keys and 128-wide values (scale 1/sqrt(192) in the pages' configuration).
 * The shapes are the pages': 64 heads, latent 512, positional key 64, 128-wide q^N and o.
 */
#ifndef MLA_H_
#define MLA_H_

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#include "kda.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Device workspace that lets mla_decode_latent / mla_decode split each sequence's cached
 * positions across several CTAs (so a small batch still fills the GPU): partial sums of each
 * split, merged by a second launch.  0 when no split pays (then no workspace is needed).
 * With less than this, the calls use as many splits as fit (down to none). */
size_t mla_decode_workspace_size(int n_seqs, int64_t cache_len);

/* Tuning and testing only: forces the split count of every later mla_decode_latent /
 * mla_decode_latent_noalloc / mla_decode call and of mla_decode_workspace_size in this
 * process (1..64; 0 restores the automatic rule: as many splits as fill the SMs in one wave,
 * each at least 512 positions).  Process-wide, not per device or stream; set it only while
 * no MLA call is being issued.  KDA_ERR_INVALID_ARG outside 0..64. */
kda_status mla_set_split_override(int n_split);

/*
 * mla_decode_latent -- the attention over the latent cache (the part that streams it).
 *
 *   q_cat      [n_seqs, 64, 576] bf16: [q~_i ; q_i^R] per head.
 *   cache      [n_seqs, cache_len, 576] bf16: row t of sequence n = [c_t ; r_t]; rows at or
 *              past lengths[n] are ignored (their contents may be anything).
 *   lengths    [n_seqs] int32 (device), 0..cache_len; a length outside that range is
 *              treated as 0 and reported (KDA_ERR_BAD_INDEX).  Length 0 gives z = 0.
 *   scale      score scale (> 0).
 *   z          [n_seqs, 64, 512] fp32 output.
 *   workspace / ws_bytes: caller-owned, up to mla_decode_workspace_size() bytes, or NULL / 0
 *              (one CTA per sequence).  Splits write each head's unnormalised sum with its
 *              running maximum and normaliser; the merge rescales them to a common maximum.
 * Scores and the weighted sum run on the tensor cores with bf16 operands and fp32
 * accumulation (the weights are rounded to bf16 as operands; the normaliser sums the same
 * rounded weights).
 */
kda_status mla_decode_latent(const void* q_cat, const void* cache, int64_t cache_len,
                             const int32_t* lengths, int n_seqs, float scale, float* z,
                             void* workspace, size_t ws_bytes, cudaStream_t stream);

/*
 * mla_decode_latent_noalloc -- mla_decode_latent with no caller workspace and no allocation.
 * No counterpart on the pages (they describe the attention, not how its scratch memory is
 * provided): the split partial sums go to a fixed 24 MiB device buffer inside the library
 * (each device its own copy), so the call needs no memory from the caller.  The split count
 * is the one mla_decode_workspace_size() sizes; if that needs more than the fixed buffer, the
 * call returns KDA_ERR_WORKSPACE and launches nothing.  Calls on one device share the buffer:
 * issue them in one stream (or otherwise ordered), never concurrently.  Arguments, layouts
 * and results as mla_decode_latent; bit-identical to it with a workspace of that size.
 */
kda_status mla_decode_latent_noalloc(const void* q_cat, const void* cache, int64_t cache_len,
                                     const int32_t* lengths, int n_seqs, float scale, float* z,
                                     cudaStream_t stream);

/*
 * mla_decode -- one absorbed gated-MLA decode step: absorption, mla_decode_latent, value
 * up-projection and gate.
 *
 *   q_nope     [n_seqs, 64, 128] bf16;  q_rope [n_seqs, 64, 64] bf16 (already rotated).
 *   w_uk, w_uv [64, 128, 512] bf16: W_K,i and W_V,i of each head.
 *   gate_logit [n_seqs, 64] bf16: one logit per head.
 *   q_cat      [n_seqs, 64, 576] bf16 and z [n_seqs, 64, 512] fp32: caller-owned
 *              intermediates (the absorbed query, the latent attention output).
 *   out        [n_seqs, 64, 128] bf16: o_i of every head.
 *   cache, cache_len, lengths, scale, workspace, ws_bytes as mla_decode_latent.
 */
kda_status mla_decode(const void* q_nope, const void* q_rope, const void* w_uk,
                      const void* w_uv, const void* cache, int64_t cache_len,
                      const int32_t* lengths, int n_seqs, const void* gate_logit, float scale,
                      void* q_cat, float* z, void* out, void* workspace, size_t ws_bytes,
                      cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif  /* MLA_H_ */

// kda_trace.h -- NVTX ranges around the C ABI's calls, so a timeline (Nsight Systems, or any
// tool attached through NVTX) shows each call's host-side span and the kernels it enqueued
// under it.  Header-only NVTX v3: with no tool attached a range costs a branch.
#pragma once

#include <nvtx3/nvToolsExt.h>

namespace kda {

// One name per traced entry point; kda_trace_ranges() returns this table.
enum TraceId {
  TR_PROLOGUE, TR_PREFILL, TR_PREFILL_FP8, TR_PREFILL_CKPT, TR_CONV_TAIL_CKPT, TR_DECODE,
  TR_DECODE_FUSED, TR_DECODE_FUSED_FP8, TR_CONV_UPDATE, TR_DECODE_MULTI, TR_STATE_ACCEPT,
  TR_PREFILL_HOST, TR_MLA_LATENT, TR_MLA_LATENT_NOALLOC, TR_MLA_DECODE, TR_CHECK_ERROR,
  TR_WAIT_PROBE, TR_COUNT
};
extern const char *const kTraceNames[TR_COUNT];

struct TraceRange {
  explicit TraceRange(TraceId id) { nvtxRangePushA(kTraceNames[id]); }
  ~TraceRange() { nvtxRangePop(); }
  TraceRange(const TraceRange &) = delete;
  TraceRange &operator=(const TraceRange &) = delete;
};

}  // namespace kda

#define KDA_TRACE(id) const ::kda::TraceRange kda_trace_range_(::kda::id)

// kda_prefill_tc.cu -- chunked KDA prefill on tcgen05 tensor cores (not yet enabled).
#include "kda_prefill_tc.h"

namespace kda {

bool prefill_tc_supported(int, bool) { return false; }

cudaError_t launch_prefill_tc(const TcArgs &, bool, cudaStream_t) {
  return cudaErrorNotSupported;
}

}  // namespace kda

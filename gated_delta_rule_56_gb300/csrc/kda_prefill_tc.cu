// kda_prefill_tc.cu -- tensor-core chunked prefill (placeholder until the kernel lands).
#include "kda_internal.h"

namespace kda {

bool tc_prefill_supported(kda_dtype, int, int, const RunParams &) { return false; }

cudaError_t launch_tc_prefill(const RunParams &, cudaStream_t) { return cudaErrorNotSupported; }

}  // namespace kda

// pa_prefill.cu -- chunked causal prefill against a paged context.
#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {

bool prefill_supported(int, int, int) { return false; }

cudaError_t launch_prefill(const PrefillArgs &, cudaStream_t) { return cudaErrorNotSupported; }

}  // namespace pa

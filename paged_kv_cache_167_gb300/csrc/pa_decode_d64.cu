// pa_decode_d64.cu -- instantiates the paged decode kernels for head_dim 64.
#include "pa_decode_kernel.cuh"

namespace pa {
cudaError_t launch_decode_d64(const DecodeArgs &a, cudaStream_t stream) {
    return decode::launch_for_dim<64>(a, stream);
}
}  // namespace pa

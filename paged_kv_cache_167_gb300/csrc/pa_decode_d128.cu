// pa_decode_d128.cu -- instantiates the paged decode kernels for head_dim 128.
#include "pa_decode_kernel.cuh"

namespace pa {
cudaError_t launch_decode_d128(const DecodeArgs &a, cudaStream_t stream) {
    return decode::launch_for_dim<128>(a, stream);
}
}  // namespace pa

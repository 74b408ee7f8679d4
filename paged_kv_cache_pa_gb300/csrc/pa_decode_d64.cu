// pa_decode_d64.cu -- paged decode attention instantiations for head_dim 64
// (fp16 / bf16, query groups 1, 2, <=4, <=6, <=8).
#include "pa_decode_launch.cuh"

namespace pa {
pa_status_t launch_decode_d64(const DecodeParams &P, pa_dtype_t dtype, int grid_cap,
                               cudaStream_t stream, int kernel) {
    return dispatch_dtype<64>(P, dtype, grid_cap, stream, kernel);
}
}  // namespace pa

// ssd_stream_f32.cu -- the streaming kernel (ssd_stream_kernel.cuh) for fp32
// logits.
#include "ssd_stream_kernel.cuh"

namespace ssd {

template cudaError_t launch_stream_dt<1>(const VerifyParams& p, int grid, cudaStream_t s);

}  // namespace ssd

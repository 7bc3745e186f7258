// ssd_stream_bf16.cu -- the streaming kernel (ssd_stream_kernel.cuh) for
// bf16 logits, and the shared-memory size every instantiation uses.
#include "ssd_stream_kernel.cuh"

namespace ssd {

int stream_smem_bytes() {
  return kStagesA * kStageBytes + 2 * (kStagesA + kPieceSlots) * (int)sizeof(uint64_t) +
         kPieceSlots * (int)sizeof(PieceRed);
}

template cudaError_t launch_stream_dt<0>(const VerifyParams& p, int grid, cudaStream_t s);

}  // namespace ssd

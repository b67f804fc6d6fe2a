// Tensor-core decode (placeholder until the tcgen05 kernel lands).
#include "common.cuh"
#include "kernels.h"

namespace mla {

bool decode_tc_supported(int, int, int, int, int) { return false; }
int decode_tc_workers(int num_sms) { return num_sms; }
cudaError_t launch_decode_tc(const DecodeArgs&, cudaStream_t) { return cudaErrorNotSupported; }

}  // namespace mla

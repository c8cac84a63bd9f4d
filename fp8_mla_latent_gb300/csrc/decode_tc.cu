// decode_tc.cu -- tcgen05 tensor-core split-T decode (under construction).
#include "kv8_common.cuh"

namespace kv8 {
bool tc_available() { return false; }
cudaError_t launch_decode_tc(const DecodeArgs&, cudaStream_t) { return cudaErrorNotSupported; }
}  // namespace kv8

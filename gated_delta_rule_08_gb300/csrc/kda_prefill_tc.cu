// KDA chunked prefill on the tcgen05 tensor cores (bf16 inputs).  Placeholder until
// the tensor-core kernels land: reports "not supported" so bf16 runs on the CUDA-core path.
#include "kda_internal.h"

namespace kda {
size_t prefill_tc_blob_bytes(int, int) { return 0; }
bool prefill_tc_supported(int, int) { return false; }
cudaError_t prefill_tc_launch(const PrefillArgs&, cudaStream_t) { return cudaErrorNotSupported; }
}  // namespace kda

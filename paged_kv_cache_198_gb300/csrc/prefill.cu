// prefill.cu -- chunked causal prefill (placeholder until the tensor-core
// kernel lands).
#include "kernels.h"

namespace tvl {

cudaError_t launch_prefill(const PrefillArgs&, cudaStream_t) { return cudaErrorNotSupported; }

}  // namespace tvl

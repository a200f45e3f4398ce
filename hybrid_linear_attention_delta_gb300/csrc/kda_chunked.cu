// kda_chunked.cu -- chunked KDA prefill on tcgen05 tensor cores (sm_103a).
#include "kda_internal.cuh"

namespace kda {

bool chunked_supported(const PrefillPlan &) { return false; }

cudaError_t launch_chunked_prefill(const PrefillPlan &) { return cudaErrorNotSupported; }

}  // namespace kda

// kda_prefill_tc.cu -- fused tensor-core (tcgen05) chunked KDA prefill.
#include "kda_internal.cuh"

namespace kda {

bool prefill_tc_supported(const kda_desc_t&) { return false; }
size_t prefill_tc_workspace(const kda_desc_t&) { return 0; }
cudaError_t launch_prefill_tc(const PrefillArgs&, cudaStream_t) { return cudaErrorNotSupported; }

}  // namespace kda

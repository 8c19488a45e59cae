// ffn_prefill.cu -- large-M grouped MXFP4 GEMMs (prefill path).
#include "moe_internal.h"

namespace moe {

bool prefill_tile_supported(int) { return false; }
bool prefill_shape_supported(int, int) { return false; }
cudaError_t launch_prefill_gate_up(const GroupedGemm&, cudaStream_t) { return cudaErrorNotSupported; }
cudaError_t launch_prefill_down(const GroupedGemm&, cudaStream_t) { return cudaErrorNotSupported; }

}  // namespace moe

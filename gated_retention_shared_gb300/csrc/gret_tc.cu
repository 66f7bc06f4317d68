// gret_tc.cu -- tensor-core (tcgen05) chunkwise gated retention.  Placeholder
// until the sm_103a kernel lands: nothing is eligible, so the CUDA-core path runs.
#include "common.cuh"
#include "kernels.h"

namespace yoco_host {
bool gret_tc_eligible(int, int, int, int, int, yoco_dtype) { return false; }
size_t gret_tc_workspace(int, int, int, int, int) { return 0; }
cudaError_t gret_prefill_tc(const GretArgs &, void *, cudaStream_t) { return cudaErrorNotSupported; }
}  // namespace yoco_host

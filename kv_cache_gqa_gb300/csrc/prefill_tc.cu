// Kernel (b), tensor-core form (tcgen05): not built yet in this revision.
#include "launch.h"

namespace kva {

bool prefill_tc_supports(int, kva_dtype) { return false; }
cudaError_t launch_prefill_tc(const PrefillArgs&, cudaStream_t) { return cudaErrorNotSupported; }

}  // namespace kva

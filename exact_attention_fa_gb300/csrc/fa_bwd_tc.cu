// Backward (placeholder until the tcgen05 backward lands).
#include "fa_internal.h"

namespace fa {
cudaError_t launch_bwd(const BwdParams&, int, cudaStream_t) { return cudaErrorNotSupported; }
}  // namespace fa

// fa_bwd.cu -- backward pass (work in progress).
#include "fa_internal.h"

namespace fa {
cudaError_t launch_bwd(const BwdLaunch&) { return cudaErrorNotSupported; }
}  // namespace fa

// kernel_splitrow.cu -- split-row variant (not built yet: never selected).
#include "launch.h"

namespace rwo {
bool splitrow_fits(const RowProblem&, const DeviceInfo&) { return false; }
cudaError_t launch_splitrow(const RowProblem&, const DeviceInfo&) { return cudaErrorNotSupported; }
}  // namespace rwo

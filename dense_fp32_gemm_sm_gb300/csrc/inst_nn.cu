// Kernel instantiations for transa = N, transb = N.
#include "simt_launch.cuh"

namespace fgemm {
FGEMM_LAUNCH_TABLE(kLaunchNN, 0, 0)
}  // namespace fgemm

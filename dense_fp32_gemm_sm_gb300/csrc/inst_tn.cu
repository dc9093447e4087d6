// Kernel instantiations for transa = T, transb = N.
#include "simt_launch.cuh"

namespace fgemm {
FGEMM_LAUNCH_TABLE(kLaunchTN, 1, 0)
}  // namespace fgemm

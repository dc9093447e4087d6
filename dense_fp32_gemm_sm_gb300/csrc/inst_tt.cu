// Kernel instantiations for transa = T, transb = T.
#include "simt_launch.cuh"

namespace fgemm {
FGEMM_LAUNCH_TABLE(kLaunchTT, 1, 1)
}  // namespace fgemm

// Kernel instantiations for transa = N, transb = T.
#include "simt_launch.cuh"

namespace fgemm {
FGEMM_LAUNCH_TABLE(kLaunchNT, 0, 1)
}  // namespace fgemm

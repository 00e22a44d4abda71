// int32 instantiation of the blocked Floyd-Warshall kernels.
#include "fw_launch_impl.cuh"

APSP_INSTANTIATE_LAUNCHERS(int32_t)

namespace apsp {
int phase3_slab_rows() { return KS; }
}  // namespace apsp

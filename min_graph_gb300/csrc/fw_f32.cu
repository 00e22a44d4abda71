// fp32 instantiation of the blocked Floyd-Warshall kernels.
#include "fw_launch_impl.cuh"

APSP_INSTANTIATE_LAUNCHERS(float)

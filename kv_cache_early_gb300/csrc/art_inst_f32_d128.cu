// Instantiations of the ART kernels for fp32 K/V with head_dim 128.
#include "art_kernel.cuh"

ART_INSTANTIATE(false, 128, 1)
ART_INSTANTIATE(false, 128, 2)
ART_INSTANTIATE(false, 128, 4)
ART_INSTANTIATE(false, 128, 7)
ART_INSTANTIATE(false, 128, 8)

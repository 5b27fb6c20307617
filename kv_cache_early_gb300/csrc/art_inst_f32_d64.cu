// Instantiations of the ART kernels for fp32 K/V with head_dim 64.
#include "art_kernel.cuh"

ART_INSTANTIATE(false, 64, 1)
ART_INSTANTIATE(false, 64, 2)
ART_INSTANTIATE(false, 64, 4)
ART_INSTANTIATE(false, 64, 7)
ART_INSTANTIATE(false, 64, 8)

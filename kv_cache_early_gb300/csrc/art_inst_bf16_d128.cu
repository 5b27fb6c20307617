// Instantiations of the ART kernels for bf16 K/V with head_dim 128.
#include "art_kernel.cuh"

ART_INSTANTIATE(true, 128, 1)
ART_INSTANTIATE(true, 128, 2)
ART_INSTANTIATE(true, 128, 4)
ART_INSTANTIATE(true, 128, 7)
ART_INSTANTIATE(true, 128, 8)

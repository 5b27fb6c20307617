// Instantiations of the ART kernels for bf16 K/V with head_dim 64.
#include "art_kernel.cuh"

ART_INSTANTIATE(true, 64, 1)
ART_INSTANTIATE(true, 64, 2)
ART_INSTANTIATE(true, 64, 4)
ART_INSTANTIATE(true, 64, 7)
ART_INSTANTIATE(true, 64, 8)

// Instantiations of the unit path (one item over many CTAs) for bf16 K/V with head_dim 128.
#include "art_units.cuh"

ART_UNITS_INSTANTIATE(128, 1)
ART_UNITS_INSTANTIATE(128, 2)
ART_UNITS_INSTANTIATE(128, 4)
ART_UNITS_INSTANTIATE(128, 7)
ART_UNITS_INSTANTIATE(128, 8)

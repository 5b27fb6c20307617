// Instantiations of the unit path (one item over many CTAs) for bf16 K/V with head_dim 64.
#include "art_units.cuh"

ART_UNITS_INSTANTIATE(64, 1)
ART_UNITS_INSTANTIATE(64, 2)
ART_UNITS_INSTANTIATE(64, 4)
ART_UNITS_INSTANTIATE(64, 7)
ART_UNITS_INSTANTIATE(64, 8)

// Affine comparison decode, code widths 6 and 8 (see kvarn_affine_dec.cuh).
#include "kvarn_affine_dec.cuh"

KVARN_AFFINE_DECODE(6)
KVARN_AFFINE_DECODE(8)

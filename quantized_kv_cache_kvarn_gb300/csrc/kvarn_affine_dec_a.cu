// Affine comparison decode, code widths 2, 3 and 4 (see kvarn_affine_dec.cuh).
#include "kvarn_affine_dec.cuh"

KVARN_AFFINE_DECODE(2)
KVARN_AFFINE_DECODE(3)
KVARN_AFFINE_DECODE(4)

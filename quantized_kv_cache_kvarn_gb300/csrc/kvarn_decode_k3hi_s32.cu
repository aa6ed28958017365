// Decode kernels for key code width 3 with value widths 5, 6, 8
// (fp32 scales, head_dim 128; the preset 4 / 2 has its own instantiation);
// the pairs are split over translation units so that they compile in
// parallel.
#include "kvarn_decode_kernel.cuh"

namespace kvarn {
KVARN_DECODE_WIDTHS(3, 5, 4)
KVARN_DECODE_WIDTHS(3, 6, 4)
KVARN_DECODE_WIDTHS(3, 8, 4)
}  // namespace kvarn

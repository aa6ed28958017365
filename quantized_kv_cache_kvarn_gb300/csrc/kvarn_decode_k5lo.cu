// Decode kernels for key code width 5 with value widths 2, 3, 4
// (fp16 scales, head_dim 128); the pairs are split over translation units so
// that they compile in parallel.
#include "kvarn_decode_kernel.cuh"

namespace kvarn {
KVARN_DECODE_WIDTHS(5, 2, 2)
KVARN_DECODE_WIDTHS(5, 3, 2)
KVARN_DECODE_WIDTHS(5, 4, 2)
}  // namespace kvarn

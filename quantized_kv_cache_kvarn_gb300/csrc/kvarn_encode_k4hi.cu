// Encode kernels for key code width 4 with value widths 5, 6, 8
// (fp16 scales, head_dim 128); the pairs are split over translation units so
// that they compile in parallel.
#include "kvarn_encode_kernel.cuh"

namespace kvarn {
KVARN_ENCODE_WIDTHS(4, 5, 2)
KVARN_ENCODE_WIDTHS(4, 6, 2)
KVARN_ENCODE_WIDTHS(4, 8, 2)
}  // namespace kvarn

// Encode kernels for key code width 4 with value widths 2, 3, 4
// (fp16 scales, head_dim 128); the pairs are split over translation units so
// that they compile in parallel.
#include "kvarn_encode_kernel.cuh"

namespace kvarn {
KVARN_ENCODE_WIDTHS(4, 2, 2)
KVARN_ENCODE_WIDTHS(4, 3, 2)
KVARN_ENCODE_WIDTHS(4, 4, 2)
}  // namespace kvarn

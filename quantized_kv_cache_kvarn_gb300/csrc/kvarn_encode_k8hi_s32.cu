// Encode kernels for key code width 8 with value widths 5, 6, 8
// (fp32 scales, head_dim 128; the preset 4 / 2 has its own instantiation);
// the pairs are split over translation units so that they compile in
// parallel.
#include "kvarn_encode_kernel.cuh"

namespace kvarn {
KVARN_ENCODE_WIDTHS(8, 5, 4)
KVARN_ENCODE_WIDTHS(8, 6, 4)
KVARN_ENCODE_WIDTHS(8, 8, 4)
}  // namespace kvarn

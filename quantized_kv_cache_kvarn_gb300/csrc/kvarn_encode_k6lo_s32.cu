// Encode kernels for key code width 6 with value widths 2, 3, 4
// (fp32 scales, head_dim 128; the preset 4 / 2 has its own instantiation);
// the pairs are split over translation units so that they compile in
// parallel.
#include "kvarn_encode_kernel.cuh"

namespace kvarn {
KVARN_ENCODE_WIDTHS(6, 2, 4)
KVARN_ENCODE_WIDTHS(6, 3, 4)
KVARN_ENCODE_WIDTHS(6, 4, 4)
}  // namespace kvarn

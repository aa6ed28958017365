// Encode kernels for code widths K4 / V4 with fp16 scales (head_dim 128).
#include "kvarn_encode_kernel.cuh"

namespace kvarn {
KVARN_ENCODE_WIDTHS(4, 4, 2)
}  // namespace kvarn

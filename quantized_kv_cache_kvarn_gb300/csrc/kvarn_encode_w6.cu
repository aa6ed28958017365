// Encode kernels for code widths K6 / V6 with fp16 scales (head_dim 128).
#include "kvarn_encode_kernel.cuh"

namespace kvarn {
KVARN_ENCODE_WIDTHS(6, 6, 2)
}  // namespace kvarn

// Encode kernels for code widths K5 / V5 with fp16 scales (head_dim 128).
#include "kvarn_encode_kernel.cuh"

namespace kvarn {
KVARN_ENCODE_WIDTHS(5, 5, 2)
}  // namespace kvarn

// Decode kernels for code widths K5 / V5 with fp16 scales (head_dim 128).
#include "kvarn_decode_kernel.cuh"

namespace kvarn {
KVARN_DECODE_WIDTHS(5, 5, 2)
}  // namespace kvarn

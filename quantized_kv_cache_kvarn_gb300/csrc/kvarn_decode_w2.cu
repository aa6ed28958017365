// Decode kernels for code widths K2 / V2 with fp16 scales (head_dim 128).
#include "kvarn_decode_kernel.cuh"

namespace kvarn {
KVARN_DECODE_WIDTHS(2, 2, 2)
}  // namespace kvarn

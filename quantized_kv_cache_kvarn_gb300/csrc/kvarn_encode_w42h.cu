// Encode kernels for code widths K4 / V2 with fp16 scales (head_dim 128).
#include "kvarn_encode_kernel.cuh"

namespace kvarn {
KVARN_ENCODE_WIDTHS(4, 2, 2)
}  // namespace kvarn

// Encode kernels for code widths K3 / V3 with fp16 scales (head_dim 128).
#include "kvarn_encode_kernel.cuh"

namespace kvarn {
KVARN_ENCODE_WIDTHS(3, 3, 2)
}  // namespace kvarn

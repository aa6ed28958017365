// Encode kernels for code widths K8 / V8 with fp16 scales (head_dim 128).
#include "kvarn_encode_kernel.cuh"

namespace kvarn {
KVARN_ENCODE_WIDTHS(8, 8, 2)
}  // namespace kvarn

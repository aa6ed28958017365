// Decode kernels for code widths K8 / V8 with fp16 scales (head_dim 128).
#include "kvarn_decode_kernel.cuh"

namespace kvarn {
KVARN_DECODE_WIDTHS(8, 8, 2)
}  // namespace kvarn

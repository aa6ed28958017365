// Decode kernels at head_dim 256 with fp16 scales for the width pairs K5V5, K6V6, K8V8.
#include "kvarn_decode_kernel.cuh"

namespace kvarn {
KVARN_DECODE_WIDTHS_256(5, 5)
KVARN_DECODE_WIDTHS_256(6, 6)
KVARN_DECODE_WIDTHS_256(8, 8)
}  // namespace kvarn

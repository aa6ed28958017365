// Decode kernels at head_dim 256 with fp16 scales for the width pairs K2V2, K3V3, K4V2, K4V4.
#include "kvarn_decode_kernel.cuh"

namespace kvarn {
KVARN_DECODE_WIDTHS_256(2, 2)
KVARN_DECODE_WIDTHS_256(3, 3)
KVARN_DECODE_WIDTHS_256(4, 2)
KVARN_DECODE_WIDTHS_256(4, 4)
}  // namespace kvarn

// Decode kernels at head_dim 256 with fp16 scales for key code width 3 and
// every value width; one translation unit per key width, so that the pairs
// compile in parallel.
#include "kvarn_decode_kernel.cuh"

namespace kvarn {
KVARN_DECODE_WIDTHS_256(3, 2)
KVARN_DECODE_WIDTHS_256(3, 3)
KVARN_DECODE_WIDTHS_256(3, 4)
KVARN_DECODE_WIDTHS_256(3, 5)
KVARN_DECODE_WIDTHS_256(3, 6)
KVARN_DECODE_WIDTHS_256(3, 8)
}  // namespace kvarn

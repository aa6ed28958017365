// Decode kernels at head_dim 256 with fp16 scales for key code width 8 and
// every value width; one translation unit per key width, so that the pairs
// compile in parallel.
#include "kvarn_decode_kernel.cuh"

namespace kvarn {
KVARN_DECODE_WIDTHS_256(8, 2)
KVARN_DECODE_WIDTHS_256(8, 3)
KVARN_DECODE_WIDTHS_256(8, 4)
KVARN_DECODE_WIDTHS_256(8, 5)
KVARN_DECODE_WIDTHS_256(8, 6)
KVARN_DECODE_WIDTHS_256(8, 8)
}  // namespace kvarn

// Encode kernels at head_dim 256 with fp16 scales for key code width 3 and
// every value width; one translation unit per key width, so that the pairs
// compile in parallel.
#include "kvarn_encode_kernel.cuh"

namespace kvarn {
KVARN_ENCODE_WIDTHS_256(3, 2)
KVARN_ENCODE_WIDTHS_256(3, 3)
KVARN_ENCODE_WIDTHS_256(3, 4)
KVARN_ENCODE_WIDTHS_256(3, 5)
KVARN_ENCODE_WIDTHS_256(3, 6)
KVARN_ENCODE_WIDTHS_256(3, 8)
}  // namespace kvarn

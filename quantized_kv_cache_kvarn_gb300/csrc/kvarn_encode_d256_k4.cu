// Encode kernels at head_dim 256 with fp16 scales for key code width 4 and
// every value width; one translation unit per key width, so that the pairs
// compile in parallel.
#include "kvarn_encode_kernel.cuh"

namespace kvarn {
KVARN_ENCODE_WIDTHS_256(4, 2)
KVARN_ENCODE_WIDTHS_256(4, 3)
KVARN_ENCODE_WIDTHS_256(4, 4)
KVARN_ENCODE_WIDTHS_256(4, 5)
KVARN_ENCODE_WIDTHS_256(4, 6)
KVARN_ENCODE_WIDTHS_256(4, 8)
}  // namespace kvarn

// Encode kernels at head_dim 256 with fp16 scales for key code width 2 and
// every value width; one translation unit per key width, so that the pairs
// compile in parallel.
#include "kvarn_encode_kernel.cuh"

namespace kvarn {
KVARN_ENCODE_WIDTHS_256(2, 2)
KVARN_ENCODE_WIDTHS_256(2, 3)
KVARN_ENCODE_WIDTHS_256(2, 4)
KVARN_ENCODE_WIDTHS_256(2, 5)
KVARN_ENCODE_WIDTHS_256(2, 6)
KVARN_ENCODE_WIDTHS_256(2, 8)
}  // namespace kvarn

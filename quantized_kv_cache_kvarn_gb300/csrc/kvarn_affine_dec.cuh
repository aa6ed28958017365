// Explicit instantiation of the affine comparison decode (the dense decode
// skeleton with the affine codec: per-token groups of 64 channels with an
// fp16 scale and offset each, original basis) for one code width, keys and
// values alike, head_dim 128 and 128-token tiles.
#pragma once

#include "kvarn_decode_kernel.cuh"

#define KVARN_AFFINE_DECODE(K)                                                                              \
  namespace kvarn {                                                                                         \
  template <>                                                                                               \
  cudaError_t run_affine_widths<K>(const DecArgs& A, bool /*bf16*/, int ctas, cudaStream_t st) {           \
    constexpr int W = width_warps<128, 128, K, K, 2, kCodecAffine>();                                       \
    return run_dense<128, 128, W, K, K, 2, kCodecAffine>(A, ctas, st);                       \
  }                                                                                                         \
  template <>                                                                                               \
  int resident_affine<K>() {                                                                                \
    return resident_dense<128, 128, width_warps<128, 128, K, K, 2, kCodecAffine>(), K, K, 2,       \
                          kCodecAffine>();                                                                  \
  }                                                                                                         \
  }

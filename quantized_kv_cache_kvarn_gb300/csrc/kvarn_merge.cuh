// Split-K merge and warp-wide Hadamard transform shared by the decode paths.
#pragma once

#include <math.h>

#include "kvarn_common.cuh"

namespace kvarn {

constexpr int kPStride(int D) { return D + 4; }  // m, l, pad, pad, acc[D]
constexpr float kLn2 = 0.6931471805599453f;

// In-place Hadamard transform (unscaled) of a vector spread over the warp:
// lane holds channels lane*E .. lane*E + E - 1.
template <int E>
__device__ __forceinline__ void warp_fwht(float* v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int h = 1; h < E; h <<= 1)
#pragma unroll
    for (int e = 0; e < E; ++e)
      if (!(e & h)) {
        float a = v[e], c = v[e + h];
        v[e] = a + c;
        v[e + h] = a - c;
      }
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const bool upper = lane & d;
#pragma unroll
    for (int e = 0; e < E; ++e) {
      float p = __shfl_xor_sync(0xffffffffu, v[e], d);
      v[e] = upper ? p - v[e] : v[e] + p;
    }
  }
}

// ------------------------------------------------------------------ merge
// One warp per (sequence, query head): LSE merge of all slots, inverse
// Hadamard of the rotated part (slots < nsplit), plus the tail slot.
template <int D>
__global__ void __launch_bounds__(128) merge_kernel(const float* __restrict__ ws, int slots,
                                                    int rows, int rotated_slots, float* out,
                                                    float* lse) {
  constexpr int E = D / 32;
  const int lane = threadIdx.x & 31;
  const int row = blockIdx.x * 4 + (threadIdx.x >> 5);
  if (row >= rows) return;
  const float* P = ws + static_cast<int64_t>(row) * slots * kPStride(D);
  float M = -INFINITY;
  for (int s = 0; s < slots; ++s) M = fmaxf(M, P[s * kPStride(D)]);
  float* o = out + static_cast<int64_t>(row) * D + lane * E;
  if (M == -INFINITY) {
#pragma unroll
    for (int e = 0; e < E; ++e) o[e] = 0.f;
    if (lse && lane == 0) lse[row] = -INFINITY;
    return;
  }
  float L = 0.f, rot[E], tl[E];
#pragma unroll
  for (int e = 0; e < E; ++e) rot[e] = tl[e] = 0.f;
  for (int s = 0; s < slots; ++s) {
    const float* p = P + s * kPStride(D);
    const float w = exp2f(p[0] - M);
    L = fmaf(p[1], w, L);
    float* dst = s < rotated_slots ? rot : tl;
#pragma unroll
    for (int e = 0; e < E; e += 4) {
      const float4 v = *reinterpret_cast<const float4*>(p + 4 + lane * E + e);
      dst[e] = fmaf(v.x, w, dst[e]);
      dst[e + 1] = fmaf(v.y, w, dst[e + 1]);
      dst[e + 2] = fmaf(v.z, w, dst[e + 2]);
      dst[e + 3] = fmaf(v.w, w, dst[e + 3]);
    }
  }
  const float invL = 1.f / L;
  warp_fwht<E>(rot);
  const float sc = invL / sqrtf(static_cast<float>(D));
#pragma unroll
  for (int e = 0; e < E; ++e) o[e] = fmaf(rot[e], sc, tl[e] * invL);
  if (lse && lane == 0) lse[row] = (M + log2f(L)) * kLn2;
}

}  // namespace kvarn

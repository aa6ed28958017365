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
// dst = sum over slots [s0, s1) of exp2(m_s - M) * (this lane's part of the
// slot vector); every lane reads the slot maxima (one broadcast load each),
// and several slot vectors are in flight at once.
template <int E>
__device__ __forceinline__ void accumulate_slots(const float* P, int stride, int s0, int s1, float M,
                                                 float (&dst)[E]) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int e = 0; e < E; ++e) dst[e] = 0.f;
#pragma unroll 4
  for (int s = s0; s < s1; ++s) {
    const float* p = P + static_cast<int64_t>(s) * stride;
    const float w = exp2f(p[0] - M);
    p += 4 + lane * E;
#pragma unroll
    for (int e = 0; e < E; e += 4) {
      const float4 v = *reinterpret_cast<const float4*>(p + e);
      dst[e] = fmaf(v.x, w, dst[e]);
      dst[e + 1] = fmaf(v.y, w, dst[e + 1]);
      dst[e + 2] = fmaf(v.z, w, dst[e + 2]);
      dst[e + 3] = fmaf(v.w, w, dst[e + 3]);
    }
  }
}

// One warp per (sequence, query head): LSE merge of the row's partials, the
// rotated ones (slots [0, counts[row]), or [0, rotated_slots) without
// counts) through the inverse Hadamard transform, plus the raw ones (slots
// [raw_begin, slots)). The lanes read the slot maxima and sums in parallel.
// ROT = false: the tile partials are in the original basis too (the affine
// comparison codec) and are added without the transform.
template <int D, bool ROT = true>
__global__ void __launch_bounds__(128) merge_kernel(const float* __restrict__ ws, int slots, int rows,
                                                    const int32_t* __restrict__ counts, int rotated_slots,
                                                    int raw_begin, float* out, float* lse) {
  constexpr int E = D / 32;
  pdl_wait_primary();
  const int lane = threadIdx.x & 31;
  const int row = blockIdx.x * 4 + (threadIdx.x >> 5);
  if (row >= rows) return;
  const int rot_end = counts ? min(counts[row], raw_begin) : rotated_slots;
  auto used = [&](int s) { return s < rot_end || s >= raw_begin; };
  const float* P = ws + static_cast<int64_t>(row) * slots * kPStride(D);
  float M = -INFINITY;
  for (int s = lane; s < slots; s += 32)
    if (used(s)) M = fmaxf(M, P[s * kPStride(D)]);
  M = warp_max_xor(M, 1, 32);
  float* o = out + static_cast<int64_t>(row) * D + lane * E;
  if (M == -INFINITY) {
#pragma unroll
    for (int e = 0; e < E; ++e) o[e] = 0.f;
    if (lse && lane == 0) lse[row] = -INFINITY;
    return;
  }
  float L = 0.f, rot[E], tl[E];
  for (int s = lane; s < slots; s += 32)
    if (used(s)) L = fmaf(P[s * kPStride(D) + 1], exp2f(P[s * kPStride(D)] - M), L);
  accumulate_slots<E>(P, kPStride(D), 0, rot_end, M, rot);
  accumulate_slots<E>(P, kPStride(D), raw_begin, slots, M, tl);
  L = warp_sum_xor(L, 1, 32);
  const float invL = 1.f / L;
  if constexpr (ROT) warp_fwht<E>(rot);
  const float sc = ROT ? invL / sqrtf(static_cast<float>(D)) : invL;
#pragma unroll
  for (int e = 0; e < E; ++e) o[e] = fmaf(rot[e], sc, tl[e] * invL);
  if (lse && lane == 0) lse[row] = (M + log2f(L)) * kLn2;
}

// Launches the merge as a programmatic dependent of the kernel before it on
// the stream.
template <int D, bool ROT = true>
cudaError_t launch_merge(const float* ws, int slots, int rows, const int32_t* counts, int rotated_slots,
                         int raw_begin, float* out, float* lse, cudaStream_t st) {
  if (rows <= 0) return cudaSuccess;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((rows + 3) / 4);
  cfg.blockDim = dim3(128);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, merge_kernel<D, ROT>, ws, slots, rows, counts, rotated_slots, raw_begin, out, lse);
}

}  // namespace kvarn

// The affine comparison codec (gmlx "KV cache quantization" page, "The two
// schemes": mlx-lm's quantized cache stores, per token, groups of 64 values
// as N-bit codes with an fp16 scale and offset per group) on this library's
// paged skeleton: the encoder below, and the decode through the dense decode
// kernel with the affine codec (kvarn_affine_dec.cuh). It is the fidelity
// and speed comparison for the KVarN codec: no rotation, no normalisation.
#include <atomic>

#include "kvarn_decode_kernel.cuh"
#include "kvarn_encode_kernel.cuh"

namespace kvarn {

namespace {

// Round-half-to-even of the exact quotient (v - of) / sc clamped to
// [0, qmax], x = (v - of) * rinv as formed by the caller: the exact side of
// a half-way point is taken as in grid_boundary_code, with a signed code
// (the stored fp16 offset may lie above some of the group's values, and the
// rounded fp16 step may make the largest quotient pass qmax).
__device__ __forceinline__ int affine_code(float v, float of, float sc, float x, int qmax) {
  const float r = rintf(x);
  int q = static_cast<int>(r);
  if (fabsf(x - r) > 0.5f - 0x1p-14f) {
    const float s = __fadd_rn(v, -of);
    const float bb = __fsub_rn(s, v);
    const float e = __fadd_rn(__fsub_rn(v, __fsub_rn(s, bb)), __fsub_rn(-of, bb));
    const float k = floorf(x);
    const float w = __fadd_rn(__fmaf_rn(-(k + 0.5f), sc, s), e);
    const int ki = static_cast<int>(k);
    q = ki + ((w > 0.f || (w == 0.f && (ki & 1))) ? 1 : 0);
  }
  return min(max(q, 0), qmax);
}

// Shared memory of one affine tile (N tokens of one KV head, one of K or V):
// the codes as bytes [N][D], the plane words of its pages, the per-token
// records [N][2G] fp16, the page addresses.
template <int D, int N, int BITS>
struct AffShape {
  static constexpr int G = D / 64;
  static constexpr int PPT = N / kPageTokens;
  static constexpr int OFF_IMG = N * D;
  static constexpr int OFF_REC = OFF_IMG + N * D * BITS / 8;
  static constexpr int OFF_PAGES = OFF_REC + N * 4 * G;
  static constexpr int SMEM = OFF_PAGES + 8 * PPT;
};

// One thread per token: the group minimum and maximum, the fp16 step
// (max - min) / (2^bits - 1) rounded once from float64 and the fp16 offset
// min, the codes against those stored values, then the page's plane words
// and records.
template <int D, int N, typename T, int BITS, bool IS_V, int KB, int VB>
__device__ __forceinline__ void affine_tile(const EncodeArgs& A, const T* __restrict__ src, int b, int head,
                                            int64_t tile, unsigned char* smem) {
  using S = AffShape<D, N, BITS>;
  constexpr AffinePage AG{D, KB, VB};
  constexpr int G = S::G, QMAX = (1 << BITS) - 1;
  const int tid = threadIdx.x;
  unsigned char* cb = smem;
  uint32_t* img = reinterpret_cast<uint32_t*>(smem + S::OFF_IMG);
  __half* rec = reinterpret_cast<__half*>(smem + S::OFF_REC);
  uint8_t** pages = reinterpret_cast<uint8_t**>(smem + S::OFF_PAGES);
  if (tid < S::PPT) {
    const int64_t lp = tile * S::PPT + tid;
    uint8_t* pg = nullptr;
    const int32_t phys =
        (lp >= 0 && lp < A.bt_stride) ? A.block_table[static_cast<int64_t>(b) * A.bt_stride + lp] : -1;
    if (phys >= 0 && phys < A.num_pages)
      pg = A.cache + (static_cast<int64_t>(phys) * A.num_kv_heads + head) * A.page_bytes;
    else
      set_error(A.err, KVARN_DEVERR_PAGE_RANGE);
    pages[tid] = pg;
  }
  const T* row = src + static_cast<int64_t>(tid) * D;
#pragma unroll 1
  for (int gr = 0; gr < G; ++gr) {
    float v[64];
#pragma unroll
    for (int k = 0; k < 8; ++k) load8<T>(row + 64 * gr + 8 * k, v + 8 * k);
    float lo = v[0], hi = v[0];
#pragma unroll
    for (int j = 1; j < 64; ++j) {
      lo = fminf(lo, v[j]);
      hi = fmaxf(hi, v[j]);
    }
    const __half sc16 = __double2half((static_cast<double>(hi) - static_cast<double>(lo)) / QMAX);
    const __half of16 = __float2half_rn(lo);
    const float sc = __half2float(sc16), of = __half2float(of16);
    const float rinv = sc > 0.f ? 1.f / sc : 0.f;
#pragma unroll
    for (int j = 0; j < 64; j += 4) {
      uint32_t w = 0;
#pragma unroll
      for (int e = 0; e < 4; ++e)
        w |= static_cast<uint32_t>(affine_code(v[j + e], of, sc, (v[j + e] - of) * rinv, QMAX)) << (8 * e);
      *reinterpret_cast<uint32_t*>(cb + tid * D + 64 * gr + j) = w;
    }
    rec[tid * 2 * G + gr] = sc16;
    rec[tid * 2 * G + G + gr] = of16;
  }
  __syncthreads();
  pack_plane_words<D, BITS, IS_V>(cb, img, S::PPT, tid, N);
  __syncthreads();
  // codes, then the token records, in 16-byte stores
  constexpr int CPP = 2 * D * BITS / 16;
  const int cbase = IS_V ? AG.k_part() : 0;
  for (int c = tid; c < S::PPT * CPP; c += N) {
    uint8_t* pg = pages[c / CPP];
    if (pg) reinterpret_cast<uint4*>(pg + cbase)[c % CPP] = reinterpret_cast<const uint4*>(img)[c];
  }
  constexpr int RPP = 4 * G * kPageTokens / 16;
  const int rbase = IS_V ? AG.k_part() + AG.v_sc() : AG.k_sc();
  for (int c = tid; c < S::PPT * RPP; c += N) {
    uint8_t* pg = pages[c / RPP];
    if (pg) reinterpret_cast<uint4*>(pg + rbase)[c % RPP] = reinterpret_cast<const uint4*>(rec)[c];
  }
}

// K and V tiles of the chunk: blockIdx.z < num_seqs encodes K, the rest V.
template <int D, int N, typename T, int KB, int VB>
__global__ void __launch_bounds__(N) encode_affine_kernel(EncodeArgs A) {
  extern __shared__ __align__(128) unsigned char smem[];
  pdl_launch_dependents();
  const bool is_v = static_cast<int>(blockIdx.z) >= A.num_seqs;
  const int u = blockIdx.x, head = blockIdx.y, b = blockIdx.z - (is_v ? A.num_seqs : 0);
  if (A.tile_start[b] < 0) return;
  const int64_t off = static_cast<int64_t>(b) * A.seq_stride + static_cast<int64_t>(head) * A.head_stride +
                      static_cast<int64_t>(u) * N * D;
  if (is_v)
    affine_tile<D, N, T, VB, true, KB, VB>(A, static_cast<const T*>(A.x[1]) + off, b, head, A.tile_start[b] + u,
                                           smem);
  else
    affine_tile<D, N, T, KB, false, KB, VB>(A, static_cast<const T*>(A.x[0]) + off, b, head, A.tile_start[b] + u,
                                            smem);
}

template <int K, typename T>
cudaError_t launch_affine_w(const EncodeArgs& A, cudaStream_t st) {
  constexpr int smem = AffShape<128, 128, K>::SMEM;
  auto kern = encode_affine_kernel<128, 128, T, K, K>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  dim3 grid(A.chunk_tiles, A.num_kv_heads, 2 * A.num_seqs);
  kern<<<grid, 128, smem, st>>>(A);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_encode_affine(const EncodeParams& p, cudaStream_t st) {
  if (p.D != 128 || p.N != 128 || p.k_bits != p.v_bits) return cudaErrorInvalidValue;
  EncodeArgs A{};
  A.x[0] = p.k;
  A.x[1] = p.v;
  A.seq_stride = p.seq_stride;
  A.head_stride = p.head_stride;
  A.chunk_tiles = p.chunk_tokens / p.N;
  A.tile_start = p.tile_start;
  A.block_table = p.block_table;
  A.bt_stride = p.bt_stride;
  A.cache = static_cast<uint8_t*>(p.cache);
  A.num_pages = p.num_pages;
  A.num_kv_heads = p.num_kv_heads;
  A.page_bytes = AffinePage(p.D, p.k_bits, p.v_bits).bytes();
  A.err = p.err;
  A.num_seqs = p.num_seqs;
  if (A.chunk_tiles == 0 || p.num_seqs == 0) return cudaSuccess;
  switch (p.k_bits) {
#define KVARN_AFF_ENC(K)                                                                      \
  case K:                                                                                     \
    return p.bf16 ? launch_affine_w<K, __nv_bfloat16>(A, st) : launch_affine_w<K, __half>(A, st);
    KVARN_AFFINE_WIDTHS(KVARN_AFF_ENC)
#undef KVARN_AFF_ENC
    default: return cudaErrorInvalidValue;
  }
}

int affine_decode_ctas_per_sm(int32_t bits) {
  static std::atomic<int> cache[9] = {};
  if (bits < 0 || bits > 8) return 1;
  const int known = cache[bits].load(std::memory_order_relaxed);
  if (known) return known;
  int c = 1;
  switch (bits) {
#define KVARN_AFF_RES(K) \
  case K: c = resident_affine<K>(); break;
    KVARN_AFFINE_WIDTHS(KVARN_AFF_RES)
#undef KVARN_AFF_RES
    default: break;
  }
  cache[bits].store(c, std::memory_order_relaxed);
  return c;
}

}  // namespace kvarn

// KVarN tile encoder: launchers (kernels in kvarn_encode_kernel.cuh; the
// k4v2 preset with fp32 scales, the latent and the append kernels are
// instantiated here, other code widths in kvarn_encode_k*{lo,hi}.cu and
// kvarn_encode_d256{a,b}.cu).
#include "kvarn_encode_kernel.cuh"

namespace kvarn {

// ------------------------------------------------------------- launchers

template <int D, int N>
static cudaError_t launch_dense_w(const EncodeArgs& A, const EncodeParams& p, cudaStream_t st) {
  const int kb = p.k_bits, vb = p.v_bits, sb = p.scale_bytes;
  if (kb == 4 && vb == 2 && sb == 4)
    return launch_dense<D, N>(A, st);
  if constexpr (D == 128) {
    if (sb == 4) {
      switch (16 * kb + vb) {
#define KVARN_ENC_CASE(K, V) \
  case 16 * K + V: return launch_encode_widths<K, V, 4>(A, N, p.bf16, st);
        KVARN_WIDTH_PAIRS_S32(KVARN_ENC_CASE)
#undef KVARN_ENC_CASE
        default: return cudaErrorInvalidValue;
      }
    }
  }
  if (sb != 2) return cudaErrorInvalidValue;
  if constexpr (D == 256) {
    switch (16 * kb + vb) {
#define KVARN_ENC_CASE(K, V) \
  case 16 * K + V: return launch_encode_widths256<K, V, 2>(A, N, p.bf16, st);
      KVARN_WIDTH_PAIRS_256(KVARN_ENC_CASE)
#undef KVARN_ENC_CASE
      default: return cudaErrorInvalidValue;
    }
  }
  if (D != 128) return cudaErrorInvalidValue;
  switch (16 * kb + vb) {
#define KVARN_ENC_CASE(K, V) \
  case 16 * K + V: return launch_encode_widths<K, V, 2>(A, N, p.bf16, st);
    KVARN_WIDTH_PAIRS(KVARN_ENC_CASE)
#undef KVARN_ENC_CASE
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_encode_dense(const EncodeParams& p, cudaStream_t st) {
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
  A.page_bytes = DensePage(p.D, p.N, p.k_bits, p.v_bits, p.scale_bytes).bytes();
  A.norm_iters = p.norm_iters;
  A.err = p.err;
  A.num_seqs = p.num_seqs;
  A.stages = p.stages;
  A.bf16 = p.bf16 ? 1 : 0;
  if (A.chunk_tiles == 0 || p.num_seqs == 0) return cudaSuccess;
  if (p.D == 128 && p.N == 128) return launch_dense_w<128, 128>(A, p, st);
  if (p.D == 128 && p.N == 64) return launch_dense_w<128, 64>(A, p, st);
  if (p.D == 256 && p.N == 128) return launch_dense_w<256, 128>(A, p, st);
  if (p.D == 256 && p.N == 64) return launch_dense_w<256, 64>(A, p, st);
  return cudaErrorInvalidValue;
}

template <int D, int N>
static cudaError_t launch_append(const EncodeArgs& A, const AppendParams& p, cudaStream_t st) {
  constexpr int smem = EncShape<D, N, 1>::SMEM;
  auto kern = append_commit_kernel<D, N>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  dim3 grid(A.num_kv_heads, p.num_seqs, 2);
  kern<<<grid, 2 * D, smem, st>>>(A, p.seq_lens, p.max_seq_len, static_cast<unsigned char*>(p.tail_k),
                                  static_cast<unsigned char*>(p.tail_v));
  return cudaGetLastError();
}

cudaError_t launch_append_commit(const AppendParams& p, cudaStream_t st) {
  if (p.num_seqs == 0) return cudaSuccess;
  EncodeArgs A{};
  A.x[0] = p.k;
  A.x[1] = p.v;
  A.block_table = p.block_table;
  A.bt_stride = p.bt_stride;
  A.cache = static_cast<uint8_t*>(p.cache);
  A.num_pages = p.num_pages;
  A.num_kv_heads = p.num_kv_heads;
  A.page_bytes = DensePage(p.D, p.N).bytes();
  A.norm_iters = p.norm_iters;
  A.err = p.err;
  A.num_seqs = p.num_seqs;
  A.bf16 = p.bf16 ? 1 : 0;
#define KV_DISPATCH(DD, NN) \
  if (p.D == DD && p.N == NN) return launch_append<DD, NN>(A, p, st);
  KV_DISPATCH(128, 128)
  KV_DISPATCH(128, 64)
  KV_DISPATCH(256, 128)
  KV_DISPATCH(256, 64)
#undef KV_DISPATCH
  return cudaErrorInvalidValue;
}

// The MLA latent: head_dim 512 as a cluster of two CTAs that split the tile's
// rows (4-bit codes, one code set for keys and values).
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(512)
    encode_latent_kernel(EncodeArgs A) {
  extern __shared__ __align__(128) unsigned char smem[];
  const int u = blockIdx.x >> 1, b = blockIdx.y;
  if (A.tile_start[b] < 0) return;  // uniform over the cluster: both CTAs share b
  const unsigned char* src = static_cast<const unsigned char*>(A.x[0]) +
                             2 * (static_cast<int64_t>(b) * A.seq_stride + static_cast<int64_t>(u) * 128 * 512);
  encode_tile<512, 128, 2, 4, 1>(A, src, b, 0, u, A.tile_start[b] + u, nullptr, smem);
}

cudaError_t launch_encode_latent(const EncodeLatentParams& p, cudaStream_t st) {
  EncodeArgs A{};
  A.x[0] = p.latent;
  A.rope = static_cast<const __half*>(p.rope);
  A.seq_stride = p.seq_stride;
  A.rope_seq_stride = p.rope_seq_stride;
  A.chunk_tiles = p.chunk_tokens / 128;
  A.tile_start = p.tile_start;
  A.block_table = p.block_table;
  A.bt_stride = p.bt_stride;
  A.cache = static_cast<uint8_t*>(p.cache);
  A.num_pages = p.num_pages;
  A.num_kv_heads = 1;
  A.page_bytes = LatentPage(512, 64, 128).bytes();
  A.norm_iters = p.norm_iters;
  A.rope_dim = 64;
  A.err = p.err;
  A.num_seqs = p.num_seqs;
  A.bf16 = p.bf16 ? 1 : 0;
  if (A.chunk_tiles == 0 || p.num_seqs == 0) return cudaSuccess;
  constexpr int smem = EncShape<512, 128, 2>::SMEM;
  auto kern = encode_latent_kernel;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  dim3 grid(2 * A.chunk_tiles, p.num_seqs);
  kern<<<grid, 512, smem, st>>>(A);
  return cudaGetLastError();
}

}  // namespace kvarn

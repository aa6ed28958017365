// KVarN tile encoder for sm_103a.
//
// KVarN review ("KVarN ... vLLM KV cache quantization"), four-stage
// paragraph: rotate each tile by an orthonormal Hadamard matrix across the
// channels, run T alternating column/row standard-deviation normalisations
// with the scales in log space, then asymmetric round-to-nearest with the
// scales folded into the stored row offsets. One CTA (or a cluster of two
// for head_dim 512) owns one N x D tile and keeps it in registers: every
// thread holds a 16-channel segment of N/32 token rows. The Hadamard
// transform runs as four in-register butterfly stages and log2(D/16) lane
// shuffles; column statistics reduce through shared memory (and the peer
// CTA's shared memory in a cluster); row statistics reduce with shuffles.
// Codes are staged in shared memory as bytes and then packed into the page
// format that the decode kernel reads as mma fragments.
#include <cooperative_groups.h>

#include "kvarn_common.cuh"
#include "kvarn_launch.h"

namespace cg = cooperative_groups;

namespace kvarn {

// Cluster size 2 splits the tile's rows over two CTAs (head_dim 512, where a
// whole 128 x 512 fp32 tile would not fit one CTA's registers).
template <int D, int N, int CS>
struct EncShape {
  static constexpr int NT = 2 * D / CS;       // threads per CTA
  static constexpr int TPR = D / 16;          // threads per token row
  static constexpr int RPW = 32 / TPR;        // rows per warp and pass
  static constexpr int NW = NT / 32;          // warps
  static constexpr int ROWS = N / CS;         // rows owned by this CTA
  static constexpr int RPT = N / 32;          // rows per thread
  static_assert(ROWS == RPT * NW * RPW, "tile rows must cover the CTA");
  static constexpr int RED_BYTES = NW * D * 4;
  static constexpr int CODE_BYTES = ROWS * D;
  static constexpr int SCRATCH = RED_BYTES > CODE_BYTES ? RED_BYTES : CODE_BYTES;
  // scratch | colbuf[D] | rowA[ROWS] | rowB[ROWS] | colC[D] | colpart[2][D] (cluster)
  static constexpr int SMEM = SCRATCH + 4 * D + 8 * ROWS + 4 * D + 8 * D;
};

struct EncodeArgs {
  const void* x[2];        // K, V (dense) or latent (x[0])
  const __half* rope;      // latent only
  int64_t seq_stride, head_stride, rope_seq_stride;
  int32_t chunk_tiles;
  const int32_t* tile_start;
  const int32_t* block_table;
  int32_t bt_stride;
  uint8_t* cache;
  int64_t num_pages;
  int32_t num_kv_heads;
  int32_t page_bytes;
  int32_t norm_iters;
  int32_t rope_dim;
  uint32_t* err;
};

// Column statistic: every thread passes its 16 per-channel partial sums over
// its rows; returns the full sums over the tile (all CS CTAs) for its 16
// channels.
template <int D, int N, int CS>
__device__ __forceinline__ void column_sum(float (&s)[16], float* red, float* colbuf,
                                           float* colpart) {
  using S = EncShape<D, N, CS>;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, seg = lane % S::TPR;
#pragma unroll
  for (int e = 0; e < 16; ++e)
    for (int o = S::TPR; o < 32; o <<= 1) s[e] += __shfl_xor_sync(0xffffffffu, s[e], o);
  if (lane < S::TPR) {
    float4* dst = reinterpret_cast<float4*>(red + warp * D + seg * 16);
#pragma unroll
    for (int e = 0; e < 4; ++e) dst[e] = make_float4(s[4 * e], s[4 * e + 1], s[4 * e + 2], s[4 * e + 3]);
  }
  __syncthreads();
  if (threadIdx.x < D) {
    float t = 0.f;
#pragma unroll 8
    for (int w = 0; w < S::NW; ++w) t += red[w * D + threadIdx.x];
    if constexpr (CS == 1) {
      colbuf[threadIdx.x] = t;
    } else {
      colpart[threadIdx.x] = t;
    }
  }
  if constexpr (CS == 1) {
    __syncthreads();
  } else {
    cg::cluster_group cl = cg::this_cluster();
    cl.sync();
    if (threadIdx.x < D) {
      float own = colpart[threadIdx.x];
      float* peer = cl.map_shared_rank(colpart, cl.block_rank() ^ 1);
      float other = peer[threadIdx.x];
      // both CTAs add in rank order, so they hold bit-identical sums
      colbuf[threadIdx.x] = cl.block_rank() == 0 ? own + other : other + own;
    }
    cl.sync();
  }
  const float4* src = reinterpret_cast<const float4*>(colbuf + seg * 16);
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    float4 v = src[e];
    s[4 * e] = v.x; s[4 * e + 1] = v.y; s[4 * e + 2] = v.z; s[4 * e + 3] = v.w;
  }
}

// Population std; 1 for a numerically constant vector (std <= 2^-20 |mean|,
// which covers the rounding residue of an exactly constant one) or a
// non-finite std.
__device__ __forceinline__ float safe_sigma(float var, float mean) {
  const float s = sqrtf(var);
  return (isfinite(s) && s > 9.5367431640625e-07f * fabsf(mean)) ? s : 1.f;
}

template <int D, int N, int CS, int BITS, int KIND, typename T>
__device__ __forceinline__ void encode_tile(const EncodeArgs& A, const T* __restrict__ src,
                                            int b, int head, int u, int which,
                                            unsigned char* smem) {
  using S = EncShape<D, N, CS>;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int seg = lane % S::TPR, rsub = lane / S::TPR;
  int crank = 0;
  if constexpr (CS > 1) crank = static_cast<int>(cg::this_cluster().block_rank());

  float* red = reinterpret_cast<float*>(smem);
  unsigned char* codes = smem;  // aliases red once the statistics are done
  float* colbuf = reinterpret_cast<float*>(smem + S::SCRATCH);
  float* rowA = colbuf + D;
  float* rowB = rowA + S::ROWS;
  float* colC = rowB + S::ROWS;
  float* colpart = colC + D;

  // ---- load: row r_local(i) = i*32 + warp*RPW + rsub (within this CTA's rows)
  float x[S::RPT][16];
#pragma unroll
  for (int i = 0; i < S::RPT; ++i) {
    const int r = crank * S::ROWS + i * (S::NW * S::RPW) + warp * S::RPW + rsub;
    const T* p = src + static_cast<int64_t>(r) * D + seg * 16;
    load8<T>(p, x[i]);
    load8<T>(p + 8, x[i] + 8);
  }

  // ---- Hadamard: 4 in-register stages, then lane butterflies, then 1/sqrt(D)
#pragma unroll
  for (int i = 0; i < S::RPT; ++i) {
#pragma unroll
    for (int h = 1; h < 16; h <<= 1)
#pragma unroll
      for (int e = 0; e < 16; ++e)
        if (!(e & h)) {
          float a = x[i][e], c = x[i][e + h];
          x[i][e] = a + c;
          x[i][e + h] = a - c;
        }
  }
#pragma unroll
  for (int d = 1; d < S::TPR; d <<= 1) {
    const bool upper = lane & d;
#pragma unroll
    for (int i = 0; i < S::RPT; ++i)
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        float p = __shfl_xor_sync(0xffffffffu, x[i][e], d);
        x[i][e] = upper ? p - x[i][e] : x[i][e] + p;
      }
  }

  {
    const float rsd = 1.f / sqrtf(static_cast<float>(D));
#pragma unroll
    for (int i = 0; i < S::RPT; ++i)
#pragma unroll
      for (int e = 0; e < 16; ++e) x[i][e] *= rsd;
  }

  // ---- variance normalisation, T iterations of (column pass, row pass)
  float logc[16], logr[S::RPT];
#pragma unroll
  for (int e = 0; e < 16; ++e) logc[e] = 0.f;
#pragma unroll
  for (int i = 0; i < S::RPT; ++i) logr[i] = 0.f;
  const float invN = 1.f / N, invD = 1.f / D;

  for (int it = 0; it < A.norm_iters; ++it) {
    float s[16];
#pragma unroll
    for (int e = 0; e < 16; ++e) {
      float t = 0.f;
#pragma unroll
      for (int i = 0; i < S::RPT; ++i) t += x[i][e];
      s[e] = t;
    }
    column_sum<D, N, CS>(s, red, colbuf, colpart);
    float mean[16];
#pragma unroll
    for (int e = 0; e < 16; ++e) {
      mean[e] = s[e] * invN;
      float t = 0.f;
#pragma unroll
      for (int i = 0; i < S::RPT; ++i) {
        float dv = x[i][e] - mean[e];
        t = fmaf(dv, dv, t);
      }
      s[e] = t;
    }
    __syncthreads();  // red is reused
    column_sum<D, N, CS>(s, red, colbuf, colpart);
#pragma unroll
    for (int e = 0; e < 16; ++e) {
      const float sig = safe_sigma(s[e] * invN, mean[e]);
      logc[e] += logf(sig);
      const float inv = 1.f / sig;
#pragma unroll
      for (int i = 0; i < S::RPT; ++i) x[i][e] *= inv;
    }
    // row pass: a row lives in TPR consecutive lanes
#pragma unroll
    for (int i = 0; i < S::RPT; ++i) {
      float t = 0.f;
#pragma unroll
      for (int e = 0; e < 16; ++e) t += x[i][e];
      t = warp_sum_xor(t, 1, S::TPR);
      const float m = t * invD;
      float v = 0.f;
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        float dv = x[i][e] - m;
        v = fmaf(dv, dv, v);
      }
      v = warp_sum_xor(v, 1, S::TPR);
      const float sig = safe_sigma(v * invD, m);
      logr[i] += logf(sig);
      const float inv = 1.f / sig;
#pragma unroll
      for (int e = 0; e < 16; ++e) x[i][e] *= inv;
    }
    __syncthreads();
  }

  // ---- asymmetric RTN per row
  constexpr int QMAX = (1 << BITS) - 1;
#pragma unroll
  for (int i = 0; i < S::RPT; ++i) {
    float lo = x[i][0], hi = x[i][0];
#pragma unroll
    for (int e = 1; e < 16; ++e) {
      lo = fminf(lo, x[i][e]);
      hi = fmaxf(hi, x[i][e]);
    }
    for (int o = 1; o < S::TPR; o <<= 1) {
      lo = fminf(lo, __shfl_xor_sync(0xffffffffu, lo, o));
      hi = fmaxf(hi, __shfl_xor_sync(0xffffffffu, hi, o));
    }
    const float delta = (hi - lo) / static_cast<float>(QMAX);
    const float inv = delta > 0.f ? 1.f / delta : 0.f;
    uint32_t w[4] = {0u, 0u, 0u, 0u};
#pragma unroll
    for (int e = 0; e < 16; ++e) {
      int q = __float2int_rn((x[i][e] - lo) * inv);
      q = min(max(q, 0), QMAX);
      w[e >> 2] |= static_cast<uint32_t>(q) << (8 * (e & 3));
    }
    const int r = i * (S::NW * S::RPW) + warp * S::RPW + rsub;  // local row
    *reinterpret_cast<uint4*>(codes + r * D + seg * 16) = make_uint4(w[0], w[1], w[2], w[3]);
    if (seg == 0) {
      const float rr = expf(logr[i]);
      rowA[r] = rr * (delta > 0.f ? delta : 0.f);
      rowB[r] = rr * lo;
    }
  }
  if (warp == 0 && rsub == 0) {
#pragma unroll
    for (int e = 0; e < 16; ++e) colC[seg * 16 + e] = expf(logc[e]);
  }
  __syncthreads();

  // ---- page addresses of this CTA's rows
  constexpr int PPT = N / kPageTokens;            // pages per tile
  constexpr int PPC = PPT / CS;                   // pages per CTA
  const int64_t lt = static_cast<int64_t>(A.tile_start[b]) + u;
  const int32_t* bt = A.block_table + static_cast<int64_t>(b) * A.bt_stride;

  auto page_ptr = [&](int p_local) -> uint8_t* {
    const int64_t lp = lt * PPT + crank * PPC + p_local;
    const int32_t phys = bt[lp];
    if (phys < 0 || phys >= A.num_pages) return nullptr;
    return A.cache + (static_cast<int64_t>(phys) * A.num_kv_heads + head) * A.page_bytes;
  };

  // ---- pack codes
  if constexpr (BITS == 4) {
    // dense K or latent: per page 2D words; a thread builds 4 words (16 B)
    constexpr int CHUNKS = PPC * 2 * D / 4;
    for (int c = tid; c < CHUNKS; c += S::NT) {
      const int W0 = c * 4;
      const int p = W0 / (2 * D), win0 = W0 % (2 * D);
      uint8_t* pg = page_ptr(p);
      if (!pg) {
        set_error(A.err, KVARN_DEVERR_PAGE_RANGE);
        continue;
      }
      uint32_t out[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int win = win0 + k;
        const int tau = win / (D / 8), rem = win % (D / 8);
        const int t = rem / (D / 32), w = rem % (D / 32);
        const unsigned char* row = codes + (p * kPageTokens + tau) * D;
        uint32_t word = 0;
#pragma unroll
        for (int n = 0; n < 8; ++n) {
          const int ch = 16 * (2 * w + ((n & 3) >> 1)) + 2 * t + 8 * (n & 1) + (n >> 2);
          word |= static_cast<uint32_t>(row[ch]) << (4 * n);
        }
        out[k] = word;
      }
      *reinterpret_cast<uint4*>(pg + 4 * win0) = make_uint4(out[0], out[1], out[2], out[3]);
    }
  } else {
    // dense V: per page D words
    constexpr int CHUNKS = PPC * D / 4;
    const int base = DensePage(D, N).v_codes();
    for (int c = tid; c < CHUNKS; c += S::NT) {
      const int W0 = c * 4;
      const int p = W0 / D, win0 = W0 % D;
      uint8_t* pg = page_ptr(p);
      if (!pg) {
        set_error(A.err, KVARN_DEVERR_PAGE_RANGE);
        continue;
      }
      uint32_t out[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int win = win0 + k;
        const int L = win / (D / 32), w = win % (D / 32);
        const int g = L >> 2, t = L & 3;
        uint32_t word = 0;
#pragma unroll
        for (int pp = 0; pp < 8; ++pp)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int nc = 4 * w + (pp >> 1), h = pp & 1;
            const int tau = 2 * t + e + 8 * h;
            const int ch = 8 * nc + g;
            word |= static_cast<uint32_t>(codes[(p * kPageTokens + tau) * D + ch]) << (2 * pp + 16 * e);
          }
        out[k] = word;
      }
      *reinterpret_cast<uint4*>(pg + base + 4 * win0) = make_uint4(out[0], out[1], out[2], out[3]);
    }
  }

  // ---- scales
  int off_a, off_b, off_c;
  if constexpr (KIND == 1) {
    constexpr LatentPage L(D, 64, N);
    off_a = L.a(); off_b = L.b(); off_c = L.col();
  } else {
    constexpr DensePage P(D, N);
    off_a = which ? P.v_a() : P.k_a();
    off_b = which ? P.v_b() : P.k_b();
    off_c = which ? P.v_col() : P.k_col();
  }
  if (tid < S::ROWS) {
    uint8_t* pg = page_ptr(tid / kPageTokens);
    if (pg) {
      reinterpret_cast<float*>(pg + off_a)[tid % kPageTokens] = rowA[tid];
      reinterpret_cast<float*>(pg + off_b)[tid % kPageTokens] = rowB[tid];
    }
  }
  {
    constexpr int C = D * kPageTokens / N;  // column scales per page
    for (int j = tid; j < PPC * C; j += S::NT) {
      uint8_t* pg = page_ptr(j / C);
      if (pg) reinterpret_cast<float*>(pg + off_c)[j % C] = colC[(crank * PPC) * C + j];
    }
  }
  if constexpr (KIND == 1) {
    // rope rows, fp16, copied as is
    constexpr LatentPage L(D, 64, N);
    const int R = A.rope_dim;
    const int vec_per_page = kPageTokens * R * 2 / 16;
    for (int c = tid; c < PPC * vec_per_page; c += S::NT) {
      const int p = c / vec_per_page, k = c % vec_per_page;
      uint8_t* pg = page_ptr(p);
      if (!pg) continue;
      const int row = crank * S::ROWS + p * kPageTokens;  // first token of the page in the tile
      const uint8_t* s = reinterpret_cast<const uint8_t*>(
          A.rope + static_cast<int64_t>(b) * A.rope_seq_stride + (static_cast<int64_t>(u) * N + row) * R);
      reinterpret_cast<uint4*>(pg + L.rope())[k] = __ldg(reinterpret_cast<const uint4*>(s) + k);
    }
  }
}

template <int D, int N, typename T>
__global__ void __launch_bounds__(2 * D) encode_dense_kernel(EncodeArgs A) {
  extern __shared__ __align__(16) unsigned char smem[];
  const int u = blockIdx.x >> 1, which = blockIdx.x & 1;
  const int head = blockIdx.y, b = blockIdx.z;
  const T* src = static_cast<const T*>(A.x[which]) + static_cast<int64_t>(b) * A.seq_stride +
                 static_cast<int64_t>(head) * A.head_stride + static_cast<int64_t>(u) * N * D;
  if (which == 0)
    encode_tile<D, N, 1, 4, 0, T>(A, src, b, head, u, 0, smem);
  else
    encode_tile<D, N, 1, 2, 0, T>(A, src, b, head, u, 1, smem);
}

template <typename T>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(512)
    encode_latent_kernel(EncodeArgs A) {
  extern __shared__ __align__(16) unsigned char smem[];
  const int u = blockIdx.x >> 1, b = blockIdx.y;
  const T* src = static_cast<const T*>(A.x[0]) + static_cast<int64_t>(b) * A.seq_stride +
                 static_cast<int64_t>(u) * 128 * 512;
  encode_tile<512, 128, 2, 4, 1, T>(A, src, b, 0, u, 0, smem);
}

// ------------------------------------------------------------- launchers
template <int D, int N, typename T>
static cudaError_t launch_dense(const EncodeArgs& A, int num_seqs, cudaStream_t st) {
  constexpr int smem = EncShape<D, N, 1>::SMEM;
  auto kern = encode_dense_kernel<D, N, T>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  dim3 grid(2 * A.chunk_tiles, A.num_kv_heads, num_seqs);
  kern<<<grid, 2 * D, smem, st>>>(A);
  return cudaGetLastError();
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
  A.page_bytes = DensePage(p.D, p.N).bytes();
  A.norm_iters = p.norm_iters;
  A.err = p.err;
  if (A.chunk_tiles == 0 || p.num_seqs == 0) return cudaSuccess;
#define KV_DISPATCH(DD, NN)                                                              \
  if (p.D == DD && p.N == NN)                                                            \
    return p.bf16 ? launch_dense<DD, NN, __nv_bfloat16>(A, p.num_seqs, st)               \
                  : launch_dense<DD, NN, __half>(A, p.num_seqs, st);
  KV_DISPATCH(128, 128)
  KV_DISPATCH(128, 64)
  KV_DISPATCH(256, 128)
  KV_DISPATCH(256, 64)
#undef KV_DISPATCH
  return cudaErrorInvalidValue;
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
  if (A.chunk_tiles == 0 || p.num_seqs == 0) return cudaSuccess;
  constexpr int smem = EncShape<512, 128, 2>::SMEM;
  auto kern = p.bf16 ? encode_latent_kernel<__nv_bfloat16> : encode_latent_kernel<__half>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  dim3 grid(2 * A.chunk_tiles, p.num_seqs);
  kern<<<grid, 512, smem, st>>>(A);
  return cudaGetLastError();
}

}  // namespace kvarn

// Uncompressed-cache decode on the KVarN decode skeleton (turbo-attn page,
// "Also a full bf16 backend": raw KV through the same kernel so that the
// codec is the only variable): the page store, and the dense decode kernel
// instantiated with no codec. Same persistent stream-K grid, same page slots
// and copies, same mma.sync hi/lo A tile and online softmax, same merge; the
// pages hold fp16 K and V in fragment order instead of codes and scales, and
// nothing is rotated.
#include <atomic>

#include "kvarn_decode_kernel.cuh"

namespace kvarn {

// ------------------------------------------------------------- page store
template <int D, typename T>
__global__ void __launch_bounds__(128) store_fp16_kernel(StoreFp16Params p) {
  const int pg_i = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int token0 = p.token0 + pg_i * kPageTokens;
  const int lp = token0 / kPageTokens;
  const int phys = p.block_table[static_cast<int64_t>(b) * p.bt_stride + lp];
  if (phys < 0 || phys >= p.num_pages) {
    if (threadIdx.x == 0) set_error(p.err, KVARN_DEVERR_PAGE_RANGE);
    return;
  }
  uint8_t* page = static_cast<uint8_t*>(p.cache) +
                  (static_cast<int64_t>(phys) * p.num_kv_heads + h) * (4 * kPageTokens * D);
  const int64_t base = static_cast<int64_t>(b) * p.seq_stride + static_cast<int64_t>(h) * p.head_stride +
                       static_cast<int64_t>(token0) * D;
  const T* K = static_cast<const T*>(p.k) + base;
  const T* V = static_cast<const T*>(p.v) + base;
  const uint16_t* K16 = reinterpret_cast<const uint16_t*>(K);
  const uint16_t* V16 = reinterpret_cast<const uint16_t*>(V);
  constexpr int U4 = 2 * kPageTokens * D / 16;  // uint4 per region
  for (int c = threadIdx.x; c < 2 * U4; c += blockDim.x) {
    const bool isv = c >= U4;
    const int ci = isv ? c - U4 : c;
    uint16_t e[8];
    if (!isv) {
      const int tau = ci / (D / 8), rem = ci % (D / 8);
      const int t = rem / (D / 32), j = rem % (D / 32);
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int wi = 4 * j + k, kc = wi >> 1, part = wi & 1;
        const int ch = 16 * kc + 2 * t + 8 * part;
        e[2 * k] = K16[tau * D + ch];
        e[2 * k + 1] = K16[tau * D + ch + 1];
      }
    } else {
      const int L = ci / (D / 16), j = ci % (D / 16);
      const int g = L >> 2, t = L & 3;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int wi = 4 * j + k, nc = wi >> 1, part = wi & 1;
        const int ch = 8 * nc + g, tau = 2 * t + 8 * part;
        e[2 * k] = V16[tau * D + ch];
        e[2 * k + 1] = V16[(tau + 1) * D + ch];
      }
    }
    uint4 v;
    v.x = e[0] | (static_cast<uint32_t>(e[1]) << 16);
    v.y = e[2] | (static_cast<uint32_t>(e[3]) << 16);
    v.z = e[4] | (static_cast<uint32_t>(e[5]) << 16);
    v.w = e[6] | (static_cast<uint32_t>(e[7]) << 16);
    reinterpret_cast<uint4*>(page)[c] = v;
  }
}

cudaError_t launch_store_fp16(const StoreFp16Params& p, cudaStream_t st) {
  if (p.count == 0 || p.num_seqs == 0) return cudaSuccess;
  dim3 grid(p.count / kPageTokens, p.num_kv_heads, p.num_seqs);
  if (p.D == 128)
    store_fp16_kernel<128, __half><<<grid, 128, 0, st>>>(p);
  else if (p.D == 256)
    store_fp16_kernel<256, __half><<<grid, 128, 0, st>>>(p);
  else
    return cudaErrorInvalidValue;
  return cudaGetLastError();
}

// The decode over these pages: the dense decode kernel with no codec (fp16
// K and V in fragment order, nothing rotated, 32-token tiles so that a warp's
// two page slots take 16 KB as the compressed tiles' do).
template <int D>
cudaError_t run_raw(const DecArgs& A, int ctas, cudaStream_t st) {
  constexpr int W = D == 256 ? 2 : 4;
  return run_dense<D, 32, W, 4, 2, 4, kCodecRaw>(A, ctas, st);
}
template <int D>
int resident_raw() {
  return resident_dense<D, 32, D == 256 ? 2 : 4, 4, 2, 4, kCodecRaw>();
}
template cudaError_t run_raw<128>(const DecArgs&, int, cudaStream_t);
template cudaError_t run_raw<256>(const DecArgs&, int, cudaStream_t);

int raw_decode_ctas_per_sm(int32_t D) {
  static std::atomic<int> cache[2] = {};
  const int i = D == 256;
  const int known = cache[i].load(std::memory_order_relaxed);
  if (known) return known;
  const int c = D == 256 ? resident_raw<256>() : resident_raw<128>();
  cache[i].store(c, std::memory_order_relaxed);
  return c;
}

}  // namespace kvarn

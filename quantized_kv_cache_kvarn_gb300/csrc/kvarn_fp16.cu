// Uncompressed-cache decode on the KVarN decode skeleton (turbo-attn page,
// "Also a full bf16 backend": raw KV through the same kernel so that the
// codec is the only variable). Same split-K grid, same per-warp bulk-copy
// ring, same mma.sync hi/lo A tile and online softmax, same merge; the pages
// hold fp16/bf16 K and V in fragment order instead of codes and scales, and
// nothing is rotated.
#include <math.h>

#include <algorithm>

#include "kvarn_common.cuh"
#include "kvarn_launch.h"
#include "kvarn_merge.cuh"

namespace kvarn {

constexpr float kLog2eF = 1.4426950408889634f;

template <int D>
struct F16Shape {
  static constexpr int PB = 4 * kPageTokens * D;  // K then V, 2 bytes each
  static constexpr int PPT = 2;                    // pages per tile (32 tokens)
  static constexpr int TILE = PPT * PB;
  static constexpr int KC = D / 16;
  static constexpr int NC = D / 8;
  static constexpr int W = 2;
  static constexpr int STAGES = W * 2 * TILE;
  static constexpr int SMEM = STAGES + W * 2 * 8;
  static_assert(W * 8 * (D + 2) * 4 <= STAGES, "merge scratch");
};

struct F16Args {
  const void* q;
  float kappa;
  const uint8_t* cache;
  int32_t Hq, Hkv, G;
  int64_t num_pages;
  const int32_t* bt;
  int32_t bt_stride;
  const int32_t* seq_lens;
  int32_t max_seq_len;
  float* ws;
  int32_t tps, nsplit, slots;
  uint32_t* err;
};

template <int D, typename T>
__global__ void __launch_bounds__(64) decode_fp16_kernel(F16Args A) {
  using S = F16Shape<D>;
  constexpr int W = S::W;
  extern __shared__ __align__(128) unsigned char smem[];
  pdl_launch_dependents();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g = lane >> 2, t = lane & 3;
  const int split = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
  const int G = A.G;
  constexpr int TT = S::PPT * kPageTokens;  // tokens per tile

  int len = A.seq_lens[b];
  if (len < 0 || len > A.max_seq_len) {
    if (threadIdx.x == 0) set_error(A.err, KVARN_DEVERR_SEQ_LEN);
    len = len < 0 ? 0 : A.max_seq_len;
  }
  const int ntiles = (len + TT - 1) / TT;
  const int npages = (len + kPageTokens - 1) / kPageTokens;
  const int t0 = split * A.tps, t1 = min(t0 + A.tps, ntiles);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S::STAGES);
  if (t0 >= t1) {
    for (int h = warp; h < G; h += W) {
      float* part = A.ws + (static_cast<int64_t>(b * A.Hq + kvh * G + h) * A.slots + split) * (D + 4);
      if (lane == 0) { part[0] = -INFINITY; part[1] = 0.f; }
      for (int j = lane; j < D; j += 32) part[4 + j] = 0.f;
    }
    return;
  }
  if (lane == 0) {
    mbar_init(&bars[2 * warp], 1);
    mbar_init(&bars[2 * warp + 1], 1);
  }
  fence_mbar_init();
  __syncthreads();

  // A fragments of the raw query (fp16 exact for fp16 q; rows >= G zero).
  uint32_t Aq[S::KC][4];
  {
    const T* qp = static_cast<const T*>(A.q) + static_cast<int64_t>(b * A.Hq + kvh * G + g) * D;
#pragma unroll
    for (int kc = 0; kc < S::KC; ++kc) {
      const int ch0 = 16 * kc + 2 * t;
      float x0 = 0.f, x1 = 0.f, x8 = 0.f, x9 = 0.f;
      if (g < G) {
        x0 = to_f32<T>(qp[ch0]); x1 = to_f32<T>(qp[ch0 + 1]);
        x8 = to_f32<T>(qp[ch0 + 8]); x9 = to_f32<T>(qp[ch0 + 9]);
      }
      split_hi_lo(x0, x1, Aq[kc][0], Aq[kc][1]);
      split_hi_lo(x8, x9, Aq[kc][2], Aq[kc][3]);
    }
  }

  const int first = t0 + warp;
  const int n_my = first < t1 ? (t1 - first + W - 1) / W : 0;
  unsigned char* ring = smem + warp * 2 * S::TILE;
  uint64_t* bar = bars + 2 * warp;
  const int32_t* bt = A.bt + static_cast<int64_t>(b) * A.bt_stride;

  auto issue = [&](int i) {
    const int tile = first + i * W, st = i & 1;
    const int np = min(S::PPT, npages - tile * S::PPT);
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) mbar_arrive_expect_tx(&bar[st], np * S::PB);
    __syncwarp();
    if (lane < np) {
      int phys = bt[tile * S::PPT + lane];
      if (phys < 0 || phys >= A.num_pages) {
        set_error(A.err, KVARN_DEVERR_PAGE_RANGE);
        phys = 0;
      }
      bulk_g2s(ring + st * S::TILE + lane * S::PB,
               A.cache + (static_cast<int64_t>(phys) * A.Hkv + kvh) * S::PB, S::PB, &bar[st]);
    }
  };
  if (n_my > 0) issue(0);
  if (n_my > 1) issue(1);

  float m = -INFINITY, lsum = 0.f;
  float acc[S::NC][2];
#pragma unroll
  for (int nc = 0; nc < S::NC; ++nc) acc[nc][0] = acc[nc][1] = 0.f;

  int i = 0;
  for (; i < n_my; ++i) {
    const int st = i & 1;
    const int tile = first + i * W;
    if (!mbar_wait_bounded(&bar[st], (i >> 1) & 1)) {
      if (lane == 0) set_error(A.err, KVARN_DEVERR_TIMEOUT);
      break;
    }
    const unsigned char* buf = ring + st * S::TILE;
    const int valid = len - tile * TT;  // tokens of this tile below len

    float s[4][2];
#pragma unroll
    for (int nb = 0; nb < 4; ++nb) {
      if ((nb >> 1) * kPageTokens >= valid) {  // page not loaded
        s[nb][0] = s[nb][1] = -INFINITY;
        continue;
      }
      const unsigned char* kp = buf + (nb >> 1) * S::PB + ((nb & 1) * 8 + g) * (2 * D) + t * (D / 2);
      float d[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int j = 0; j < S::KC / 2; ++j) {
        const uint4 kw = *reinterpret_cast<const uint4*>(kp + 16 * j);
        mma_f16(d, Aq[2 * j][0], Aq[2 * j][1], Aq[2 * j][2], Aq[2 * j][3], kw.x, kw.y);
        mma_f16(d, Aq[2 * j + 1][0], Aq[2 * j + 1][1], Aq[2 * j + 1][2], Aq[2 * j + 1][3], kw.z, kw.w);
      }
      const int tok = nb * 8 + 2 * t;
      s[nb][0] = tok < valid ? (d[0] + d[2]) * A.kappa : -INFINITY;
      s[nb][1] = tok + 1 < valid ? (d[1] + d[3]) * A.kappa : -INFINITY;
    }
    float mt = -INFINITY;
#pragma unroll
    for (int nb = 0; nb < 4; ++nb) mt = fmaxf(mt, fmaxf(s[nb][0], s[nb][1]));
    mt = warp_max_xor(mt, 1, 4);
    const float m_new = fmaxf(m, mt);
    const float alpha = exp2f(m - m_new);
    float psum = 0.f;
#pragma unroll
    for (int nb = 0; nb < 4; ++nb) {
      s[nb][0] = exp2f(s[nb][0] - m_new);
      s[nb][1] = exp2f(s[nb][1] - m_new);
      psum += s[nb][0] + s[nb][1];
    }
    lsum = fmaf(lsum, alpha, psum);
    m = m_new;

    uint32_t Ap[S::PPT][4];
#pragma unroll
    for (int pp = 0; pp < S::PPT; ++pp) {
      split_hi_lo(s[2 * pp][0], s[2 * pp][1], Ap[pp][0], Ap[pp][1]);
      split_hi_lo(s[2 * pp + 1][0], s[2 * pp + 1][1], Ap[pp][2], Ap[pp][3]);
    }
#pragma unroll
    for (int nc = 0; nc < S::NC; ++nc) {
      acc[nc][0] *= alpha;
      acc[nc][1] *= alpha;
    }
#pragma unroll
    for (int pp = 0; pp < S::PPT; ++pp) {
      if (pp * kPageTokens >= valid) break;
      const unsigned char* vp = buf + pp * S::PB + 2 * kPageTokens * D + (4 * g + t) * D;
      // rows past seq_len in a partial page carry weight 0 but may hold any
      // bits; clear them so that 0 * (inf or nan) never reaches the sum
      const int tb = pp * kPageTokens + 2 * t;
      const uint32_t m01 = (tb < valid ? 0x0000FFFFu : 0u) | (tb + 1 < valid ? 0xFFFF0000u : 0u);
      const uint32_t m89 = (tb + 8 < valid ? 0x0000FFFFu : 0u) | (tb + 9 < valid ? 0xFFFF0000u : 0u);
#pragma unroll
      for (int j = 0; j < S::NC / 2; ++j) {
        uint4 vw = *reinterpret_cast<const uint4*>(vp + 16 * j);
        vw.x &= m01; vw.y &= m89; vw.z &= m01; vw.w &= m89;
        float u0[4] = {0.f, 0.f, 0.f, 0.f}, u1[4] = {0.f, 0.f, 0.f, 0.f};
        mma_f16(u0, Ap[pp][0], Ap[pp][1], Ap[pp][2], Ap[pp][3], vw.x, vw.y);
        mma_f16(u1, Ap[pp][0], Ap[pp][1], Ap[pp][2], Ap[pp][3], vw.z, vw.w);
        acc[2 * j][0] += u0[0] + u0[2];
        acc[2 * j][1] += u0[1] + u0[3];
        acc[2 * j + 1][0] += u1[0] + u1[2];
        acc[2 * j + 1][1] += u1[1] + u1[3];
      }
    }
    if (i + 2 < n_my) issue(i + 2);
  }
  if (i < n_my) {
    for (int j = i; j < min(n_my, i + 2); ++j) mbar_wait_bounded(&bar[j & 1], (j >> 1) & 1, 100000000LL);
  }
  lsum = warp_sum_xor(lsum, 1, 4);

  __syncthreads();
  float* mrg = reinterpret_cast<float*>(smem);
  float* mw = mrg + warp * 8 * (D + 2);
  if (t == 0) {
    mw[g * (D + 2)] = n_my > 0 ? m : -INFINITY;
    mw[g * (D + 2) + 1] = n_my > 0 ? lsum : 0.f;
  }
#pragma unroll
  for (int nc = 0; nc < S::NC; ++nc) {
    mw[g * (D + 2) + 2 + 8 * nc + 2 * t] = acc[nc][0];
    mw[g * (D + 2) + 2 + 8 * nc + 2 * t + 1] = acc[nc][1];
  }
  __syncthreads();
  for (int idx = threadIdx.x; idx < G * D; idx += W * 32) {
    const int gg = idx / D, j = idx % D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < W; ++w) M = fmaxf(M, mrg[(w * 8 + gg) * (D + 2)]);
    float a = 0.f, L = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < W; ++w) {
        const float* r = mrg + (w * 8 + gg) * (D + 2);
        const float sc = exp2f(r[0] - M);
        a = fmaf(r[2 + j], sc, a);
        L = fmaf(r[1], sc, L);
      }
    }
    float* part = A.ws + (static_cast<int64_t>(b * A.Hq + kvh * G + gg) * A.slots + split) * (D + 4);
    part[4 + j] = a;
    if (j == 0) {
      part[0] = M;
      part[1] = L;
    }
  }
}

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

template <int D>
static cudaError_t run_fp16(const F16Args& A, int num_seqs, cudaStream_t st) {
  using S = F16Shape<D>;
  auto kern = decode_fp16_kernel<D, __half>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, S::SMEM);
  if (e != cudaSuccess) return e;
  dim3 grid(A.nsplit, A.Hkv, num_seqs);
  kern<<<grid, S::W * 32, S::SMEM, st>>>(A);
  return cudaGetLastError();
}

cudaError_t launch_decode_fp16(const DecodeParams& p, const SplitPlan& plan, cudaStream_t st) {
  if (p.num_seqs == 0) return cudaSuccess;
  F16Args A{};
  A.q = p.q;
  A.kappa = p.sm_scale * kLog2eF;
  A.cache = p.cache;
  A.Hq = p.num_q_heads;
  A.Hkv = p.num_kv_heads;
  A.G = p.num_q_heads / p.num_kv_heads;
  A.num_pages = p.num_pages;
  A.bt = p.block_table;
  A.bt_stride = p.bt_stride;
  A.seq_lens = p.seq_lens;
  A.max_seq_len = p.max_seq_len;
  A.ws = static_cast<float*>(p.workspace);
  A.tps = plan.tiles_per_split;
  A.nsplit = plan.nsplit;
  A.slots = plan.slots;
  A.err = p.err;
  cudaError_t e = cudaErrorInvalidValue;
  if (p.D == 128) e = run_fp16<128>(A, p.num_seqs, st);
  else if (p.D == 256) e = run_fp16<256>(A, p.num_seqs, st);
  if (e != cudaSuccess) return e;
  const int rows = p.num_seqs * p.num_q_heads;
  return p.D == 128 ? launch_merge<128>(A.ws, A.slots, rows, nullptr, 0, 0, p.out, p.lse, st)
                    : launch_merge<256>(A.ws, A.slots, rows, nullptr, 0, 0, p.out, p.lse, st);
}

}  // namespace kvarn

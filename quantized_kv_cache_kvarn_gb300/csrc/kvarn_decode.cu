// KVarN decode attention over the compressed paged cache, sm_103a.
//
// Paged, split-K, GQA-grouped decode that streams the packed codes and
// scales straight from HBM and dequantises them on chip; no fp16 K or V
// buffer is ever formed in memory (turbo-attn page, "Inline dequant").
// Scores are taken in the rotated basis: the query is rotated once per CTA
// and the output un-rotated once in the merge (turbo-attn page, "How it
// works").
//
// Kernel 1 (decode_dense_kernel): one CTA per (KV head, split, sequence),
// one thread per channel (D threads). The split's tiles stream through a
// two-stage shared-memory ring filled by one-dimensional bulk copies (one
// per page, completion counted on an mbarrier) with the pages further
// ahead prefetched into L2. Per tile, on the fifth-generation tensor cores:
//   Q K:  thread i turns token i's packed K codes into exact fp16 integers
//         (code - 8) and stores them in tensor memory: A = K~ [128 tokens x
//         D]. q~ = (kappa q H) * c_K, split into fp16 hi + lo rows, is the
//         shared-memory B operand [16 x D] (rows 0-7 hi, 8-15 lo of the
//         G <= 8 heads of the group); S^T = K~ q~^T lands in tensor memory;
//   s  = a_K * (S_hi + S_lo) + (b_K + 8 a_K) * sum(q~)  (row scales folded);
//   online softmax in base 2, rescaling only when a running maximum rises;
//   P V:  thread j turns channel j's V codes into fp16 (code - 2) in tensor
//         memory: A = V~^T [D x tokens]; the weights p * a_V (hi + lo) are
//         the B operand, so U^T = V~^T (p a_V)^T; a second product against
//         an all-ones A block gives beta = sum_i p_i (b_V + 2 a_V) for every
//         lane without a cross-thread reduction;
//   acc_j = acc_j * alpha + c_V[j] * (U_j + beta)    (thread j, all heads).
// The CTA writes one partial (max, sum, unnormalised output) per split and
// head; the last split slot holds the fp16 tail (tokens past the last full
// tile, in the original basis).
// Kernel 2 (merge_kernel): log-sum-exp merge of the partials, inverse
// Hadamard transform of the rotated part, plus the tail part.
#include <math.h>

#include "kvarn_common.cuh"
#include "kvarn_launch.h"
#include "kvarn_merge.cuh"
#include "kvarn_tc.cuh"
#include <algorithm>

namespace kvarn {

constexpr float kLog2e = 1.4426950408889634f;

constexpr int align_up(int x, int a) { return (x + a - 1) / a * a; }

template <int D, int N>
struct DecShape {
  static constexpr DensePage PG{D, N};
  static constexpr int NT = D;                 // one thread per channel
  static constexpr int NWARP = NT / 32;
  static constexpr int PPT = N / kPageTokens;  // pages per tile
  static constexpr int PB = PG.bytes();
  static constexpr int TILE = PPT * PB;        // staged bytes per tile
  static constexpr int STAGES = 2;
  static constexpr int CPP = PG.cols();        // column scales per page
  static constexpr int DB = D / 128;           // 128-channel blocks of V~^T
  static constexpr int HPT = 8 / DB;           // heads per thread in the softmax
  // tensor-memory columns
  static constexpr int TM_A = 0;               // A operand (K~ or V~^T): D/2 columns
  static constexpr int TM_S = D / 2;           // S^T, 16 columns
  static constexpr int TM_U = TM_S + 16;       // U^T, 16 per channel block
  static constexpr int TM_B = TM_U + 16 * DB;  // beta, 16
  static constexpr int TM_ONE = TM_B + 16;     // all-ones A block, 8 (K = 16)
  static constexpr int TM_COLS = TM_ONE + 8 <= 128 ? 128 : 256;
  // shared memory
  static constexpr int OFF_BP = align_up(STAGES * TILE, 1024);  // B of P V: [16 x N] f16, MN-major
  static constexpr int OFF_BQ = OFF_BP + align_up(32 * N, 1024);  // B of Q K [16 x D], K-major; then beta weights
  static constexpr int BQ_BYTES = align_up(32 * (D > N ? D : N), 1024);
  static constexpr int OFF_QSUM = OFF_BQ + BQ_BYTES;  // [8] f32
  static constexpr int OFF_TMAX = OFF_QSUM + 32;      // [NWARP][8] f32
  static constexpr int OFF_FLAG = OFF_TMAX + NWARP * 32;  // [NWARP] u32
  static constexpr int OFF_BAR = align_up(OFF_FLAG + NWARP * 4, 16);  // STAGES + 2 mbarriers
  static constexpr int OFF_TMEM = OFF_BAR + 8 * (STAGES + 2);
  static constexpr int OFF_PAGES = align_up(OFF_TMEM + 4, 16);  // the split's page ids
  // at least this much shared memory, so that no more CTAs share an SM than
  // its 512 tensor-memory columns hold
  static constexpr int SMEM_FLOOR = 228 * 1024 / (512 / TM_COLS + 1) + 1024;
  static constexpr uint32_t IDESC_K = idesc_f16(128, 16, false);
  static constexpr uint32_t IDESC_MN = idesc_f16(128, 16, true);
  static_assert(TM_ONE + 8 <= TM_COLS, "tensor-memory plan");
  static_assert(TILE % 16 == 0 && PB % 16 == 0, "bulk copies keep 16-byte alignment");
};

struct DecArgs {
  const void* q;
  float kappa;  // sm_scale * log2(e)
  const uint8_t* cache;
  int32_t Hq, Hkv, G;
  int64_t num_pages;
  const int32_t* bt;
  int32_t bt_stride;
  const int32_t* seq_lens;
  int32_t max_seq_len;
  const void* tail_k;
  const void* tail_v;
  float* ws;
  int32_t tps, nsplit, slots;
  uint32_t* err;
};

template <typename T, int E>
__device__ __forceinline__ void load_vec(const T* p, float* out) {
  if constexpr (E == 4) {
    uint2 u = __ldg(reinterpret_cast<const uint2*>(p));
    const T* h = reinterpret_cast<const T*>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) out[i] = to_f32<T>(h[i]);
  } else {
    static_assert(E % 8 == 0, "vector width");
#pragma unroll
    for (int k = 0; k < E; k += 8) load8<T>(p + k, out + k);
  }
}

__device__ __forceinline__ void write_empty(float* part, int D, int lane) {
  if (lane == 0) {
    part[0] = -INFINITY;
    part[1] = 0.f;
  }
  for (int j = lane; j < D; j += 32) part[4 + j] = 0.f;
}

// fp16 tail over tokens [committed, len): dense attention in the original
// basis, one warp per query head.
template <int D, int N, typename T, int W>
__device__ void tail_partials(const DecArgs& A, int b, int kvh, int tail, unsigned char* smem) {
  constexpr int E = D / 32;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  float* sbuf = reinterpret_cast<float*>(smem) + warp * N;
  for (int h = warp; h < A.G; h += W) {
    const int hq = kvh * A.G + h;
    float* part = A.ws + (static_cast<int64_t>(b * A.Hq + hq) * A.slots + A.nsplit) * kPStride(D);
    if (tail == 0 || A.tail_k == nullptr || A.tail_v == nullptr) {
      if (tail > 0 && lane == 0) set_error(A.err, KVARN_DEVERR_NO_TAIL);
      write_empty(part, D, lane);
      continue;
    }
    float qv[E];
    load_vec<T, E>(static_cast<const T*>(A.q) + static_cast<int64_t>(b * A.Hq + hq) * D + lane * E, qv);
#pragma unroll
    for (int e = 0; e < E; ++e) qv[e] *= A.kappa;
    const int64_t row0 = (static_cast<int64_t>(b) * A.Hkv + kvh) * N;
    const T* tk = static_cast<const T*>(A.tail_k);
    const T* tv = static_cast<const T*>(A.tail_v);
    float mx = -INFINITY;
    for (int tau = 0; tau < tail; ++tau) {
      float kv[E];
      load_vec<T, E>(tk + (row0 + tau) * D + lane * E, kv);
      float dot = 0.f;
#pragma unroll
      for (int e = 0; e < E; ++e) dot = fmaf(qv[e], kv[e], dot);
      dot = warp_sum_xor(dot, 1, 32);
      if (lane == 0) sbuf[tau] = dot;
      mx = fmaxf(mx, dot);
    }
    __syncwarp();
    float l = 0.f, acc[E];
#pragma unroll
    for (int e = 0; e < E; ++e) acc[e] = 0.f;
    for (int tau = 0; tau < tail; ++tau) {
      const float p = exp2f(sbuf[tau] - mx);
      l += p;
      float vv[E];
      load_vec<T, E>(tv + (row0 + tau) * D + lane * E, vv);
#pragma unroll
      for (int e = 0; e < E; ++e) acc[e] = fmaf(p, vv[e], acc[e]);
    }
    __syncwarp();
    if (lane == 0) {
      part[0] = mx;
      part[1] = l;
    }
#pragma unroll
    for (int e = 0; e < E; ++e) part[4 + lane * E + e] = acc[e];
  }
}

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Warp maximum of a float through the integer reduction unit: the map
// below is monotone on IEEE floats and its own inverse.
__device__ __forceinline__ float warp_max_redux(float v) {
  int k = __float_as_int(v);
  k = k >= 0 ? k : (k ^ 0x7FFFFFFF);
  k = __reduce_max_sync(0xffffffffu, k);
  return __int_as_float(k >= 0 ? k : (k ^ 0x7FFFFFFF));
}

template <int D, int N, typename T>
__global__ void __launch_bounds__(D, (D == 128 ? 4 : 2)) decode_dense_kernel(DecArgs A) {
  using S = DecShape<D, N>;
  constexpr DensePage PG{D, N};
  extern __shared__ __align__(1024) unsigned char smem[];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // token role: token tid % 128; kh = channel half (K~) and head group
  // (softmax) for D = 256, always 0 for D = 128
  const int tok = tid & 127, kh = DecShape<D, N>::DB == 1 ? 0 : (tid >> 7);
  const int kvh = blockIdx.x, split = blockIdx.y, b = blockIdx.z;
  const int G = A.G;

  int len = A.seq_lens[b];
  if (len < 0 || len > A.max_seq_len) {
    if (tid == 0) set_error(A.err, KVARN_DEVERR_SEQ_LEN);
    len = len < 0 ? 0 : A.max_seq_len;
  }
  const int ntiles = len / N;
  if (split == A.nsplit) {
    tail_partials<D, N, T, S::NWARP>(A, b, kvh, len - ntiles * N, smem);
    return;
  }
  const int t0 = split * A.tps, t1 = min(t0 + A.tps, ntiles);
  if (t0 >= t1) {
    for (int h = warp; h < G; h += S::NWARP)
      write_empty(A.ws + (static_cast<int64_t>(b * A.Hq + kvh * G + h) * A.slots + split) * kPStride(D),
                  D, lane);
    return;
  }
  const int nt = t1 - t0;

  unsigned char* bp = smem + S::OFF_BP;
  unsigned char* bq = smem + S::OFF_BQ;
  float* qsum = reinterpret_cast<float*>(smem + S::OFF_QSUM);
  float* tmax = reinterpret_cast<float*>(smem + S::OFF_TMAX);
  uint32_t* flag = reinterpret_cast<uint32_t*>(smem + S::OFF_FLAG);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S::OFF_BAR);
  uint64_t* barQ = bars + S::STAGES;
  uint64_t* barP = barQ + 1;
  uint32_t* tslot = reinterpret_cast<uint32_t*>(smem + S::OFF_TMEM);
  int32_t* pages = reinterpret_cast<int32_t*>(smem + S::OFF_PAGES);
  const int32_t* bt = A.bt + static_cast<int64_t>(b) * A.bt_stride;

  // the split's block-table entries, checked once, into shared memory
  for (int e = tid; e < nt * S::PPT; e += S::NT) {
    int phys = bt[t0 * S::PPT + e];
    if (phys < 0 || phys >= A.num_pages) {
      set_error(A.err, KVARN_DEVERR_PAGE_RANGE);
      phys = 0;
    }
    pages[e] = phys;
  }
  if (tid == 0) {
    for (int s = 0; s < S::STAGES + 2; ++s) mbar_init(bars + s, 1);
    fence_mbar_init();
  }
  if (warp == 0) tmem_alloc<S::TM_COLS>(tslot);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tslot;
  const uint32_t tq = tbase + (static_cast<uint32_t>(32 * (warp & 3)) << 16);  // this warp's lane quarter

  auto page_src = [&](int i, int p) -> const unsigned char* {
    return A.cache + (static_cast<int64_t>(pages[i * S::PPT + p]) * A.Hkv + kvh) * S::PB;
  };
  auto issue = [&](int i) {  // thread 0: tile i of the split into stage i % STAGES
    uint64_t* bar = bars + i % S::STAGES;
    unsigned char* dst = smem + (i % S::STAGES) * S::TILE;
    fence_proxy_async_smem();
    mbar_arrive_expect_tx(bar, S::TILE);
    for (int p = 0; p < S::PPT; ++p) bulk_g2s(dst + p * S::PB, page_src(i, p), S::PB, bar);
  };
  auto prefetch = [&](int i) {
    for (int p = 0; p < S::PPT; ++p) prefetch_l2(page_src(i, p), S::PB);
  };
  int issued = min(S::STAGES, nt);  // tiles whose copies have been started (uniform)
  if (tid == 0) {
    for (int i = 0; i < issued; ++i) issue(i);
    if (S::STAGES < nt) prefetch(S::STAGES);
  }

  // ---- rotated, scaled query rows (fp32, staged in the B_q area), then
  //      each thread keeps the 8 channels of its q~ role in registers
  {
    float* qrot = reinterpret_cast<float*>(bq);
    constexpr int E = D / 32;
    for (int h = warp; h < 8; h += S::NWARP) {
      float v[E];
      if (h < G) {
        load_vec<T, E>(static_cast<const T*>(A.q) + static_cast<int64_t>(b * A.Hq + kvh * G + h) * D + lane * E, v);
        warp_fwht<E>(v);
        const float sc = A.kappa / sqrtf(static_cast<float>(D));
#pragma unroll
        for (int e = 0; e < E; ++e) v[e] *= sc;
      } else {
#pragma unroll
        for (int e = 0; e < E; ++e) v[e] = 0.f;
      }
#pragma unroll
      for (int e = 0; e < E; ++e) qrot[h * D + lane * E + e] = v[e];
    }
  }
  // the all-ones A block (fp16 1.0 pairs), once
  if (warp < 4) {
    uint32_t ones[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) ones[j] = 0x3C003C00u;
    tmem_st8(tq + S::TM_ONE, ones);
    tmem_wait_st();
  }
  __syncthreads();
  const int qh = tid / (D / 8), qc = tid % (D / 8);  // q~ role: head row, 8-channel chunk
  float qf[8];
  {
    const float4* src = reinterpret_cast<const float4*>(reinterpret_cast<float*>(bq) + qh * D + 8 * qc);
    const float4 u0 = src[0], u1 = src[1];
    qf[0] = u0.x; qf[1] = u0.y; qf[2] = u0.z; qf[3] = u0.w;
    qf[4] = u1.x; qf[5] = u1.y; qf[6] = u1.z; qf[7] = u1.w;
  }
  __syncthreads();  // B_q area free

  float m[8], alpha[8], lpart[S::HPT], acc[8];
#pragma unroll
  for (int h = 0; h < 8; ++h) m[h] = -INFINITY, acc[h] = 0.f, alpha[h] = 1.f;
#pragma unroll
  for (int j = 0; j < S::HPT; ++j) lpart[j] = 0.f;

  int i = 0;
  int to = 0;
  for (; i < nt; ++i) {
    const int st = i % S::STAGES;
    if (!mbar_wait_bounded(bars + st, (i / S::STAGES) & 1)) to = 1;
    to = __any_sync(0xffffffffu, to);  // warp-uniform: warp-collective TMEM moves follow
    const unsigned char* tile = smem + st * S::TILE;

    // -- (a) K~ rows into tensor memory; q~ into the B operand
    if (tok < N && !to) {
      const unsigned char* kp = tile + (tok / kPageTokens) * S::PB + (tok % kPageTokens) * (D / 2) + 16 * kh;
      uint4 kw[4];
#pragma unroll
      for (int t = 0; t < 4; ++t) kw[t] = *reinterpret_cast<const uint4*>(kp + t * (D / 8));
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        uint32_t r[32];
#pragma unroll
        for (int t = 0; t < 4; ++t)
#pragma unroll
          for (int ww = 0; ww < 2; ++ww) {
            const int w4 = 2 * half + ww;
            const uint32_t word = w4 == 0 ? kw[t].x : w4 == 1 ? kw[t].y : w4 == 2 ? kw[t].z : kw[t].w;
            uint32_t bf[4];
            dequant_k_word(word, bf);
            // channel pairs 16 ww + t (+4, +8, +12) of this 64-channel half
            r[16 * ww + t] = bf[0];
            r[16 * ww + t + 4] = bf[1];
            r[16 * ww + t + 8] = bf[2];
            r[16 * ww + t + 12] = bf[3];
          }
        tmem_st32(tq + S::TM_A + 64 * kh + 32 * half, r);
      }
    }
    if (!to) {
      const float* cp = reinterpret_cast<const float*>(tile + ((8 * qc) / S::CPP) * S::PB + PG.k_col() +
                                                       ((8 * qc) % S::CPP) * 4);
      const float4 c0 = reinterpret_cast<const float4*>(cp)[0], c1 = reinterpret_cast<const float4*>(cp)[1];
      const float x[8] = {qf[0] * c0.x, qf[1] * c0.y, qf[2] * c0.z, qf[3] * c0.w,
                          qf[4] * c1.x, qf[5] * c1.y, qf[6] * c1.z, qf[7] * c1.w};
      uint32_t hi[4], lo[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) split_hi_lo(x[2 * e], x[2 * e + 1], hi[e], lo[e]);
      // K-major [16 x D]: row n at (n % 8) 16 + (n / 8) 16D, k-chunk at 128 (k / 8)
      *reinterpret_cast<uint4*>(bq + qh * 16 + qc * 128) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
      *reinterpret_cast<uint4*>(bq + 16 * D + qh * 16 + qc * 128) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
      float qs = ((x[0] + x[1]) + (x[2] + x[3])) + ((x[4] + x[5]) + (x[6] + x[7]));
      qs = warp_sum_xor(qs, 1, D / 8);
      if (qc == 0) qsum[qh] = qs;
    }
    tmem_wait_st();
    fence_proxy_async_smem();
    tc_fence_before();
    if (__syncthreads_or(to)) {
      to = 1;
      break;
    }

    // -- (b) S^T = K~ q~^T
    if (tid == 0) {
      tc_fence_after();
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk)
        umma_ts(tbase + S::TM_S, tbase + S::TM_A + 8 * kk,
                smem_desc(tc_smem(bq) + 256 * kk, 128, 16 * D), S::IDESC_K, kk > 0);
      umma_commit(barQ);
    }
    if (!mbar_wait_bounded(barQ, i & 1)) to = 1;
    to = __any_sync(0xffffffffu, to);
    tc_fence_after();

    // -- (c) scores, running maximum, weights
    float sc[S::HPT];
    float over = -INFINITY;
    const bool has_tok = tok < N;
    const unsigned char* kpg = tile + (tok / kPageTokens) * S::PB;
    if (has_tok) {  // warp-uniform
      uint32_t sr[16];
      tmem_ld16(tq + S::TM_S, sr);
      const float ka = reinterpret_cast<const float*>(kpg + PG.k_a())[tok % kPageTokens];
      const float kb = reinterpret_cast<const float*>(kpg + PG.k_b())[tok % kPageTokens];
      const float kb8 = fmaf(8.f, ka, kb);
      tmem_wait_ld();
#pragma unroll
      for (int j = 0; j < S::HPT; ++j) {
        const int h = kh * S::HPT + j;
        const float shi = kh ? __uint_as_float(sr[S::HPT + j]) : __uint_as_float(sr[j]);
        const float slo = kh ? __uint_as_float(sr[S::HPT + j + 8]) : __uint_as_float(sr[j + 8]);
        const float mh = kh ? m[S::HPT + j] : m[j];
        sc[j] = fmaf(ka, shi + slo, kb8 * qsum[h]);
        over = fmaxf(over, sc[j] - mh);
      }
    }
    const uint32_t any = __any_sync(0xffffffffu, over > 0.f);
    if (lane == 0) flag[warp] = any;
    __syncthreads();
    uint32_t rescale = 0;
#pragma unroll
    for (int w = 0; w < S::NWARP; ++w) rescale |= flag[w];
    if (rescale) {  // CTA-uniform: a running maximum rises
#pragma unroll
      for (int j = 0; j < S::HPT; ++j) {
        const float v = warp_max_redux(has_tok ? sc[j] : -INFINITY);
        if (lane == 0) tmax[warp * 8 + j] = v;
      }
      __syncthreads();
#pragma unroll
      for (int h = 0; h < 8; ++h) {
        const int grp = h / S::HPT, j = h % S::HPT;  // warps 4 grp .. 4 grp + 3 hold head h
        float mt = m[h];
#pragma unroll
        for (int w = 0; w < 4; ++w) mt = fmaxf(mt, tmax[(4 * grp + w) * 8 + j]);
        alpha[h] = fast_exp2(m[h] - mt);
        m[h] = mt;
      }
#pragma unroll
      for (int j = 0; j < S::HPT; ++j) lpart[j] *= kh ? alpha[S::HPT + j] : alpha[j];
    }
    if (has_tok) {
      const unsigned char* vpg = kpg + PG.k_part();
      const float va = reinterpret_cast<const float*>(vpg + PG.v_a() - PG.k_part())[tok % kPageTokens];
      const float vb = reinterpret_cast<const float*>(vpg + PG.v_b() - PG.k_part())[tok % kPageTokens];
      const float vb2 = fmaf(2.f, va, vb);
      float pa[S::HPT], pb[S::HPT];
#pragma unroll
      for (int j = 0; j < S::HPT; ++j) {
        const float p = fast_exp2(sc[j] - (kh ? m[S::HPT + j] : m[j]));
        lpart[j] += p;
        pa[j] = p * va;
        pb[j] = p * vb2;
      }
      // MN-major [16 x N]: token k at (k % 8) 16 + (k / 8) 128, head row n at
      // (n % 8) 2 + (n / 8) 16N
      const int o = (tok % 8) * 16 + (tok / 8) * 128 + kh * (2 * S::HPT);
      if constexpr (S::HPT == 8) {
        uint32_t h0[4], l0[4], h1[4], l1[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          split_hi_lo(pa[2 * e], pa[2 * e + 1], h0[e], l0[e]);
          split_hi_lo(pb[2 * e], pb[2 * e + 1], h1[e], l1[e]);
        }
        *reinterpret_cast<uint4*>(bp + o) = make_uint4(h0[0], h0[1], h0[2], h0[3]);
        *reinterpret_cast<uint4*>(bp + 16 * N + o) = make_uint4(l0[0], l0[1], l0[2], l0[3]);
        *reinterpret_cast<uint4*>(bq + o) = make_uint4(h1[0], h1[1], h1[2], h1[3]);
        *reinterpret_cast<uint4*>(bq + 16 * N + o) = make_uint4(l1[0], l1[1], l1[2], l1[3]);
      } else {
        uint32_t h0[2], l0[2], h1[2], l1[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          split_hi_lo(pa[2 * e], pa[2 * e + 1], h0[e], l0[e]);
          split_hi_lo(pb[2 * e], pb[2 * e + 1], h1[e], l1[e]);
        }
        *reinterpret_cast<uint2*>(bp + o) = make_uint2(h0[0], h0[1]);
        *reinterpret_cast<uint2*>(bp + 16 * N + o) = make_uint2(l0[0], l0[1]);
        *reinterpret_cast<uint2*>(bq + o) = make_uint2(h1[0], h1[1]);
        *reinterpret_cast<uint2*>(bq + 16 * N + o) = make_uint2(l1[0], l1[1]);
      }
    }

    // -- (d) V~^T rows (channel tid) into tensor memory
    float cv;
    {
      const int d = tid;
      cv = reinterpret_cast<const float*>(tile + (d / S::CPP) * S::PB + PG.v_col())[d % S::CPP];
      constexpr int GROUPS = (S::PPT + 3) / 4;  // 4 pages = 32 columns per store
#pragma unroll
      for (int gi = 0; gi < GROUPS; ++gi) {
        uint32_t r[32];
#pragma unroll
        for (int pp = 0; pp < 4; ++pp) {
          const uint32_t word =
              reinterpret_cast<const uint32_t*>(tile + (4 * gi + pp) * S::PB + PG.v_codes())[d];
          uint32_t vf[8];
          dequant_v_word(word, vf);
#pragma unroll
          for (int q = 0; q < 8; ++q) r[8 * pp + q] = vf[q];
        }
        tmem_st32(tq + S::TM_A + (d >> 7) * (N / 2) + 32 * gi, r);
      }
    }
    tmem_wait_st();
    fence_proxy_async_smem();
    tc_fence_before();
    if (__syncthreads_or(to)) {
      to = 1;
      break;
    }
    // the stage is consumed: refill it with tile i + STAGES
    if (i + S::STAGES < nt) {
      if (tid == 0) {
        issue(i + S::STAGES);
        if (i + S::STAGES + 1 < nt) prefetch(i + S::STAGES + 1);
      }
      issued = i + S::STAGES + 1;
    }

    // -- (e) U^T = V~^T (p a_V)^T per channel block, beta = 1 (p (b_V + 2 a_V))^T
    if (tid == 0) {
      tc_fence_after();
#pragma unroll
      for (int db = 0; db < S::DB; ++db)
#pragma unroll
        for (int kk = 0; kk < N / 16; ++kk)
          umma_ts(tbase + S::TM_U + 16 * db, tbase + S::TM_A + db * (N / 2) + 8 * kk,
                  smem_desc(tc_smem(bp) + 256 * kk, 128, 16 * N), S::IDESC_MN, kk > 0);
#pragma unroll
      for (int kk = 0; kk < N / 16; ++kk)
        umma_ts(tbase + S::TM_B, tbase + S::TM_ONE, smem_desc(tc_smem(bq) + 256 * kk, 128, 16 * N),
                S::IDESC_MN, kk > 0);
      umma_commit(barP);
    }
    if (!mbar_wait_bounded(barP, i & 1)) to = 1;
    to = __any_sync(0xffffffffu, to);
    tc_fence_after();

    // -- (f) accumulate (thread = channel, all heads)
    {
      uint32_t u[16], be[16];
      tmem_ld16(tq + S::TM_U + 16 * kh, u);
      tmem_ld16(tq + S::TM_B, be);
      tmem_wait_ld();
#pragma unroll
      for (int h = 0; h < 8; ++h) {
        const float t = (__uint_as_float(u[h]) + __uint_as_float(u[h + 8])) +
                        (__uint_as_float(be[h]) + __uint_as_float(be[h + 8]));
        acc[h] = fmaf(acc[h], alpha[h], cv * t);
      }
    }
    if (rescale) {
#pragma unroll
      for (int h = 0; h < 8; ++h) alpha[h] = 1.f;
    }
    tc_fence_before();
  }

  if (to) {
    if (tid == 0) set_error(A.err, KVARN_DEVERR_TIMEOUT);
    // let the copies and products this CTA started finish before its
    // shared and tensor memory go away
    for (int j = i; j < issued; ++j) mbar_wait_bounded(bars + j % S::STAGES, (j / S::STAGES) & 1, 100000000LL);
    mbar_wait_bounded(barQ, i & 1, 100000000LL);
    mbar_wait_bounded(barP, i & 1, 100000000LL);
  }

  // ---- per-head sums of the weights: warp sums, then across the warps of
  //      the head's group
  __syncthreads();
  float* lred = tmax;  // [NWARP][8]
#pragma unroll
  for (int j = 0; j < S::HPT; ++j) {
    const float v = warp_sum_xor(lpart[j], 1, 32);
    if (lane == 0) lred[warp * 8 + j] = v;
  }
  __syncthreads();
#pragma unroll
  for (int h = 0; h < 8; ++h) {
    if (h >= G) break;
    float* part = A.ws + (static_cast<int64_t>(b * A.Hq + kvh * G + h) * A.slots + split) * kPStride(D);
    part[4 + tid] = to ? 0.f : acc[h];
    if (tid == 0) {
      const int grp = h / S::HPT, j = h % S::HPT;
      float l = 0.f;
      for (int w = 0; w < 4; ++w) l += lred[(4 * grp + w) * 8 + j];
      part[0] = to ? -INFINITY : m[h];
      part[1] = to ? 0.f : l;
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc<S::TM_COLS>(tbase);
}

// ------------------------------------------------------------- planning
int device_sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
    return 148;
  return n;
}

SplitPlan plan_dense(int32_t num_seqs, int32_t num_kv_heads, int32_t max_seq_len, int32_t N,
                     int32_t warps, int32_t ctas_per_sm) {
  SplitPlan p{};
  const int tiles = max_seq_len / N;
  const int units = std::max(1, num_seqs * num_kv_heads);
  if (tiles == 0) {
    p.tiles_per_split = 1;
    p.nsplit = 0;
  } else {
    // Split count whose CTA count fills whole waves best (resident CTAs per
    // SM times the SM count), keeping at least 4 tiles per concurrently
    // processed tile slot of a CTA (`warps`); ties go to
    // fewer splits (fewer partials to merge).
    const double slots = static_cast<double>(device_sm_count()) * ctas_per_sm;
    const int max_split = std::max(1, tiles / (4 * warps));
    int best = 1;
    double best_eff = 0.0;
    for (int n = 1; n <= max_split; ++n) {
      const double waves = units * static_cast<double>(n) / slots;
      const double eff = waves / std::ceil(waves);
      if (eff > best_eff + 0.02) {
        best_eff = eff;
        best = n;
      }
    }
    p.tiles_per_split = (tiles + best - 1) / best;
    p.nsplit = (tiles + p.tiles_per_split - 1) / p.tiles_per_split;
  }
  p.slots = p.nsplit + 1;
  return p;
}

// Tiles a CTA of the compressed decode works on at once (the whole CTA
// cooperates on one tile).
int dense_decode_warps(int32_t) { return 1; }

// CTAs of the compressed decode kernel resident on one SM: bounded by the
// 512 tensor-memory columns (128 per CTA for head_dim 128, 256 for 256).
int dense_decode_ctas_per_sm(int32_t D, int32_t) { return D == 256 ? 2 : 4; }

int64_t dense_workspace_bytes(int32_t num_seqs, int32_t num_q_heads, int32_t D,
                              const SplitPlan& plan) {
  return static_cast<int64_t>(num_seqs) * num_q_heads * plan.slots * kPStride(D) * 4;
}

template <int D, int N, typename T>
static cudaError_t run_dense(const DecArgs& A, int num_seqs, cudaStream_t st) {
  using S = DecShape<D, N>;
  auto kern = decode_dense_kernel<D, N, T>;
  const int smem = std::max(S::OFF_PAGES + A.tps * S::PPT * 4, S::SMEM_FLOOR);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  dim3 grid(A.Hkv, A.nsplit + 1, num_seqs);
  kern<<<grid, S::NT, smem, st>>>(A);
  return cudaGetLastError();
}

cudaError_t launch_decode_dense(const DecodeParams& p, const SplitPlan& plan, cudaStream_t st) {
  if (p.num_seqs == 0) return cudaSuccess;
  DecArgs A{};
  A.q = p.q;
  A.kappa = p.sm_scale * kLog2e;
  A.cache = p.cache;
  A.Hq = p.num_q_heads;
  A.Hkv = p.num_kv_heads;
  A.G = p.num_q_heads / p.num_kv_heads;
  A.num_pages = p.num_pages;
  A.bt = p.block_table;
  A.bt_stride = p.bt_stride;
  A.seq_lens = p.seq_lens;
  A.max_seq_len = p.max_seq_len;
  A.tail_k = p.tail_k;
  A.tail_v = p.tail_v;
  A.ws = static_cast<float*>(p.workspace);
  A.tps = plan.tiles_per_split;
  A.nsplit = plan.nsplit;
  A.slots = plan.slots;
  A.err = p.err;
  cudaError_t e = cudaErrorInvalidValue;
#define KV_DISPATCH(DD, NN)                                                            \
  if (p.D == DD && p.N == NN)                                                          \
    e = p.bf16 ? run_dense<DD, NN, __nv_bfloat16>(A, p.num_seqs, st)                   \
               : run_dense<DD, NN, __half>(A, p.num_seqs, st);
  KV_DISPATCH(128, 128)
  KV_DISPATCH(128, 64)
  KV_DISPATCH(256, 128)
  KV_DISPATCH(256, 64)
#undef KV_DISPATCH
  if (e != cudaSuccess) return e;
  const int rows = p.num_seqs * p.num_q_heads;
  if (p.D == 128)
    merge_kernel<128><<<(rows + 3) / 4, 128, 0, st>>>(A.ws, A.slots, rows, A.nsplit, p.out, p.lse);
  else
    merge_kernel<256><<<(rows + 3) / 4, 128, 0, st>>>(A.ws, A.slots, rows, A.nsplit, p.out, p.lse);
  return cudaGetLastError();
}

}  // namespace kvarn

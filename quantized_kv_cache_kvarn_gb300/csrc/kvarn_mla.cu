// MLA latent-cache decode, sm_103a.
//
// KVarN review, MLA paragraph: the compressed latent is quantised to int4;
// one code set serves as key and value, the rope part stays fp16. Query head
// h scores token i as sm_scale (q_lat . latent_i + q_rope . rope_i), with the
// latent dequantised inline from its codes (rotated basis, scales folded in
// as for the dense cache), and returns sum_i p_i latent_i.
//
// One CTA per (group of 16 heads, split, sequence), 8 warps. Per 128-token
// tile, staged by one-dimensional bulk copies:
//   * the CTA writes the tile's A operand to shared memory once: q~ =
//     (kappa q_lat H) * c split into fp16 hi and lo planes, plus the rope
//     query (kappa q_rope, hi and lo), 16 rows x 576 columns;
//   * Q K: warp w scores the 16 tokens of page w for all 16 heads with
//     mma.sync m16n8k16; the B fragments are the page's packed codes turned
//     into exact fp16 integers (code - 8) in registers; hi and lo A planes
//     accumulate into one fp32 tile, rope into a second one;
//   * the row scales fold in, the CTA agrees on the tile maximum per head
//     through shared memory, and the weights p * a go to shared memory as
//     the A operand of P V, split into fp16 hi and lo planes;
//   * P V: warp w owns 64 of the 512 channels; it reads the same packed
//     codes (token-major) and transposes each 8x8 fp16 block with movmatrix
//     into the channel-major B fragments, so one packed copy serves both
//     products;
//   * acc = acc * alpha + c * (u + sum p (b + 8 a)) per channel.
// The partials merge in the dense merge kernel (inverse Hadamard of width
// 512). The tail (tokens past the last full tile) is scored in fp32 by the
// extra split, in the original basis.
#include <math.h>

#include <algorithm>

#include "kvarn_common.cuh"
#include "kvarn_launch.h"
#include "kvarn_merge.cuh"

namespace kvarn {

namespace {

constexpr int kDl = 512, kR = 64, kN = 128, kPPT = kN / kPageTokens;
constexpr int kHeads = 16;                   // heads per CTA
constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr LatentPage kPG{kDl, kR, kN};
constexpr int kPB = kPG.bytes();             // 6528
constexpr int kTile = kPPT * kPB;            // 52224
constexpr int kLDA = kDl + kR + 8;           // A-plane row stride in halves (padded)
constexpr int kLDP = kN + 8;                 // P-plane row stride in halves (padded)
constexpr int kMlaPStride = kDl + 4;
constexpr float kLog2eM = 1.4426950408889634f;

// shared-memory map
constexpr int kStages = 2;
constexpr int kOffStage = 0;                                   // tile pages, two stages
constexpr int kOffQ = kOffStage + kStages * kTile;             // q' [16][512] fp32
constexpr int kOffAhi = kOffQ + kHeads * kDl * 4;              // A hi [16][kLDA] f16
constexpr int kOffAlo = kOffAhi + kHeads * kLDA * 2;           // A lo
constexpr int kOffP = kOffAlo + kHeads * kLDA * 2;             // P hi [16][kLDP] f16
constexpr int kOffPlo = kOffP + kHeads * kLDP * 2;             // P lo
constexpr int kOffRed = kOffPlo + kHeads * kLDP * 2;           // [8 warps][16] floats x 2
constexpr int kOffQsum = kOffRed + 2 * kWarps * kHeads * 4;    // [16]
constexpr int kOffBar = kOffQsum + kHeads * 4;                 // mbarriers, one per stage
constexpr int kOffPages = kOffBar + 8 * kStages;               // page ids
constexpr int kSmemBase = kOffPages;
static_assert(kOffAhi % 16 == 0 && kOffP % 16 == 0 && kOffPlo % 16 == 0 && kOffBar % 8 == 0, "alignment");

struct MlaArgs {
  const void* ql;
  const void* qr;
  float kappa;
  const uint8_t* cache;
  int32_t H;
  int64_t num_pages;
  const int32_t* bt;
  int32_t bt_stride;
  const int32_t* seq_lens;
  int32_t max_seq_len;
  const void* tail_lat;
  const __half* tail_rope;
  float* ws;
  int32_t tps, nsplit, slots;
  uint32_t* err;
};

__device__ __forceinline__ void ldsm_x4(uint32_t* r, const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(smem_addr(p)));
}

__device__ __forceinline__ uint32_t movm_t(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}

template <typename T>
__device__ void mla_tail(const MlaArgs& A, int b, int hg, int tail, unsigned char* smem) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  float* sbuf = reinterpret_cast<float*>(smem) + warp * kN;
  for (int hl = warp; hl < kHeads; hl += kWarps) {
    const int h = hg * kHeads + hl;
    float* part = A.ws + (static_cast<int64_t>(b * A.H + h) * A.slots + A.nsplit) * kMlaPStride;
    if (tail == 0 || !A.tail_lat || !A.tail_rope) {
      if (tail > 0 && lane == 0) set_error(A.err, KVARN_DEVERR_NO_TAIL);
      if (lane == 0) { part[0] = -INFINITY; part[1] = 0.f; }
      for (int j = lane; j < kDl; j += 32) part[4 + j] = 0.f;
      continue;
    }
    float ql[16], qr[2];
    const T* qlp = static_cast<const T*>(A.ql) + static_cast<int64_t>(b * A.H + h) * kDl + lane * 16;
    load8<T>(qlp, ql);
    load8<T>(qlp + 8, ql + 8);
    const T* qrp = static_cast<const T*>(A.qr) + static_cast<int64_t>(b * A.H + h) * kR + lane * 2;
    qr[0] = to_f32<T>(qrp[0]) * A.kappa;
    qr[1] = to_f32<T>(qrp[1]) * A.kappa;
#pragma unroll
    for (int e = 0; e < 16; ++e) ql[e] *= A.kappa;
    const T* tl = static_cast<const T*>(A.tail_lat) + static_cast<int64_t>(b) * kN * kDl;
    const __half* tr = A.tail_rope + static_cast<int64_t>(b) * kN * kR;
    float mx = -INFINITY;
    for (int tau = 0; tau < tail; ++tau) {
      float kvv[16];
      load8<T>(tl + tau * kDl + lane * 16, kvv);
      load8<T>(tl + tau * kDl + lane * 16 + 8, kvv + 8);
      float dot = qr[0] * __half2float(tr[tau * kR + lane * 2]) + qr[1] * __half2float(tr[tau * kR + lane * 2 + 1]);
#pragma unroll
      for (int e = 0; e < 16; ++e) dot = fmaf(ql[e], kvv[e], dot);
      dot = warp_sum_xor(dot, 1, 32);
      if (lane == 0) sbuf[tau] = dot;
      mx = fmaxf(mx, dot);
    }
    __syncwarp();
    float l = 0.f, acc[16];
#pragma unroll
    for (int e = 0; e < 16; ++e) acc[e] = 0.f;
    for (int tau = 0; tau < tail; ++tau) {
      const float p = exp2f(sbuf[tau] - mx);
      l += p;
      float vv[16];
      load8<T>(tl + tau * kDl + lane * 16, vv);
      load8<T>(tl + tau * kDl + lane * 16 + 8, vv + 8);
#pragma unroll
      for (int e = 0; e < 16; ++e) acc[e] = fmaf(p, vv[e], acc[e]);
    }
    __syncwarp();
    if (lane == 0) { part[0] = mx; part[1] = l; }
#pragma unroll
    for (int e = 0; e < 16; ++e) part[4 + lane * 16 + e] = acc[e];
    __syncwarp();
  }
}

template <typename T>
__global__ void __launch_bounds__(kThreads, 1) mla_decode_kernel(MlaArgs A) {
  extern __shared__ __align__(128) unsigned char smem[];
  pdl_launch_dependents();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, t = lane & 3;
  const int hg = blockIdx.x, split = blockIdx.y, b = blockIdx.z;
  const int h0 = hg * kHeads;

  int len = A.seq_lens[b];
  if (len < 0 || len > A.max_seq_len) {
    if (tid == 0) set_error(A.err, KVARN_DEVERR_SEQ_LEN);
    len = len < 0 ? 0 : A.max_seq_len;
  }
  const int ntiles = len / kN;
  if (split == A.nsplit) {
    mla_tail<T>(A, b, hg, len - ntiles * kN, smem);
    return;
  }
  const int t0 = split * A.tps, t1 = min(t0 + A.tps, ntiles);
  if (t0 >= t1) {
    for (int hl = warp; hl < kHeads; hl += kWarps) {
      float* part = A.ws + (static_cast<int64_t>(b * A.H + h0 + hl) * A.slots + split) * kMlaPStride;
      if (lane == 0) { part[0] = -INFINITY; part[1] = 0.f; }
      for (int j = lane; j < kDl; j += 32) part[4 + j] = 0.f;
    }
    return;
  }

  float* qrot = reinterpret_cast<float*>(smem + kOffQ);
  __half* Ahi = reinterpret_cast<__half*>(smem + kOffAhi);
  __half* Alo = reinterpret_cast<__half*>(smem + kOffAlo);
  __half* Pm = reinterpret_cast<__half*>(smem + kOffP);
  __half* Pl = reinterpret_cast<__half*>(smem + kOffPlo);
  float* red = reinterpret_cast<float*>(smem + kOffRed);
  float* qsum = reinterpret_cast<float*>(smem + kOffQsum);
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + kOffBar);
  int32_t* pages = reinterpret_cast<int32_t*>(smem + kOffPages);
  const int32_t* bt = A.bt + static_cast<int64_t>(b) * A.bt_stride;

  for (int e = tid; e < (t1 - t0) * kPPT; e += kThreads) {
    int phys = bt[t0 * kPPT + e];
    if (phys < 0 || phys >= A.num_pages) {
      set_error(A.err, KVARN_DEVERR_PAGE_RANGE);
      phys = 0;
    }
    pages[e] = phys;
  }
  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) mbar_init(bar + s, 1);
  }
  fence_mbar_init();
  __syncthreads();

  // tile `tile` of the split lives in stage (tile - t0) % 2
  auto stage_of = [&](int tile) -> unsigned char* { return smem + kOffStage + ((tile - t0) & 1) * kTile; };
  auto issue = [&](int tile) {  // warp 0
    uint64_t* sb = bar + ((tile - t0) & 1);
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) mbar_arrive_expect_tx(sb, kTile);
    __syncwarp();
    if (lane < kPPT)
      bulk_g2s(stage_of(tile) + lane * kPB,
               A.cache + static_cast<int64_t>(pages[(tile - t0) * kPPT + lane]) * kPB, kPB, sb);
  };
  if (warp == 0) {
    issue(t0);
    if (t0 + 1 < t1) issue(t0 + 1);
    if (t0 + 2 < t1 && lane < kPPT)
      prefetch_l2(A.cache + static_cast<int64_t>(pages[2 * kPPT + lane]) * kPB, kPB);
  }

  // ---- rotated, scaled latent query rows (q'), rope query planes (once)
  for (int hl = warp; hl < kHeads; hl += kWarps) {
    const int h = h0 + hl;
    float v[16];
    const T* qp = static_cast<const T*>(A.ql) + static_cast<int64_t>(b * A.H + h) * kDl + lane * 16;
    load8<T>(qp, v);
    load8<T>(qp + 8, v + 8);
    warp_fwht<16>(v);
    const float sc = A.kappa / sqrtf(static_cast<float>(kDl));
#pragma unroll
    for (int e = 0; e < 16; ++e) qrot[hl * kDl + lane * 16 + e] = v[e] * sc;
    const T* qr = static_cast<const T*>(A.qr) + static_cast<int64_t>(b * A.H + h) * kR + lane * 2;
    uint32_t hi, lo;
    split_hi_lo(to_f32<T>(qr[0]) * A.kappa, to_f32<T>(qr[1]) * A.kappa, hi, lo);
    *reinterpret_cast<uint32_t*>(Ahi + hl * kLDA + kDl + lane * 2) = hi;
    *reinterpret_cast<uint32_t*>(Alo + hl * kLDA + kDl + lane * 2) = lo;
  }

  __syncthreads();  // q' rows and rope planes visible to every warp

  // per-thread state: heads g and g+8 (rows of the mma tiles)
  float m[2] = {-INFINITY, -INFINITY}, lsum[2] = {0.f, 0.f};
  float acc[8][4];  // P V output: 8 channel blocks of this warp, rows g / g+8
#pragma unroll
  for (int k = 0; k < 8; ++k) acc[k][0] = acc[k][1] = acc[k][2] = acc[k][3] = 0.f;
  int timed_out = 0;

  for (int tile = t0; tile < t1; ++tile) {
    const uint32_t par = ((tile - t0) >> 1) & 1;
    uint64_t* sbar = bar + ((tile - t0) & 1);
    unsigned char* stage = stage_of(tile);
    if (!mbar_wait_bounded(sbar, par)) timed_out = true;
    // -- A planes: q~ = q' * c, hi and lo, and the per-head sum of q~
    {
      // 16 threads per head; thread r takes channel pairs 2r + 32i, so that
      // neighbouring threads touch neighbouring words
      const int hl = tid >> 4, j0 = (tid & 15) * 2;
      float s = 0.f;
#pragma unroll
      for (int e = 0; e < 32; e += 2) {
        const int j = j0 + 16 * e;
        const float2 c = *reinterpret_cast<const float2*>(stage + (j / 64) * kPB + kPG.col() + (j % 64) * 4);
        const float2 q = *reinterpret_cast<const float2*>(qrot + hl * kDl + j);
        const float x0 = q.x * c.x, x1 = q.y * c.y;
        s += x0 + x1;
        uint32_t hi, lo;
        split_hi_lo(x0, x1, hi, lo);
        *reinterpret_cast<uint32_t*>(Ahi + hl * kLDA + j) = hi;
        *reinterpret_cast<uint32_t*>(Alo + hl * kLDA + j) = lo;
      }
      s = warp_sum_xor(s, 1, 16);
      if ((tid & 15) == 0) qsum[hl] = s;
    }
    __syncthreads();

    // -- Q K for the 16 tokens of page `warp` (two 8-token blocks)
    const unsigned char* pg = stage + warp * kPB;
    float sl[2][4], sr[2][4];
#pragma unroll
    for (int j = 0; j < 2; ++j)
#pragma unroll
      for (int e = 0; e < 4; ++e) sl[j][e] = sr[j][e] = 0.f;
    // ldmatrix addresses: lane supplies row (lane & 15), column block 8*(lane >> 4)
    const __half* arow_hi = Ahi + (lane & 15) * kLDA + 8 * (lane >> 4);
    const __half* arow_lo = Alo + (lane & 15) * kLDA + 8 * (lane >> 4);
#pragma unroll 2
    for (int q4 = 0; q4 < 4; ++q4) {  // 8 k-chunks (4 words) per step
      uint4 kw[2];
#pragma unroll
      for (int j = 0; j < 2; ++j)
        kw[j] = *reinterpret_cast<const uint4*>(pg + (j * 8 + g) * (kDl / 2) + 16 * ((4 * q4 + t) ^ (4 * (g & 1))));
#pragma unroll
      for (int w4 = 0; w4 < 4; ++w4) {
        uint32_t bf[2][4];
#pragma unroll
        for (int j = 0; j < 2; ++j)
          dequant_k_word(w4 == 0 ? kw[j].x : w4 == 1 ? kw[j].y : w4 == 2 ? kw[j].z : kw[j].w, bf[j]);
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
          const int kc = 8 * q4 + 2 * w4 + h2;
          uint32_t ah[4], al[4];
          ldsm_x4(ah, arow_hi + 16 * kc);
          ldsm_x4(al, arow_lo + 16 * kc);
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            mma_f16(sl[j], ah[0], ah[1], ah[2], ah[3], bf[j][2 * h2], bf[j][2 * h2 + 1]);
            mma_f16(sl[j], al[0], al[1], al[2], al[3], bf[j][2 * h2], bf[j][2 * h2 + 1]);
          }
        }
      }
    }
    // rope: fp16 rows in the page, B fragments straight from shared memory
#pragma unroll
    for (int kc = 0; kc < kR / 16; ++kc) {
      uint32_t ah[4], al[4];
      ldsm_x4(ah, arow_hi + kDl + 16 * kc);
      ldsm_x4(al, arow_lo + kDl + 16 * kc);
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const __half* rp = reinterpret_cast<const __half*>(pg + kPG.rope()) + (j * 8 + g) * kR + 16 * kc + 2 * t;
        const uint32_t b0 = *reinterpret_cast<const uint32_t*>(rp);
        const uint32_t b1 = *reinterpret_cast<const uint32_t*>(rp + 8);
        mma_f16(sr[j], ah[0], ah[1], ah[2], ah[3], b0, b1);
        mma_f16(sr[j], al[0], al[1], al[2], al[3], b0, b1);
      }
    }
    // -- fold row scales; scores of heads g (e = 0, 1) and g + 8 (e = 2, 3)
    const float qs0 = qsum[g], qs1 = qsum[g + 8];
    float s[2][4];
    float mt0 = -INFINITY, mt1 = -INFINITY;
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const int idx = j * 8 + 2 * t;
      const float2 ka = *reinterpret_cast<const float2*>(pg + kPG.a() + idx * 4);
      const float2 kb = *reinterpret_cast<const float2*>(pg + kPG.b() + idx * 4);
      const float b0 = fmaf(8.f, ka.x, kb.x), b1 = fmaf(8.f, ka.y, kb.y);
      s[j][0] = fmaf(ka.x, sl[j][0], fmaf(b0, qs0, sr[j][0]));
      s[j][1] = fmaf(ka.y, sl[j][1], fmaf(b1, qs0, sr[j][1]));
      s[j][2] = fmaf(ka.x, sl[j][2], fmaf(b0, qs1, sr[j][2]));
      s[j][3] = fmaf(ka.y, sl[j][3], fmaf(b1, qs1, sr[j][3]));
      mt0 = fmaxf(mt0, fmaxf(s[j][0], s[j][1]));
      mt1 = fmaxf(mt1, fmaxf(s[j][2], s[j][3]));
    }
    mt0 = warp_max_xor(mt0, 1, 4);
    mt1 = warp_max_xor(mt1, 1, 4);
    if (t == 0) {
      red[warp * kHeads + g] = mt0;
      red[warp * kHeads + g + 8] = mt1;
    }
    __syncthreads();
    float mn0 = m[0], mn1 = m[1];
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      mn0 = fmaxf(mn0, red[w * kHeads + g]);
      mn1 = fmaxf(mn1, red[w * kHeads + g + 8]);
    }
    const float al0 = fast_exp2(m[0] - mn0), al1 = fast_exp2(m[1] - mn1);
    m[0] = mn0;
    m[1] = mn1;
    // -- weights p * a (fp16 A operand of P V) and the offset sums
    float ps0 = 0.f, ps1 = 0.f, be0 = 0.f, be1 = 0.f;
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const int idx = j * 8 + 2 * t;
      const float2 ka = *reinterpret_cast<const float2*>(pg + kPG.a() + idx * 4);
      const float2 kb = *reinterpret_cast<const float2*>(pg + kPG.b() + idx * 4);
      const float p0 = fast_exp2(s[j][0] - mn0), p1 = fast_exp2(s[j][1] - mn0);
      const float p2 = fast_exp2(s[j][2] - mn1), p3 = fast_exp2(s[j][3] - mn1);
      ps0 += p0 + p1;
      ps1 += p2 + p3;
      const float b0 = fmaf(8.f, ka.x, kb.x), b1 = fmaf(8.f, ka.y, kb.y);
      be0 = fmaf(p0, b0, fmaf(p1, b1, be0));
      be1 = fmaf(p2, b0, fmaf(p3, b1, be1));
      const int tok = warp * kPageTokens + idx;
      uint32_t hi, lo;
      split_hi_lo(p0 * ka.x, p1 * ka.y, hi, lo);
      *reinterpret_cast<uint32_t*>(Pm + g * kLDP + tok) = hi;
      *reinterpret_cast<uint32_t*>(Pl + g * kLDP + tok) = lo;
      split_hi_lo(p2 * ka.x, p3 * ka.y, hi, lo);
      *reinterpret_cast<uint32_t*>(Pm + (g + 8) * kLDP + tok) = hi;
      *reinterpret_cast<uint32_t*>(Pl + (g + 8) * kLDP + tok) = lo;
    }
    lsum[0] = fmaf(lsum[0], al0, ps0);
    lsum[1] = fmaf(lsum[1], al1, ps1);
    be0 = warp_sum_xor(be0, 1, 4);
    be1 = warp_sum_xor(be1, 1, 4);
    __syncthreads();  // everyone has read red (maxima) before it is reused
    if (t == 0) {
      red[warp * kHeads + g] = be0;
      red[warp * kHeads + g + 8] = be1;
    }
    __syncthreads();
    float beta0 = 0.f, beta1 = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      beta0 += red[w * kHeads + g];
      beta1 += red[w * kHeads + g + 8];
    }

    // -- P V for channels [64 warp, +64): eight 8-channel blocks
    float u[8][4];
#pragma unroll
    for (int k = 0; k < 8; ++k) u[k][0] = u[k][1] = u[k][2] = u[k][3] = 0.f;
    const __half* prow = Pm + (lane & 15) * kLDP + 8 * (lane >> 4);
    const __half* prow_lo = Pl + (lane & 15) * kLDP + 8 * (lane >> 4);
#pragma unroll 2
    for (int pp = 0; pp < kPPT; ++pp) {
      uint32_t ap[4], aq[4];
      ldsm_x4(ap, prow + 16 * pp);
      ldsm_x4(aq, prow_lo + 16 * pp);
      const unsigned char* cp = stage + pp * kPB;
      // codes of page tokens g and 8+g, channels 16kc..16kc+15 for kc = 4 warp .. 4 warp + 3
      // latent unit order: unit 4q + t at (4q + t) XOR 4 (tau % 2); this
      // warp's words 2 warp, 2 warp + 1 are unit q = warp / 2, bytes 8 (warp % 2)
      const int uo = 16 * ((4 * (warp >> 1) + t) ^ (4 * (g & 1))) + 8 * (warp & 1);
      const uint2 w0 = *reinterpret_cast<const uint2*>(cp + g * (kDl / 2) + uo);
      const uint2 w1 = *reinterpret_cast<const uint2*>(cp + (8 + g) * (kDl / 2) + uo);
#pragma unroll
      for (int wi = 0; wi < 2; ++wi) {
        uint32_t f0[4], f1[4];
        dequant_k_word(wi ? w0.y : w0.x, f0);  // token g:   (kc even: b01, b23), (kc odd: b01, b23)
        dequant_k_word(wi ? w1.y : w1.x, f1);  // token 8+g
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
          // channel block 16kc + 0..7 and 16kc + 8..15 of k-chunk kc = 4 warp + 2 wi + h2
          const int nc = 4 * wi + 2 * h2;  // local channel block of this warp
          const uint32_t b0 = movm_t(f0[2 * h2]), b1 = movm_t(f1[2 * h2]);
          const uint32_t b2 = movm_t(f0[2 * h2 + 1]), b3 = movm_t(f1[2 * h2 + 1]);
          mma_f16(u[nc], ap[0], ap[1], ap[2], ap[3], b0, b1);
          mma_f16(u[nc], aq[0], aq[1], aq[2], aq[3], b0, b1);
          mma_f16(u[nc + 1], ap[0], ap[1], ap[2], ap[3], b2, b3);
          mma_f16(u[nc + 1], aq[0], aq[1], aq[2], aq[3], b2, b3);
        }
      }
    }
    // -- fold the column scales: channel 64 warp + 8 nc + 2t + {0, 1}
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int ch = 64 * warp + 8 * k + 2 * t;
      const float2 c = *reinterpret_cast<const float2*>(stage + (ch / 64) * kPB + kPG.col() + (ch % 64) * 4);
      acc[k][0] = fmaf(acc[k][0], al0, c.x * (u[k][0] + beta0));
      acc[k][1] = fmaf(acc[k][1], al0, c.y * (u[k][1] + beta0));
      acc[k][2] = fmaf(acc[k][2], al1, c.x * (u[k][2] + beta1));
      acc[k][3] = fmaf(acc[k][3], al1, c.y * (u[k][3] + beta1));
    }
    // stage, A planes, P and red are free; a copy that never landed stops
    // the whole CTA (uniformly) after waiting a bounded time for it
    if (__syncthreads_or(timed_out)) {
      if (tid == 0) set_error(A.err, KVARN_DEVERR_TIMEOUT);
      // the copies still in flight: this tile's stage and the next one's
      mbar_wait_bounded(sbar, par, 100000000LL);
      if (tile + 1 < t1) mbar_wait_bounded(bar + ((tile + 1 - t0) & 1), ((tile + 1 - t0) >> 1) & 1, 100000000LL);
      break;
    }
    // this stage is free: refill it with tile + 2
    if (warp == 0 && tile + 2 < t1) {
      issue(tile + 2);
      if (tile + 3 < t1 && lane < kPPT)
        prefetch_l2(A.cache + static_cast<int64_t>(pages[(tile + 3 - t0) * kPPT + lane]) * kPB, kPB);
    }
  }

  // ---- partial of this split: m, l (summed over all lanes of all warps), acc
  lsum[0] = warp_sum_xor(lsum[0], 1, 4);
  lsum[1] = warp_sum_xor(lsum[1], 1, 4);
  if (t == 0) {
    red[warp * kHeads + g] = lsum[0];
    red[warp * kHeads + g + 8] = lsum[1];
  }
  __syncthreads();
  if (tid < kHeads) {
    float L = 0.f;
    for (int w = 0; w < kWarps; ++w) L += red[w * kHeads + tid];
    float* part = A.ws + (static_cast<int64_t>(b * A.H + h0 + tid) * A.slots + split) * kMlaPStride;
    part[1] = L;
  }
  if (t == 0) {
    float* p0 = A.ws + (static_cast<int64_t>(b * A.H + h0 + g) * A.slots + split) * kMlaPStride;
    float* p1 = A.ws + (static_cast<int64_t>(b * A.H + h0 + g + 8) * A.slots + split) * kMlaPStride;
    if (warp == 0) {
      p0[0] = m[0];
      p1[0] = m[1];
    }
  }
  float* p0 = A.ws + (static_cast<int64_t>(b * A.H + h0 + g) * A.slots + split) * kMlaPStride + 4;
  float* p1 = A.ws + (static_cast<int64_t>(b * A.H + h0 + g + 8) * A.slots + split) * kMlaPStride + 4;
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const int ch = 64 * warp + 8 * k + 2 * t;
    *reinterpret_cast<float2*>(p0 + ch) = make_float2(acc[k][0], acc[k][1]);
    *reinterpret_cast<float2*>(p1 + ch) = make_float2(acc[k][2], acc[k][3]);
  }
}

}  // namespace

SplitPlan plan_mla(int32_t num_seqs, int32_t max_seq_len) {
  SplitPlan p{};
  const int tiles = max_seq_len / kN;
  if (tiles == 0) {
    p.tiles_per_split = 1;
    p.nsplit = 0;
  } else {
    // CTAs of 16 heads: 8 per (sequence, split) at 128 heads; one CTA per SM
    // Every split writes a 512-float partial per head that the merge reads
    // back, so take the fewest splits whose wave efficiency is within 0.05
    // of the best one.
    const double slots = device_sm_count();
    const int units = std::max(1, num_seqs) * 8;
    const int max_split = std::max(1, tiles / 2);
    auto eff_of = [&](int n) {
      const double waves = units * static_cast<double>(n) / slots;
      return waves / std::ceil(waves);
    };
    double top = 0.0;
    for (int n = 1; n <= max_split; ++n) top = std::max(top, eff_of(n));
    int best = 1;
    while (best < max_split && eff_of(best) < top - 0.05) ++best;
    p.tiles_per_split = (tiles + best - 1) / best;
    p.nsplit = (tiles + p.tiles_per_split - 1) / p.tiles_per_split;
  }
  p.slots = p.nsplit + 1;
  return p;
}

int64_t mla_workspace_bytes(int32_t num_seqs, int32_t num_heads, const SplitPlan& plan) {
  return static_cast<int64_t>(num_seqs) * num_heads * plan.slots * kMlaPStride * 4;
}

cudaError_t launch_decode_mla(const DecodeParams& p, const SplitPlan& plan, cudaStream_t st) {
  if (p.num_seqs == 0) return cudaSuccess;
  MlaArgs A{};
  A.ql = p.q;
  A.qr = p.q_rope;
  A.kappa = p.sm_scale * kLog2eM;
  A.cache = p.cache;
  A.H = p.num_q_heads;
  A.num_pages = p.num_pages;
  A.bt = p.block_table;
  A.bt_stride = p.bt_stride;
  A.seq_lens = p.seq_lens;
  A.max_seq_len = p.max_seq_len;
  A.tail_lat = p.tail_k;
  A.tail_rope = static_cast<const __half*>(p.tail_v);
  A.ws = static_cast<float*>(p.workspace);
  A.tps = plan.tiles_per_split;
  A.nsplit = plan.nsplit;
  A.slots = plan.slots;
  A.err = p.err;
  const int smem = kSmemBase + plan.tiles_per_split * kPPT * 4;
  auto kern = p.bf16 ? mla_decode_kernel<__nv_bfloat16> : mla_decode_kernel<__half>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  dim3 grid(p.num_q_heads / kHeads, plan.nsplit + 1, p.num_seqs);
  kern<<<grid, kThreads, smem, st>>>(A);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int rows = p.num_seqs * p.num_q_heads;
  return launch_merge<512>(A.ws, A.slots, rows, nullptr, A.nsplit, A.nsplit, p.out, p.lse, st);
}

}  // namespace kvarn

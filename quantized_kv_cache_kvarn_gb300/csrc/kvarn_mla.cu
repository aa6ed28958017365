// MLA latent-cache decode, sm_103a.
//
// KVarN review, MLA paragraph: the compressed latent is quantised to int4;
// one code set serves as key and value, the rope part stays fp16. Query head
// h scores token i as sm_scale (q_lat . latent_i + q_rope . rope_i), with the
// latent dequantised inline from its codes (rotated basis, scales folded in
// as for the dense cache), and returns sum_i p_i latent_i.
//
// The committed tiles go through the tensor-core (tcgen05) kernel below,
// two CTAs per (split, sequence) with the accumulators in tensor memory. The
// partials merge in the dense merge kernel (inverse Hadamard of width 512).
// The tail (tokens past the last full tile) is scored in fp32 by the extra
// split, in the original basis.
#include <math.h>

#include <algorithm>

#include "kvarn_common.cuh"
#include "kvarn_launch.h"
#include "kvarn_merge.cuh"
#include "kvarn_tcgen05.cuh"

namespace kvarn {

namespace {

constexpr int kDl = 512, kR = 64, kN = 128, kPPT = kN / kPageTokens;
constexpr int kHeads = 16;                   // heads per tail group
constexpr int kWarps = 8;                    // warps that score the tail
constexpr LatentPage kPG{kDl, kR, kN};
constexpr int kPB = kPG.bytes();             // 6528
constexpr int kTile = kPPT * kPB;            // 52224
constexpr int kMlaPStride = kDl + 4;
constexpr float kLog2eM = 1.4426950408889634f;

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
  float* qbuf;          // q' rows [num_seqs][128][Dl] fp32 (workspace)
  unsigned char* qimg;  // rope query hi/lo operand image [num_seqs][2][128][128 B] (workspace)
};

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

// ---------------------------------------------------------------------------
// Tensor-core (tcgen05) decode. Two CTAs per (split, sequence): CTA `half`
// owns the latent output channels [256 half, +256); both score the whole
// tile for all 128 (zero-padded) heads in the same order, so that their
// weights agree bit for bit. Per 128-token tile:
//   * producer warps (8) expand the page codes into exact fp16 (code - 8)
//     operand blocks (128 tokens x 64 channels, 128-byte swizzle) and build
//     q~ = q' * c as fp16 hi and lo planes chunk by chunk (2-stage ring);
//   * one thread issues S = q~ K^T (latent: 8 chunks x 4 k-steps x 2 planes)
//     and the rope scores into two tensor-memory accumulators (M = 128
//     heads, N = 128 tokens);
//   * consumer warps (4, thread = head = tensor-memory lane) fold the row
//     scales (s = a S_lat + b' w + S_rope), run the online softmax and write
//     the weights p * a as fp16 hi and lo planes (the A operand of P V);
//   * P V (K = 128 tokens, N = 2 x 128 own channels, the codes read as an
//     MN-major operand of the same blocks) lands in tensor memory, and the
//     consumers fold it in: acc = alpha acc + c (u + beta), acc kept in
//     tensor memory (256 columns).
// Tensor memory: [0, 128) latent scores, then P V channels 0..127;
// [128, 256) rope scores, then P V channels 128..255; [256, 512) acc.
namespace tc {
constexpr int kM = 128;                   // heads per CTA (zero-padded)
constexpr int kCh = 64;                   // channels per K chunk
constexpr int kChunks = kDl / kCh + 1;    // eight latent chunks, then rope
constexpr int kBlk = kM * 128;            // one 128-row x 128-byte operand block
constexpr int kStage = 3 * kBlk;          // ring stage: A hi, A lo, B
constexpr int kOffOwn = 0;                // this half's four latent code blocks
constexpr int kOffRing = kOffOwn + 4 * kBlk;
constexpr int kOffP = kOffRing;           // P hi (2 K blocks), P lo (2); aliases the ring
constexpr int kOffRaw = kOffRing + 2 * kStage;
constexpr int kMeta = (kDl + 3 * kM) * 4;  // c[512], a[128], b' = b + 8a [128], w[128]
constexpr int kOffMeta = kOffRaw + kTile;
constexpr int kOffBar = kOffMeta + 2 * kMeta;
constexpr int kSmem = kOffBar + 128 + 1024;  // + room to align the base to 1024 bytes
constexpr int kConsumers = 128, kProducers = 256;
constexpr int kThreads = kConsumers + kProducers + 32;
constexpr int kMmaWarp = kThreads / 32 - 1;
// BAR_OFULL: P V of the tile complete; BAR_OFULL_A: its first 128 channels
enum { BAR_AFULL = 0, BAR_AEMPTY = 2, BAR_SFULL = 4, BAR_PFULL, BAR_OFULL, BAR_OFULL_A, BAR_TFREE, BAR_RAW, BAR_META, BAR_PSYNC,
       BAR_FIN, NBARS };
static_assert(kOffRaw % 16 == 0 && kOffMeta % 16 == 0 && kOffBar % 8 == 0 && NBARS * 8 + 8 <= 128, "layout");
static_assert(kSmem <= 232448, "one CTA per SM");
constexpr uint32_t kIdQK = tc_idesc_f16(128, 128, false, false);
constexpr uint32_t kIdPV = tc_idesc_f16(128, 128, false, true);
constexpr long long kWaitLimit = 2000000000LL;

// fp16 (code - 8) of nibbles k and k + 4 of a latent code word (channels
// +0 and +1 of the word's k-th pair): 1024 + code by the exponent trick, then
// an exact subtraction.
__device__ __forceinline__ uint32_t code_pair_m8(uint32_t x, int k) {
  const uint32_t v = ((x >> (4 * k)) & 0x000F000Fu) | 0x64006400u;
  return h2_as_u32(__hsub2(u32_as_h2(v), __float2half2_rn(1032.f)));
}
}  // namespace tc

// One probe of an mbarrier phase without a suspend-time hint: the thread
// returns as soon as the phase completes or a short, implementation-defined
// time passes, so that hand-offs between the roles cost no wake-up delay.
__device__ __forceinline__ bool mbar_probe(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Non-blocking test of an mbarrier phase.
__device__ __forceinline__ bool mbar_test(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ void mbar_arrive_plain(uint64_t* bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

// q' = kappa q_lat H / sqrt(Dl) as fp32 rows of 128 (zero-padded) heads, and
// the rope query kappa q_rope as fp16 hi and lo planes in the swizzled
// operand layout that the decode copies into shared memory every tile.
template <typename T>
__global__ void __launch_bounds__(256) mla_qprep_kernel(MlaArgs A) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int b = blockIdx.y, h = blockIdx.x * 8 + warp;
  float v[16];
  float r0 = 0.f, r1 = 0.f;
  if (h < A.H) {
    const T* qp = static_cast<const T*>(A.ql) + static_cast<int64_t>(b * A.H + h) * kDl + lane * 16;
    load8<T>(qp, v);
    load8<T>(qp + 8, v + 8);
    warp_fwht<16>(v);
    const float sc = A.kappa / sqrtf(static_cast<float>(kDl));
#pragma unroll
    for (int e = 0; e < 16; ++e) v[e] *= sc;
    const T* qr = static_cast<const T*>(A.qr) + static_cast<int64_t>(b * A.H + h) * kR + lane * 2;
    r0 = to_f32<T>(qr[0]) * A.kappa;
    r1 = to_f32<T>(qr[1]) * A.kappa;
  } else {
#pragma unroll
    for (int e = 0; e < 16; ++e) v[e] = 0.f;
  }
  float4* dst = reinterpret_cast<float4*>(A.qbuf + (static_cast<int64_t>(b) * tc::kM + h) * kDl + lane * 16);
#pragma unroll
  for (int k = 0; k < 4; ++k) dst[k] = make_float4(v[4 * k], v[4 * k + 1], v[4 * k + 2], v[4 * k + 3]);
  uint32_t hi, lo;
  split_hi_lo(r0, r1, hi, lo);
  unsigned char* img = A.qimg + static_cast<int64_t>(b) * 2 * tc::kBlk;
  const uint32_t off = sw128_unit(h, lane >> 2) + 4 * (lane & 3);  // channels 2 lane, 2 lane + 1
  *reinterpret_cast<uint32_t*>(img + off) = hi;
  *reinterpret_cast<uint32_t*>(img + tc::kBlk + off) = lo;
}

template <typename T>
__global__ void __launch_bounds__(tc::kThreads, 1) mla_tc_kernel(MlaArgs A) {
  using namespace tc;
  extern __shared__ __align__(1024) unsigned char smem[];
  pdl_launch_dependents();
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int half = blockIdx.x, split = blockIdx.y, b = blockIdx.z;
  int len = A.seq_lens[b];
  if (len < 0 || len > A.max_seq_len) {
    if (tid == 0) set_error(A.err, KVARN_DEVERR_SEQ_LEN);
    len = len < 0 ? 0 : A.max_seq_len;
  }
  const int ntiles = len / kN;
  if (split == A.nsplit) {  // the tail: warps 0..7, the 16-head groups of this half
    if (warp < kWarps)
      for (int hg = half; hg < A.H / kHeads; hg += 2) mla_tail<T>(A, b, hg, len - ntiles * kN, smem);
    return;
  }
  const int t0 = split * A.tps, t1 = min(t0 + A.tps, ntiles);
  if (t0 >= t1) {
    for (int h = warp; h < A.H; h += tc::kThreads / 32) {
      float* part = A.ws + (static_cast<int64_t>(b * A.H + h) * A.slots + split) * kMlaPStride;
      if (half == 0 && lane == 0) {
        part[0] = -INFINITY;
        part[1] = 0.f;
      }
      for (int j = lane; j < kDl / 2; j += 32) part[4 + (kDl / 2) * half + j] = 0.f;
    }
    return;
  }
  const int n = t1 - t0;
  unsigned char* sm = smem + ((1024u - (smem_addr(smem) & 1023u)) & 1023u);
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + tc::kOffBar);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + tc::kOffBar + NBARS * 8);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + tc::kOffBar + NBARS * 8 + 4);
  const int32_t* bt = A.bt + static_cast<int64_t>(b) * A.bt_stride;
  auto issue_raw = [&](int tile) {  // one thread: the tile's eight pages into the raw stage
    mbar_arrive_expect_tx(bars + BAR_RAW, kTile);
    for (int p = 0; p < kPPT; ++p) {
      int phys = bt[tile * kPPT + p];
      if (phys < 0 || phys >= A.num_pages) {
        set_error(A.err, KVARN_DEVERR_PAGE_RANGE);
        phys = 0;
      }
      bulk_g2s(sm + kOffRaw + p * kPB, A.cache + static_cast<int64_t>(phys) * kPB, kPB, bars + BAR_RAW);
    }
  };
  // Bounded wait, uniform over the warp; gives up (and tells every role to)
  // after about a second or once another warp has given up.
  auto wait = [&](int bar, uint32_t parity) -> bool {
    if (__all_sync(0xffffffffu, mbar_test(bars + bar, parity))) return true;
    bool ok = true;
    const long long start = clock64();
    while (!mbar_probe(bars + bar, parity)) {
      if (*abort_flag || clock64() - start > kWaitLimit) {
        ok = false;
        break;
      }
    }
    ok = __all_sync(0xffffffffu, ok);
    if (!ok) *abort_flag = 1;
    return ok;
  };

  if (warp == kMmaWarp) tc_alloc(tslot, 512);
  if (tid == 0) {
    mbar_init(bars + BAR_AFULL, kProducers);
    mbar_init(bars + BAR_AFULL + 1, kProducers);
    mbar_init(bars + BAR_AEMPTY, 1);
    mbar_init(bars + BAR_AEMPTY + 1, 1);
    mbar_init(bars + BAR_SFULL, 1);
    mbar_init(bars + BAR_PFULL, kConsumers);
    mbar_init(bars + BAR_OFULL, 1);
    mbar_init(bars + BAR_OFULL_A, 1);
    mbar_init(bars + BAR_TFREE, kConsumers);
    mbar_init(bars + BAR_RAW, 1);
    mbar_init(bars + BAR_META, kProducers);
    mbar_init(bars + BAR_PSYNC, kProducers);
    mbar_init(bars + BAR_FIN, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;
  if (tid == kConsumers) issue_raw(t0);

  if (tid >= kConsumers && tid < kConsumers + kProducers) {
    // ---------------------------------------------------------- producers
    const int p = tid - kConsumers;
    // A operand: thread (warp pw, lane l) builds rows 16 pw + 2 k + l / 16
    // (k = 0..7), channels 4 (l % 16) .. + 3 of each chunk, so that a warp's
    // load of q' covers two whole 256-byte row pieces
    const int pw = p >> 5, pl = p & 31, piece = pl & 15;
    const float* qrow = A.qbuf + (static_cast<int64_t>(b) * kM + 16 * pw + (pl >> 4)) * kDl + 4 * piece;
    const uint4* qimg = reinterpret_cast<const uint4*>(A.qimg + static_cast<int64_t>(b) * 2 * kBlk);
    const unsigned char* raw = sm + kOffRaw;
    int raw_last = 0;  // local index of the last raw copy issued
    // q' of this thread's pieces of the next two latent chunks (q' does not
    // change from tile to tile): qa serves the chunk being built, qb is in
    // flight for the one after
    float4 qa[8], qb[8];
    auto load_q = [&](int c, float4 (&dst)[8]) {
#pragma unroll
      for (int k = 0; k < 8; ++k) dst[k] = *reinterpret_cast<const float4*>(qrow + 2 * k * kDl + c * kCh);
    };
    load_q(0, qa);
    load_q(1, qb);
    for (int i = 0; i < n; ++i) {
      const int par = i & 1;
      // this tile's pages have landed (its scales go to the meta buffer of
      // tile i - 2, long free)
      if (!wait(BAR_RAW, i & 1)) break;
      float* meta = reinterpret_cast<float*>(sm + kOffMeta + par * kMeta);
      {  // column scales (page q of the tile holds channels [64 q, +64)), row scales
        const int j = 2 * p;
        *reinterpret_cast<float2*>(meta + j) =
            *reinterpret_cast<const float2*>(raw + (j / 64) * kPB + kPG.col() + (j % 64) * 4);
        if (p < kN) {
          const float a = *reinterpret_cast<const float*>(raw + (p / 16) * kPB + kPG.a() + (p % 16) * 4);
          const float bb = *reinterpret_cast<const float*>(raw + (p / 16) * kPB + kPG.b() + (p % 16) * 4);
          meta[kDl + p] = a;
          meta[kDl + kM + p] = fmaf(8.f, a, bb);
        }
      }
      mbar_arrive_plain(bars + BAR_PSYNC);
      if (!wait(BAR_PSYNC, 0)) break;  // phase 2i
      // the previous tile's P V is done: P, which aliases the ring, and this
      // half's code blocks are free
      if (i > 0 && !wait(BAR_OFULL, (i - 1) & 1)) break;
      float wk[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
      // chunk c: wait for its ring stage, build A (and B) into it, publish it
      auto chunk = [&](int c, const float4 (&q)[8]) -> bool {
        const int g = i * kChunks + c, s = g & 1, u = g >> 1;
        if (u > 0 && !wait(BAR_AEMPTY + s, (u - 1) & 1)) return false;
        unsigned char* st = sm + kOffRing + s * kStage;
        if (c < kChunks - 1) {
          // B: codes of token p / 2, channels 64 c + 32 (p % 2) + [0, 32): word
          // w = 2 c + p % 2 of each of the row's four lane chunks t; its pair
          // k (nibbles k, k + 4) is channels 32 w + 8 k + 2 t + {0, 1}
          const int tau = p >> 1, wp = p & 1, w = 2 * c + wp;
          const unsigned char* row = raw + (tau / 16) * kPB + (tau % 16) * (kDl / 2);
          // token rows are 256 bytes apart (one bank set): the lanes of a
          // warp read the four words in an order rotated by (tau / 2) % 4,
          // so that one load instruction touches 16 banks instead of 4
          const int rot = (tau >> 1) & 3;
          uint32_t y[4];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const int t = (j + rot) & 3;
            y[j] = *reinterpret_cast<const uint32_t*>(row + 16 * ((4 * (w >> 2) + t) ^ (4 * (tau & 1))) + 4 * (w & 3));
          }
          // x[t] = y[(t - rot) mod 4], in two conditional rotations
          uint32_t x[4];
#pragma unroll
          for (int t = 0; t < 4; ++t) x[t] = (rot & 1) ? y[(t + 3) & 3] : y[t];
#pragma unroll
          for (int t = 0; t < 4; ++t) y[t] = x[t];
#pragma unroll
          for (int t = 0; t < 4; ++t) x[t] = (rot & 2) ? y[(t + 2) & 3] : y[t];
          unsigned char* bdst = (c / 4 == half) ? sm + kOffOwn + (c % 4) * kBlk : st + 2 * kBlk;
#pragma unroll
          for (int k = 0; k < 4; ++k)
            *reinterpret_cast<uint4*>(bdst + sw128_unit(tau, 4 * wp + k)) =
                make_uint4(code_pair_m8(x[0], k), code_pair_m8(x[1], k), code_pair_m8(x[2], k), code_pair_m8(x[3], k));
          // A: q~ = q' * c, fp16 hi and lo planes; w partial sums per row
          const float4 cv = *reinterpret_cast<const float4*>(meta + c * kCh + 4 * piece);
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const int r = 16 * pw + 2 * k + (pl >> 4);
            const float2 x01 = f2mul(make_float2(q[k].x, q[k].y), make_float2(cv.x, cv.y));
            const float2 x23 = f2mul(make_float2(q[k].z, q[k].w), make_float2(cv.z, cv.w));
            const float2 xs = f2add(x01, x23);
            wk[k] += xs.x + xs.y;
            uint32_t h0, l0, h1, l1;
            split_hi_lo2(x01, h0, l0);
            split_hi_lo2(x23, h1, l1);
            const uint32_t off = sw128_unit(r, piece >> 1) + 8 * (piece & 1);
            *reinterpret_cast<uint2*>(st + off) = make_uint2(h0, h1);
            *reinterpret_cast<uint2*>(st + kBlk + off) = make_uint2(l0, l1);
          }
        } else {
          // A: the rope query planes (hi block, lo block); B: the tile's rope keys
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const int idx = p + kProducers * k;
            *reinterpret_cast<uint4*>(st + 16 * idx) = __ldg(qimg + idx);
          }
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const int idx = p + kProducers * k, tau = idx >> 3, un = idx & 7;
            *reinterpret_cast<uint4*>(st + 2 * kBlk + sw128_unit(tau, un)) = *reinterpret_cast<const uint4*>(
                raw + (tau / 16) * kPB + kPG.rope() + (tau % 16) * 2 * kR + 16 * un);
          }
        }
        fence_proxy_async_smem();  // generic writes -> tensor-core reads
        mbar_arrive_plain(bars + BAR_AFULL + s);
        return true;
      };
      // latent chunks in pairs: qa and qb alternate, each reloaded (for the
      // chunk two ahead, wrapping into the next tile) right after its use
      bool failed = false;
#pragma unroll 1
      for (int c = 0; c < kChunks - 1 && !failed; c += 2) {
        failed = !chunk(c, qa);
        load_q((c + 2) % (kChunks - 1), qa);
        if (!failed) failed = !chunk(c + 1, qb);
        load_q((c + 3) % (kChunks - 1), qb);
      }
      if (!failed) failed = !chunk(kChunks - 1, qa);  // rope (q unused)
      if (failed) break;
      // w = sum_j q~_j per head (16 lanes per row), for the row offsets
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        float v = wk[k];
#pragma unroll
        for (int o = 1; o < 16; o <<= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
        if (piece == 0) meta[kDl + 2 * kM + 16 * pw + 2 * k + (pl >> 4)] = v;
      }
      mbar_arrive_plain(bars + BAR_META);
      // every producer is done with the raw stage: fetch the next tile
      mbar_arrive_plain(bars + BAR_PSYNC);
      if (!wait(BAR_PSYNC, 1)) break;  // phase 2i + 1
      if (p == 0 && i + 1 < n) {
        fence_proxy_async_smem();
        issue_raw(t0 + i + 1);
        raw_last = i + 1;
      }
    }
    // a copy still in flight lands before the CTA exits
    if (p == 0) mbar_wait_bounded(bars + BAR_RAW, raw_last & 1, kWaitLimit);
  }

  if (tid < kConsumers) {
    // ---------------------------------------------------------- consumers
    const int m = tid;  // head = tensor-memory lane
    const uint32_t tl = tmem + (static_cast<uint32_t>(warp * 32) << 16);
    unsigned char* P = sm + tc::kOffP;
    float m_run = -INFINITY, l_run = 0.f;
    bool ok = true;
    for (int i = 0; i < n; ++i) {
      const int par = i & 1;
      if (!wait(BAR_SFULL, par) || !wait(BAR_META, par)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const float* meta = reinterpret_cast<const float*>(sm + kOffMeta + par * kMeta);
      const float* av = meta + kDl;
      const float* bv = meta + kDl + kM;
      const float w = meta[kDl + 2 * kM + m];
      // scores of tokens 32 q .. 32 q + 31: s = a S_lat + (b' w + S_rope)
      auto scores = [&](int q, float (&s)[32]) {
        uint32_t sl[32], sr[32];
        tc_ld32(tl + 32 * q, sl);
        tc_ld32(tl + 128 + 32 * q, sr);
        tc_wait_ld();
#pragma unroll
        for (int e = 0; e < 32; e += 4) {
          const float4 a4 = *reinterpret_cast<const float4*>(av + 32 * q + e);
          const float4 b4 = *reinterpret_cast<const float4*>(bv + 32 * q + e);
          s[e] = fmaf(a4.x, __uint_as_float(sl[e]), fmaf(b4.x, w, __uint_as_float(sr[e])));
          s[e + 1] = fmaf(a4.y, __uint_as_float(sl[e + 1]), fmaf(b4.y, w, __uint_as_float(sr[e + 1])));
          s[e + 2] = fmaf(a4.z, __uint_as_float(sl[e + 2]), fmaf(b4.z, w, __uint_as_float(sr[e + 2])));
          s[e + 3] = fmaf(a4.w, __uint_as_float(sl[e + 3]), fmaf(b4.w, w, __uint_as_float(sr[e + 3])));
        }
      };
      float mx = -INFINITY;
#pragma unroll 1
      for (int q = 0; q < 4; ++q) {
        float s[32];
        scores(q, s);
#pragma unroll
        for (int e = 0; e < 32; ++e) mx = fmaxf(mx, s[e]);
      }
      const float m_new = fmaxf(m_run, mx);
      const float alpha = fast_exp2(m_run - m_new);
      float lsum = 0.f, beta = 0.f;
#pragma unroll 1
      for (int q = 0; q < 4; ++q) {
        float s[32];
        scores(q, s);
#pragma unroll
        for (int e8 = 0; e8 < 4; ++e8) {  // tokens 32 q + 8 e8 .. + 7: one 16-byte unit
          uint32_t hi[4], lo[4];
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const int e = 8 * e8 + 2 * k, tok = 32 * q + e;
            const float p0 = fast_exp2(s[e] - m_new), p1 = fast_exp2(s[e + 1] - m_new);
            lsum += p0 + p1;
            beta = fmaf(p0, bv[tok], fmaf(p1, bv[tok + 1], beta));
            split_hi_lo(p0 * av[tok], p1 * av[tok + 1], hi[k], lo[k]);
          }
          const int tok0 = 32 * q + 8 * e8;
          const uint32_t off = (tok0 / 64) * kBlk + sw128_unit(m, (tok0 % 64) / 8);
          *reinterpret_cast<uint4*>(P + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
          *reinterpret_cast<uint4*>(P + 2 * kBlk + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
        }
      }
      l_run = fmaf(l_run, alpha, lsum);
      m_run = m_new;
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive_plain(bars + BAR_PFULL);
      // acc = alpha acc + c (u + beta), own channel 32 q + e: the first 128
      // channels as soon as their P V completes, while the rest still runs
#pragma unroll 1
      for (int q = 0; q < 8; ++q) {
        if ((q & 3) == 0) {
          if (!wait(q == 0 ? BAR_OFULL_A : BAR_OFULL, par)) {
            ok = false;
            break;
          }
          tc_fence_after();
        }
        uint32_t ot[32], oa[32];
        tc_ld32(tl + 32 * q, ot);
        if (i > 0) tc_ld32(tl + 256 + 32 * q, oa);
        tc_wait_ld();
        const float* cv = meta + (kDl / 2) * half + 32 * q;
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          const float prev = i > 0 ? alpha * __uint_as_float(oa[e]) : 0.f;
          oa[e] = __float_as_uint(fmaf(cv[e], __uint_as_float(ot[e]) + beta, prev));
        }
        tc_st32(tl + 256 + 32 * q, oa);
      }
      if (!ok) break;
      tc_wait_st();
      tc_fence_before();
      mbar_arrive_plain(bars + BAR_TFREE);
    }
    if (ok) {  // warp-uniform: every lane takes part in the tensor-memory loads
      const bool row = m < A.H;
      float* part = A.ws + (static_cast<int64_t>(b * A.H + (row ? m : 0)) * A.slots + split) * kMlaPStride;
      if (row && half == 0) {
        part[0] = m_run;
        part[1] = l_run;
      }
      float* pa = part + 4 + (kDl / 2) * half;
#pragma unroll 1
      for (int q = 0; q < 8; ++q) {
        uint32_t oa[32];
        tc_ld32(tl + 256 + 32 * q, oa);
        tc_wait_ld();
        if (row) {
#pragma unroll
          for (int e = 0; e < 32; e += 4)
            *reinterpret_cast<float4*>(pa + 32 * q + e) =
                make_float4(__uint_as_float(oa[e]), __uint_as_float(oa[e + 1]), __uint_as_float(oa[e + 2]),
                            __uint_as_float(oa[e + 3]));
        }
      }
    }
  }

  if (warp == kMmaWarp) {
    // -------------------------------------------------------- MMA issue
    const uint32_t own = smem_addr(sm + kOffOwn), ring = smem_addr(sm + kOffRing), pa = smem_addr(sm + tc::kOffP);
    for (int i = 0; i < n; ++i) {
      bool ok = !(i > 0) || wait(BAR_TFREE, (i - 1) & 1);  // the score/P V columns are free
      tc_fence_after();
      for (int c = 0; ok && c < kChunks; ++c) {
        const int g = i * kChunks + c, s = g & 1, u = g >> 1;
        if (!wait(BAR_AFULL + s, u & 1)) {
          ok = false;
          break;
        }
        tc_fence_after();
        if (lane == 0) {
          const uint32_t st = ring + s * kStage;
          const uint32_t bb = (c < kChunks - 1 && c / 4 == half) ? own + (c % 4) * kBlk : st + 2 * kBlk;
          const uint32_t d = tmem + (c < kChunks - 1 ? 0 : 128);
#pragma unroll
          for (int ks = 0; ks < 4; ++ks)
#pragma unroll
            for (int pl = 0; pl < 2; ++pl)
              tc_mma_f16(d, tc_desc_sw128(st + pl * kBlk + 32 * ks, 16, 1024), tc_desc_sw128(bb + 32 * ks, 16, 1024),
                         kIdQK, !((c == 0 || c == kChunks - 1) && ks == 0 && pl == 0));
          tc_commit(bars + BAR_AEMPTY + s);
        }
        __syncwarp();
      }
      if (!ok) break;
      if (lane == 0) tc_commit(bars + BAR_SFULL);
      __syncwarp();
      if (!wait(BAR_PFULL, i & 1)) break;
      tc_fence_after();
      if (lane == 0) {
        // channels 128 r .. 128 r + 127 of this half: code blocks 2 r, 2 r + 1
        // read MN-major (64-channel atoms one block apart, 8-token groups
        // 1024 bytes apart); P K-major in two 64-token blocks
#pragma unroll 1
        for (int r = 0; r < 2; ++r) {
#pragma unroll
          for (int ks = 0; ks < 8; ++ks)
#pragma unroll
            for (int pl = 0; pl < 2; ++pl)
              tc_mma_f16(tmem + 128 * r, tc_desc_sw128(pa + pl * 2 * kBlk + (ks / 4) * kBlk + 32 * (ks % 4), 16, 1024),
                         tc_desc_sw128(own + 2 * r * kBlk + ks * 2048, kBlk, 1024), kIdPV, ks > 0 || pl > 0);
          tc_commit(bars + (r == 0 ? BAR_OFULL_A : BAR_OFULL));
        }
      }
      __syncwarp();
    }
    if (lane == 0) tc_commit(bars + BAR_FIN);
    __syncwarp();
    mbar_wait_bounded(bars + BAR_FIN, 0, kWaitLimit);  // every MMA issued has completed
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tc_dealloc(tmem, 512);
  }
  if (tid == 0 && *abort_flag) set_error(A.err, KVARN_DEVERR_TIMEOUT);
}

}  // namespace

SplitPlan plan_mla(int32_t num_seqs, int32_t max_seq_len) {
  SplitPlan p{};
  const int tiles = max_seq_len / kN;
  if (tiles == 0) {
    p.tiles_per_split = 1;
    p.nsplit = 0;
  } else {
    // Two CTAs per (sequence, split), one CTA per SM, so SMs / 2 splits run
    // at once. A split of t tiles costs about t + 1/2 tile times (its
    // prologue and the 512-float partial per head that it writes and the
    // merge reads back); with S = num_seqs * ceil(tiles / t) equal splits the
    // call takes ceil(S / (SMs / 2)) such rounds. Take the split length of
    // the fewest rounds x cost, the longer one on a tie.
    const int pairs = std::max(1, device_sm_count() / 2);
    const int max_split = std::max(1, tiles / 2);
    double best_cost = 0.0;
    int best_tps = tiles;
    for (int n = 1; n <= max_split; ++n) {
      const int tps = (tiles + n - 1) / n;
      const int64_t items = static_cast<int64_t>(std::max(1, num_seqs)) * ((tiles + tps - 1) / tps);
      const double cost = static_cast<double>((items + pairs - 1) / pairs) * (tps + 0.5);
      if (n == 1 || cost < best_cost - 1e-9) {
        best_cost = cost;
        best_tps = tps;
      }
    }
    p.tiles_per_split = best_tps;
    p.nsplit = (tiles + best_tps - 1) / best_tps;
  }
  p.slots = p.nsplit + 1;
  return p;
}

// Split partials, then the prepared queries (q' rows and the rope operand
// image) of every sequence.
int64_t mla_workspace_bytes(int32_t num_seqs, int32_t num_heads, const SplitPlan& plan) {
  return static_cast<int64_t>(num_seqs) * num_heads * plan.slots * kMlaPStride * 4 +
         static_cast<int64_t>(num_seqs) * (tc::kM * kDl * 4 + 2 * tc::kBlk);
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
  unsigned char* ws = static_cast<unsigned char*>(p.workspace);
  A.qbuf = reinterpret_cast<float*>(ws + static_cast<int64_t>(p.num_seqs) * p.num_q_heads * plan.slots * kMlaPStride * 4);
  A.qimg = reinterpret_cast<unsigned char*>(A.qbuf) + static_cast<int64_t>(p.num_seqs) * tc::kM * kDl * 4;
  auto prep = p.bf16 ? mla_qprep_kernel<__nv_bfloat16> : mla_qprep_kernel<__half>;
  prep<<<dim3(tc::kM / 8, p.num_seqs), 256, 0, st>>>(A);
  auto kern = p.bf16 ? mla_tc_kernel<__nv_bfloat16> : mla_tc_kernel<__half>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, tc::kSmem);
  if (e != cudaSuccess) return e;
  kern<<<dim3(2, plan.nsplit + 1, p.num_seqs), tc::kThreads, tc::kSmem, st>>>(A);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int rows = p.num_seqs * p.num_q_heads;
  return launch_merge<512>(A.ws, A.slots, rows, nullptr, A.nsplit, A.nsplit, p.out, p.lse, st);
}

}  // namespace kvarn

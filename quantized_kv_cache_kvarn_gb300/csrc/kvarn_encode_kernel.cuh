// KVarN tile encoder for sm_103a.
//
// KVarN review ("KVarN ... vLLM KV cache quantization"), four-stage
// paragraph: rotate each tile by an orthonormal Hadamard matrix across the
// channels, run T alternating column/row standard-deviation normalisations,
// then asymmetric round-to-nearest with the scales folded into the stored
// row offsets. One CTA (or a cluster of two for head_dim 512) owns one N x D
// tile and keeps it in registers: every thread holds a 16-channel segment of
// N/32 token rows. The Hadamard transform runs as four in-register butterfly
// stages and log2(D/16) lane shuffles. Column statistics reduce through
// shared memory (and the peer CTA's shared memory in a cluster) and are
// finished once per channel by thread `channel`, which broadcasts the result;
// row statistics reduce with shuffles. The scales accumulate as products of
// the per-pass standard deviations (the exponential of the summed logs, up
// to rounding). Codes are packed in registers straight into the page's word
// order, staged in shared memory and written out in 16-byte stores.
#pragma once

#include <cooperative_groups.h>

#include "kvarn_common.cuh"
#include "kvarn_launch.h"

namespace cg = cooperative_groups;

namespace kvarn {

// Cluster size 2 splits the tile's rows over two CTAs (head_dim 512, where a
// whole 128 x 512 fp32 tile would not fit one CTA's registers).
template <int D, int N, int CS, bool GEN = false>
struct EncShape {
  static constexpr int NT = 2 * D / CS;       // threads per CTA
  static constexpr int TPR = D / 16;          // threads per token row
  static constexpr int RPW = 32 / TPR;        // rows per warp and pass
  static constexpr int NW = NT / 32;          // warps
  static constexpr int ROWS = N / CS;         // rows owned by this CTA
  static constexpr int RPT = N / 32;          // rows per thread
  static constexpr int PPC = ROWS / kPageTokens;  // pages per CTA
  static_assert(ROWS == RPT * NW * RPW, "tile rows must cover the CTA");
  static_assert(NT >= D, "one thread per channel finishes the column statistics");
  static constexpr int RED_BYTES = NW * D * 8;  // (mean, M2) per warp and channel
  // packed words (4-bit K / 2-bit V); the generic path stages one byte per
  // code plus the packed image of up to 8 bits per code
  static constexpr int CODE_BYTES = GEN ? 2 * ROWS * D : ROWS * D / 2;
  static constexpr int SCRATCH = RED_BYTES > CODE_BYTES ? RED_BYTES : CODE_BYTES;
  // scratch | colbuf[D] | rowA[ROWS] | rowB[ROWS] | colC[D] | colpart[2][2][D] | pages[PPC]
  static constexpr int OFF_COLBUF = SCRATCH;
  static constexpr int OFF_ROWA = OFF_COLBUF + 4 * D;
  static constexpr int OFF_ROWB = OFF_ROWA + 4 * ROWS;
  static constexpr int OFF_COLC = OFF_ROWB + 4 * ROWS;
  static constexpr int OFF_COLPART = OFF_COLC + 4 * D;
  static constexpr int OFF_PAGES = OFF_COLPART + 16 * D;
  static constexpr int SMEM = OFF_PAGES + 8 * PPC;
};

struct EncodeArgs {
  const void* x[2];        // K, V (dense) or latent (x[0])
  const __half* rope;      // latent only
  int64_t seq_stride, head_stride, rope_seq_stride;
  int32_t chunk_tiles;
  int32_t num_seqs;
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
  int32_t bf16;  // storage dtype of the dense and latent inputs: 0 fp16, 1 bf16
  // optional fp32 intermediates of every encoded dense tile (null in normal
  // use): per (sequence, KV head, chunk tile, K|V) the rotated tile Y, the
  // normalised tile Z (both N x D, token rows), then r, lo, delta per token
  // and c per channel
  float* stages;
};


// Per-channel shared buffers are written a 16-byte chunk per lane: lane seg
// holds channels 16 seg .. 16 seg + 15, its chunk e channels 16 seg + 4e ..
// + 3. Chunk (e, seg) goes to slot e * (D / 16) + (seg ^ 2e): for one e the
// lanes' chunks fill consecutive slots (a permutation of them), and the 32
// consecutive channels a warp reads one per thread fall in 32 different
// banks (the XOR spreads the four chunks e of one lane over the 128-byte
// rows). chunk_slot is that slot, chunk_pos the float position of channel c.
template <int D>
__device__ __forceinline__ int chunk_slot(int e, int seg) {
  return e * (D / 16) + (seg ^ (2 * e));
}
template <int D>
__device__ __forceinline__ int chunk_pos(int c) {
  return chunk_slot<D>((c & 15) >> 2, c >> 4) * 4 + (c & 3);
}

// Merge of two (mean, M2) summaries of n values each (Chan, Golub and
// LeVeque's pairwise update of the sum of squared deviations): the mean of
// 2n values and their M2. Written symmetrically in a and b, so that the two
// lanes of a butterfly (or the two CTAs of a cluster) hold bit-identical
// results.
__device__ __forceinline__ float2 merge_moments(float2 a, float2 b, float n) {
  const float d = b.x - a.x;
  return make_float2(0.5f * (a.x + b.x), (a.y + b.y) + 0.5f * n * d * d);
}

// Column moments in one reduction: every thread passes, per channel of its
// segment, the mean and M2 of its RPT rows. Returns, in thread tid < D, the
// population mean and variance over the whole tile (both CTAs of a cluster)
// of channel tid; other threads get (0, 0). colpart (2 x D floats) is this
// statistic's cluster exchange buffer (callers alternate two).
template <int D, int N, int CS>
__device__ __forceinline__ float2 column_moments(float2 (&mo)[16], float* red, float* colpart) {
  using S = EncShape<D, N, CS>;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, seg = lane % S::TPR;
  float n = static_cast<float>(S::RPT);
#pragma unroll
  for (int o = S::TPR; o < 32; o <<= 1) {
#pragma unroll
    for (int e = 0; e < 16; ++e) {
      const float2 b = make_float2(__shfl_xor_sync(0xffffffffu, mo[e].x, o), __shfl_xor_sync(0xffffffffu, mo[e].y, o));
      mo[e] = merge_moments(mo[e], b, n);
    }
    n *= 2.f;
  }
  if (lane < S::TPR) {
    float4* dm = reinterpret_cast<float4*>(red + warp * D);
    float4* dv = reinterpret_cast<float4*>(red + (S::NW + warp) * D);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      dm[chunk_slot<D>(e, seg)] = make_float4(mo[4 * e].x, mo[4 * e + 1].x, mo[4 * e + 2].x, mo[4 * e + 3].x);
      dv[chunk_slot<D>(e, seg)] = make_float4(mo[4 * e].y, mo[4 * e + 1].y, mo[4 * e + 2].y, mo[4 * e + 3].y);
    }
  }
  __syncthreads();
  float2 t = make_float2(0.f, 0.f);
  if (threadIdx.x < D) {
    float2 w[S::NW];
#pragma unroll
    for (int i = 0; i < S::NW; ++i) {
      const int pos = chunk_pos<D>(threadIdx.x);
      w[i] = make_float2(red[i * D + pos], red[(S::NW + i) * D + pos]);
    }
    float nw = static_cast<float>(S::RPT * S::RPW);  // rows per warp
#pragma unroll
    for (int st = 1; st < S::NW; st *= 2) {
#pragma unroll
      for (int i = 0; i + st < S::NW; i += 2 * st) w[i] = merge_moments(w[i], w[i + st], nw);
      nw *= 2.f;
    }
    t = w[0];
  }
  if constexpr (CS > 1) {
    cg::cluster_group cl = cg::this_cluster();
    if (threadIdx.x < D) {
      colpart[threadIdx.x] = t.x;
      colpart[D + threadIdx.x] = t.y;
    }
    cl.sync();
    if (threadIdx.x < D) {
      const float* o = cl.map_shared_rank(colpart, cl.block_rank() ^ 1);
      t = merge_moments(t, make_float2(o[threadIdx.x], o[D + threadIdx.x]), static_cast<float>(S::ROWS));
    }
  }
  return make_float2(t.x, t.y * (1.f / N));
}

// Population std; 1 for a constant vector or a non-finite std. The sums
// behind `var` are pairwise trees and pairwise (mean, M2) merges, so a vector
// of equal entries gives var == 0 exactly (every partial mean is exact and
// every deviation zero), and one whose entries differ gives var > 0 (some
// deviation or merge difference is non-zero; only differences below ~1e-19
// would square to zero in fp32): var == 0 is the test max == min.
__device__ __forceinline__ float safe_sigma(float var) {
  const float s = sqrtf(var);
  return (isfinite(s) && s > 0.f) ? s : 1.f;
}

// Round-to-nearest of normalised values on their row's grid (lo, delta),
// four codes at a time as the bytes of one word (pair k, element e at byte
// 2k + e). x = (z - lo) * (1/delta) as the caller formed it; the sum
// x + 1.5 * 2^23 rounds x to an integer, half to even, in the addition
// itself, and the integer is the sum's low byte (x lies in [0, 2^bits - 1]
// up to rounding, so no clamp is needed; a non-finite input gives unspecified
// codes in its own row). x minus that integer says how near x lies to a
// half-way point. The product is within a few units in the last place of the
// exact quotient (z - lo) / delta of the fp32 operands, so only where one of
// the four lands within 2^-14 of a half-way point is the word redone,
// exactly, out of line. The result is the round-half-to-even of the exact
// quotient.
static __device__ __noinline__ uint32_t grid_word_exact(float2 z0, float2 z1, float lo, float delta, float2 x0,
                                                        float2 x1, uint32_t w);

__device__ __forceinline__ uint32_t grid_codes4(float2 z0, float2 z1, float lo, float delta, float2 x0, float2 x1) {
  constexpr float kRound = 12582912.f;  // 1.5 * 2^23
  const float2 t0 = f2add(x0, f2(kRound)), t1 = f2add(x1, f2(kRound));
  const float2 d0 = f2fma(f2add(t0, f2(-kRound)), f2(-1.f), x0);
  const float2 d1 = f2fma(f2add(t1, f2(-kRound)), f2(-1.f), x1);
  uint32_t w = __byte_perm(__byte_perm(__float_as_uint(t0.x), __float_as_uint(t0.y), 0x0040),
                           __byte_perm(__float_as_uint(t1.x), __float_as_uint(t1.y), 0x0040), 0x5410);
  const float m = fmaxf(fmaxf(fabsf(d0.x), fabsf(d0.y)), fmaxf(fabsf(d1.x), fabsf(d1.y)));
  if (m > 0.5f - 0x1p-14f) w = grid_word_exact(z0, z1, lo, delta, x0, x1, w);
  return w;
}

// The side of the half-way point k + 1/2 nearest x, decided exactly: z - lo
// is the rounded sum s plus its rounding error e (the two-sum), and
// s - (k + 1/2) delta, a small multiple of the finer of the two operands'
// last-place units near the boundary, is formed exactly by the fused
// multiply-add; the sign of that plus e is the sign of the exact
// (z - lo) - (k + 1/2) delta. A tie goes to the even code.
__device__ __forceinline__ uint32_t grid_boundary_code(float z, float lo, float delta, float x) {
  const float s = __fadd_rn(z, -lo);
  const float bb = __fsub_rn(s, z);
  const float e = __fadd_rn(__fsub_rn(z, __fsub_rn(s, bb)), __fsub_rn(-lo, bb));
  const float k = floorf(x);
  const float w = __fadd_rn(__fmaf_rn(-(k + 0.5f), delta, s), e);
  const uint32_t ki = static_cast<uint32_t>(k);
  return ki + ((w > 0.f || (w == 0.f && (ki & 1u))) ? 1u : 0u);
}

static __device__ __noinline__ uint32_t grid_word_exact(float2 z0, float2 z1, float lo, float delta, float2 x0,
                                                        float2 x1, uint32_t w) {
  const float z[4] = {z0.x, z0.y, z1.x, z1.y}, x[4] = {x0.x, x0.y, x1.x, x1.y};
#pragma unroll
  for (int i = 0; i < 4; ++i)
    if (fabsf(x[i] - rintf(x[i])) > 0.5f - 0x1p-14f)
      w = (w & ~(0xFFu << (8 * i))) | ((grid_boundary_code(z[i], lo, delta, x[i]) & 0xFFu) << (8 * i));
  return w;
}

// Latent page word order (before the 16-byte unit swizzle): the 32-bit word
// tau * (D/8) + t * (D/32) + w of token tau holds, at nibbles 0,1,4,5, the
// codes of channels 2t, 2t+8, 2t+1, 2t+9 of 16-channel segment 2w and, at
// nibbles 2,3,6,7, the same channels of segment 2w+1 (the B-fragment order
// of an m16n8k16 mma). `P` holds the row's 16 codes of one segment as bytes;
// returns this segment's nibbles of word t, placed for segment parity `s`.
__device__ __forceinline__ uint32_t k_word_part(const uint32_t (&P)[4], int t, int s) {
  const uint32_t v = __byte_perm(P[t >> 1], P[2 + (t >> 1)], (t & 1) ? 0x7362 : 0x5140);
  return ((v | (v >> 4)) & 0x00FF00FFu) << (8 * s);
}

// The plane words of `pages` pages of codes staged as bytes cb [16 pages][D]
// (one byte per code, token-major), in the dense page's K (IS_V false) or V
// placement at BITS bits: img[p * D * BITS / 2 + w] is word w of page p's
// code region. Threads tid, tid + nt, ... build one word each.
template <int D, int BITS, bool IS_V>
__device__ __forceinline__ void pack_plane_words(const unsigned char* cb, uint32_t* img, int pages, int tid, int nt) {
  constexpr int W0 = plane_w0(BITS), W1 = plane_w1(BITS);
  constexpr int WPP = D * BITS / 2;  // 32-bit words of codes per page
  for (int ws = tid; ws < pages * WPP; ws += nt) {
    const int pg = ws / WPP, rem = ws % WPP;
    const bool p1 = rem >= D * W0 / 2;
    const int w = p1 ? W1 : W0, shift = p1 ? W0 : 0, wi = p1 ? rem - D * W0 / 2 : rem;
    const int U = IS_V ? w : min(4, D * w / 64);
    const int L = (wi % (32 * U)) / U, i = (wi / (32 * U)) * U + wi % U;
    const int g = L >> 2, t = L & 3, F = 8 / w;
    uint32_t word = 0;
    for (int f = 0; f < F; ++f) {
      const int fg = i * F + f;
#pragma unroll
      for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int ep = 0; ep < 2; ++ep) {
          const int ch = IS_V ? 8 * fg + g : 16 * (fg >> 1) + 2 * t + ep + 8 * h;
          const int tok = IS_V ? 2 * t + ep + 8 * h : 8 * (fg & 1) + g;
          const uint32_t field = (cb[(pg * kPageTokens + tok) * D + ch] >> shift) & ((1u << w) - 1u);
          word |= field << plane_bit(w, f, h, ep);
        }
    }
    img[ws] = word;
  }
}

// Encodes rows [0, N) of `src` as logical tile `tile` of sequence b (u: the
// tile's index in the chunk, for the latent rope rows). With last_row set,
// row N - 1 comes from last_row instead of src (the newest token, appended
// in the same launch).
// KIND 0: a dense tile, SIDE_V selecting its V (else K) part of pages of code
// widths KB, VB and SB-byte scales; KIND 1: a latent tile (4-bit, fp32).
template <int D, int N, int CS, int BITS, int KIND, bool SIDE_V = false, int KB = 4, int VB = 2,
          int SB = 4>
__device__ __forceinline__ void encode_tile(const EncodeArgs& A, const unsigned char* __restrict__ src,
                                            int b, int head, int u, int64_t tile, const unsigned char* last_row,
                                            unsigned char* smem) {
  constexpr bool IS_V = KIND == 0 && SIDE_V;
  // the 4-bit K and 2-bit V placements pack in registers; other widths take
  // the generic plane path
  constexpr bool GEN = KIND == 0 && !(SIDE_V ? BITS == 2 : BITS == 4);
  using S = EncShape<D, N, CS, GEN>;
  constexpr DensePage PGE{D, N, KB, VB, SB};
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int seg = lane % S::TPR, rsub = lane / S::TPR;
  int crank = 0;
  if constexpr (CS > 1) crank = static_cast<int>(cg::this_cluster().block_rank());

  float* red = reinterpret_cast<float*>(smem);
  unsigned char* stage = smem;  // aliases red once the statistics are done
  float* colbuf = reinterpret_cast<float*>(smem + S::OFF_COLBUF);
  float* rowA = reinterpret_cast<float*>(smem + S::OFF_ROWA);
  float* rowB = reinterpret_cast<float*>(smem + S::OFF_ROWB);
  float* colC = reinterpret_cast<float*>(smem + S::OFF_COLC);
  float* colpart = reinterpret_cast<float*>(smem + S::OFF_COLPART);
  uint8_t** pages = reinterpret_cast<uint8_t**>(smem + S::OFF_PAGES);

  // ---- load. Dense tiles: thread group j = warp*RPW + rsub (0..31) holds
  // tokens j%8 and j%8 + 8 of RPT/2 pages, so that the two tokens sharing a
  // packed byte of the dense page are in one thread. Latent tiles: row
  // i*32 + j of this CTA's rows.
  // channel pairs (2e, 2e + 1) of the thread's 16 channels, so that the
  // arithmetic below runs as packed fp32 pair instructions
  float2 xp[S::RPT][8];
  auto local_row = [&](int i) -> int {
    const int j = warp * S::RPW + rsub;
    if constexpr (KIND == 0)
      return kPageTokens * ((S::RPT / 2) * (j >> 3) + (i >> 1)) + (j & 7) + 8 * (i & 1);
    else
      return i * (S::NW * S::RPW) + j;
  };
  static_assert(KIND != 0 || (S::NW * S::RPW == 32 && S::RPT % 2 == 0), "dense row pairing");
#pragma unroll
  for (int i = 0; i < S::RPT; ++i) {
    const int r = crank * S::ROWS + local_row(i);
    // 16-bit elements (fp16 or bf16 by A.bf16, uniform over the grid)
    const unsigned char* p = (last_row != nullptr && r == N - 1)
                                 ? last_row + 2 * (seg * 16)
                                 : src + 2 * (static_cast<int64_t>(r) * D + seg * 16);
    float v[16];
    if (A.bf16) {
      load8<__nv_bfloat16>(reinterpret_cast<const __nv_bfloat16*>(p), v);
      load8<__nv_bfloat16>(reinterpret_cast<const __nv_bfloat16*>(p) + 8, v + 8);
    } else {
      load8<__half>(reinterpret_cast<const __half*>(p), v);
      load8<__half>(reinterpret_cast<const __half*>(p) + 8, v + 8);
    }
#pragma unroll
    for (int e = 0; e < 8; ++e) xp[i][e] = make_float2(v[2 * e], v[2 * e + 1]);
  }

  // ---- page addresses of this CTA's rows (read by the stores at the end)
  constexpr int PPT = N / kPageTokens;  // pages per tile
  if (tid < S::PPC) {
    const int64_t lp = tile * PPT + crank * S::PPC + tid;
    uint8_t* pg = nullptr;
    const int32_t phys =
        (lp >= 0 && lp < A.bt_stride) ? A.block_table[static_cast<int64_t>(b) * A.bt_stride + lp] : -1;
    if (phys >= 0 && phys < A.num_pages)
      pg = A.cache + (static_cast<int64_t>(phys) * A.num_kv_heads + head) * A.page_bytes;
    else
      set_error(A.err, KVARN_DEVERR_PAGE_RANGE);
    pages[tid] = pg;
  }

  // ---- the optional stage record of this tile (dense tiles only)
  float* rec = nullptr;
  if constexpr (KIND == 0 && CS == 1) {
    if (A.stages != nullptr)
      rec = A.stages + ((static_cast<int64_t>(b) * A.num_kv_heads + head) * A.chunk_tiles + u) * 2 * stage_floats(D, N) +
            (IS_V ? stage_floats(D, N) : 0);
  }
  auto record_tile = [&](float* dst) {  // this thread's values of the N x D tile, token rows
#pragma unroll
    for (int i = 0; i < S::RPT; ++i)
#pragma unroll
      for (int e = 0; e < 8; ++e)
        *reinterpret_cast<float2*>(dst + static_cast<int64_t>(local_row(i)) * D + seg * 16 + 2 * e) = xp[i][e];
  };

  // ---- Hadamard: 4 in-register stages, then lane butterflies, then 1/sqrt(D)
#pragma unroll
  for (int i = 0; i < S::RPT; ++i) {
#pragma unroll
    for (int e = 0; e < 8; ++e) {  // stage 1: within a pair
      const float a = xp[i][e].x, c = xp[i][e].y;
      xp[i][e] = make_float2(a + c, a - c);
    }
#pragma unroll
    for (int h = 1; h < 8; h <<= 1)  // stages 2, 4, 8: between pairs
#pragma unroll
      for (int e = 0; e < 8; ++e)
        if (!(e & h)) {
          const float2 a = xp[i][e], c = xp[i][e + h];
          xp[i][e] = f2add(a, c);
          xp[i][e + h] = f2fma(c, f2(-1.f), a);
        }
  }
#pragma unroll
  for (int d = 1; d < S::TPR; d <<= 1) {
    // lower lane: x + partner; upper lane: partner - x  (one FFMA either way)
    const float2 sgn = f2((lane & d) ? -1.f : 1.f);
#pragma unroll
    for (int i = 0; i < S::RPT; ++i)
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const float2 o = make_float2(__shfl_xor_sync(0xffffffffu, xp[i][e].x, d),
                                     __shfl_xor_sync(0xffffffffu, xp[i][e].y, d));
        xp[i][e] = f2fma(sgn, xp[i][e], o);
      }
  }
  {
    const float2 rsd = f2(1.f / sqrtf(static_cast<float>(D)));
#pragma unroll
    for (int i = 0; i < S::RPT; ++i)
#pragma unroll
      for (int e = 0; e < 8; ++e) xp[i][e] = f2mul(xp[i][e], rsd);
  }
  if (rec != nullptr) record_tile(rec);

  // ---- variance normalisation, T iterations of (column pass, row pass)
  float cscale = 1.f;  // column scale of channel tid (tid < D)
  float rscale[S::RPT];
#pragma unroll
  for (int i = 0; i < S::RPT; ++i) rscale[i] = 1.f;
  const float invD = 1.f / D;

#pragma unroll 1
  for (int it = 0; it < A.norm_iters; ++it) {
    // column pass: mean and M2 of this thread's rows per channel, merged
    // over the tile in one reduction
    float2 mo[16];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      // pairwise, so that equal entries sum exactly
      float2 cs[S::RPT];
#pragma unroll
      for (int i = 0; i < S::RPT; ++i) cs[i] = xp[i][e];
      const float2 t = tree_reduce(cs, [](float2 u, float2 w) { return f2add(u, w); });
      const float2 m = f2mul(t, f2(1.f / S::RPT)), nm = f2mul(m, f2(-1.f));
      float2 v = f2(0.f);
#pragma unroll
      for (int i = 0; i < S::RPT; ++i) {
        const float2 dv = f2add(xp[i][e], nm);
        v = f2fma(dv, dv, v);
      }
      mo[2 * e] = make_float2(m.x, v.x);
      mo[2 * e + 1] = make_float2(m.y, v.y);
    }
    const float2 cm = column_moments<D, N, CS>(mo, red, colpart + (it & 1) * 2 * D);
    if (tid < D) {
      const float sig = safe_sigma(cm.y);
      cscale *= sig;
      colbuf[chunk_pos<D>(tid)] = 1.f / sig;
    }
    __syncthreads();
    float2 inv[8];
    {
      const float4* src = reinterpret_cast<const float4*>(colbuf);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float4 f = src[chunk_slot<D>(e, seg)];
        inv[2 * e] = make_float2(f.x, f.y);
        inv[2 * e + 1] = make_float2(f.z, f.w);
      }
    }
#pragma unroll
    for (int i = 0; i < S::RPT; ++i)
#pragma unroll
      for (int e = 0; e < 8; ++e) xp[i][e] = f2mul(xp[i][e], inv[e]);
    // row pass: a row lives in TPR consecutive lanes; mean and M2 of the
    // lane's 16 channels, merged over the row's lanes
#pragma unroll
    for (int i = 0; i < S::RPT; ++i) {
      float2 ts[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) ts[e] = xp[i][e];
      const float2 tt = tree_reduce(ts, [](float2 u, float2 w) { return f2add(u, w); });
      const float m0 = (tt.x + tt.y) * (1.f / 16.f);
      const float2 nm = f2(-m0);
      float2 vs[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const float2 dv = f2add(xp[i][e], nm);
        vs[e] = f2mul(dv, dv);
      }
      const float2 vt = tree_reduce(vs, [](float2 u, float2 w) { return f2add(u, w); });
      float2 r = make_float2(m0, vt.x + vt.y);
      float n = 16.f;
#pragma unroll
      for (int o = 1; o < S::TPR; o <<= 1) {
        r = merge_moments(r, make_float2(__shfl_xor_sync(0xffffffffu, r.x, o), __shfl_xor_sync(0xffffffffu, r.y, o)), n);
        n *= 2.f;
      }
      const float sig = safe_sigma(r.y * invD);
      rscale[i] *= sig;
      const float2 ri = f2(1.f / sig);
#pragma unroll
      for (int e = 0; e < 8; ++e) xp[i][e] = f2mul(xp[i][e], ri);
    }
    // colbuf is rewritten next only after the next column reduction's barrier
  }
  if (rec != nullptr) {
    record_tile(rec + static_cast<int64_t>(N) * D);
    if (tid < D) rec[2 * N * D + 3 * N + tid] = cscale;
  }

  // ---- asymmetric RTN per row: codes as bytes, Pc[i][k] byte e = channel 4k + e
  constexpr int QMAX = (1 << BITS) - 1;
  uint32_t Pc[S::RPT][4];
#pragma unroll
  for (int i = 0; i < S::RPT; ++i) {
    float lo = fminf(xp[i][0].x, xp[i][0].y), hi = fmaxf(xp[i][0].x, xp[i][0].y);
#pragma unroll
    for (int e = 1; e < 8; ++e) {
      lo = fminf(lo, fminf(xp[i][e].x, xp[i][e].y));
      hi = fmaxf(hi, fmaxf(xp[i][e].x, xp[i][e].y));
    }
#pragma unroll
    for (int o = 1; o < S::TPR; o <<= 1) {
      lo = fminf(lo, __shfl_xor_sync(0xffffffffu, lo, o));
      hi = fmaxf(hi, __shfl_xor_sync(0xffffffffu, hi, o));
    }
    const float delta = (hi - lo) / static_cast<float>(QMAX);
    const float rinv = delta > 0.f ? 1.f / delta : 0.f;
    const float2 nlo = f2(-lo), rv = f2(rinv);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      // z - lo lies in [0, hi - lo], so the codes lie in [0, QMAX]
      const float2 z0 = xp[i][2 * k], z1 = xp[i][2 * k + 1];
      Pc[i][k] = grid_codes4(z0, z1, lo, delta, f2mul(f2add(z0, nlo), rv), f2mul(f2add(z1, nlo), rv));
    }
    if (seg == 0) {
      const int r = local_row(i);
      rowA[r] = rscale[i] * (delta > 0.f ? delta : 0.f);
      rowB[r] = rscale[i] * lo;
      if (rec != nullptr) {
        rec[2 * N * D + r] = rscale[i];
        rec[2 * N * D + N + r] = lo;
        rec[2 * N * D + 2 * N + r] = delta;
      }
    }
  }

  // ---- codes packed into the page's word order in `stage`
  const int s_par = seg & 1, w_pair = seg >> 1;
  if constexpr (KIND == 1) {
#pragma unroll
    for (int i = 0; i < S::RPT; ++i) {
      const int r = local_row(i);
      const int pg = r / kPageTokens, tau = r % kPageTokens;
      // each lane pair shares words; the even lane writes t = 0, 1, the odd lane t = 2, 3
      uint32_t* img = reinterpret_cast<uint32_t*>(stage) + pg * 2 * D + tau * (D / 8);
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const uint32_t lo_t = k_word_part(Pc[i], j, s_par), hi_t = k_word_part(Pc[i], 2 + j, s_par);
        const uint32_t other = __shfl_xor_sync(0xffffffffu, s_par ? lo_t : hi_t, 1);
        const int t = 2 * s_par + j;
        // 16-byte units 4q + t, XOR 4 on odd tokens
        const int word = 4 * ((4 * (w_pair >> 2) + t) ^ (4 * (tau & 1))) + (w_pair & 3);
        img[word] = (s_par ? hi_t : lo_t) | other;
      }
    }
  } else if constexpr (GEN) {
    // stage the codes as bytes [ROWS][D], then build every plane word
    unsigned char* cb = stage;
#pragma unroll
    for (int i = 0; i < S::RPT; ++i)
      *reinterpret_cast<uint4*>(cb + local_row(i) * D + seg * 16) = make_uint4(Pc[i][0], Pc[i][1], Pc[i][2], Pc[i][3]);
    __syncthreads();
    pack_plane_words<D, BITS, IS_V>(cb, reinterpret_cast<uint32_t*>(stage + S::ROWS * D), S::PPC, tid, S::NT);
  } else {
    const int j = warp * S::RPW + rsub, g = j & 7;
#pragma unroll
    for (int ip = 0; ip < S::RPT / 2; ++ip) {
      const int pg = (S::RPT / 2) * (j >> 3) + ip;
      const uint32_t* P0 = Pc[2 * ip];      // token g of the page
      const uint32_t* P1 = Pc[2 * ip + 1];  // token g + 8
      if constexpr (!IS_V) {
        // 4-bit: word (kc = seg, lane 4g + t) bytes = channels 2t, 2t+1,
        // 2t+8, 2t+9; token g in the low nibble, token g + 8 in the high one
        uint32_t* img = reinterpret_cast<uint32_t*>(stage) + pg * 2 * D;
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          const uint32_t sel = (t & 1) ? 0x7632u : 0x5410u;
          const uint32_t w0 = __byte_perm(P0[t >> 1], P0[2 + (t >> 1)], sel);
          const uint32_t w1 = __byte_perm(P1[t >> 1], P1[2 + (t >> 1)], sel);
          img[((seg >> 2) * 32 + 4 * g + t) * 4 + (seg & 3)] = w0 | (w1 << 4);
        }
      } else {
        // 2-bit: byte c of word (lane 4g' + t, w) is channel 8(4w + c) + g'
        // with tokens 2t, 2t + 8, 2t + 1, 2t + 9 at bits 0, 2, 4, 6. This
        // thread holds tokens g and g + 8 of channels 16 seg + 0..15; the
        // thread of token g ^ 1 (lane ^ TPR) holds the other two, so the
        // pair exchanges its half-bytes and each writes four half-words:
        // channels g' and 8 + g' (blocks 2 seg and 2 seg + 1) of lane
        // 4g' + g/2, word seg/2, half-word seg % 2.
        uint32_t Z[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const uint32_t a = P0[k] | (P1[k] << 2);
          const uint32_t o = __shfl_xor_sync(0xffffffffu, a, S::TPR);
          Z[k] = (g & 1) ? (o | (a << 4)) : (a | (o << 4));
        }
        uint16_t* img = reinterpret_cast<uint16_t*>(stage) + pg * 2 * D;
        const int t = g >> 1, wi = seg >> 1;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int gp = 4 * (g & 1) + q;  // g' = 0..3 from the even thread, 4..7 from the odd one
          const uint32_t hw = __byte_perm(Z[gp >> 2], Z[2 + (gp >> 2)], q | ((4 + q) << 4));
          const int word = 2 * (32 * (wi >> 1) + 4 * gp + t) + (wi & 1);
          img[2 * word + (seg & 1)] = static_cast<uint16_t>(hw);
        }
      }
    }
  }
  if (tid < D) colC[tid] = cscale;
  __syncthreads();

  // ---- codes: 16-byte stores of the staged page words
  {
    constexpr int CPP = 2 * D * BITS / 16;  // 16-byte chunks per page
    const int base = IS_V ? PGE.v_codes() : 0;
    const uint4* img = reinterpret_cast<const uint4*>(stage + (GEN ? S::ROWS * D : 0));
    for (int c = tid; c < S::PPC * CPP; c += S::NT) {
      uint8_t* pg = pages[c / CPP];
      if (pg) reinterpret_cast<uint4*>(pg + base)[c % CPP] = img[c];
    }
  }

  // ---- scales
  int off_a, off_b, off_c;
  if constexpr (KIND == 1) {
    constexpr LatentPage L(D, 64, N);
    off_a = L.a(); off_b = L.b(); off_c = L.col();
  } else {
    off_a = IS_V ? PGE.v_a() : PGE.k_a();
    off_b = IS_V ? PGE.v_b() : PGE.k_b();
    off_c = IS_V ? PGE.v_col() : PGE.k_col();
  }
  auto put = [&](uint8_t* at, int idx, float x) {
    if constexpr (SB == 4) reinterpret_cast<float*>(at)[idx] = x;
    else reinterpret_cast<__half*>(at)[idx] = __float2half_rn(x);
  };
  if (tid < S::ROWS) {
    uint8_t* pg = pages[tid / kPageTokens];
    if (pg) {
      put(pg + off_a, tid % kPageTokens, rowA[tid]);
      put(pg + off_b, tid % kPageTokens, rowB[tid]);
    }
  }
  {
    constexpr int C = D * kPageTokens / N;  // column scales per page
    for (int j = tid; j < S::PPC * C; j += S::NT) {
      uint8_t* pg = pages[j / C];
      if (pg) put(pg + off_c, j % C, colC[(crank * S::PPC) * C + j]);
    }
  }
  if constexpr (KIND == 1) {
    // rope rows, fp16, copied as is
    constexpr LatentPage L(D, 64, N);
    const int R = A.rope_dim;
    const int vec_per_page = kPageTokens * R * 2 / 16;
    for (int c = tid; c < S::PPC * vec_per_page; c += S::NT) {
      const int p = c / vec_per_page, k = c % vec_per_page;
      uint8_t* pg = pages[p];
      if (!pg) continue;
      const int row = crank * S::ROWS + p * kPageTokens;  // first token of the page in the tile
      const uint8_t* s = reinterpret_cast<const uint8_t*>(
          A.rope + static_cast<int64_t>(b) * A.rope_seq_stride + (static_cast<int64_t>(u) * N + row) * R);
      reinterpret_cast<uint4*>(pg + L.rope())[k] = __ldg(reinterpret_cast<const uint4*>(s) + k);
    }
  }
  // a CTA of a cluster exits only after its peer has read its last column
  // statistics from this CTA's shared memory
  if constexpr (CS > 1) cg::this_cluster().sync();
}

// K (4-bit) and V (2-bit) tiles share one launch: blockIdx.z < num_seqs
// encodes K, the rest V, so that the K half of a large grid runs before the
// V half and an SM mostly runs one of the two code paths.
template <int D, int N, int KB = 4, int VB = 2, int SB = 4>
__global__ void __launch_bounds__(2 * D, D == 128 ? 2 : 1) encode_dense_kernel(EncodeArgs A) {
  extern __shared__ __align__(128) unsigned char smem[];
  // the decode launched after a commit may be scheduled once every CTA here
  // has started; it waits for this grid's completion before it reads
  pdl_launch_dependents();
  const bool is_v = static_cast<int>(blockIdx.z) >= A.num_seqs;
  const int u = blockIdx.x, head = blockIdx.y, b = blockIdx.z - (is_v ? A.num_seqs : 0);
  if (A.tile_start[b] < 0) return;  // nothing to commit for this sequence (uniform per CTA)
  const int64_t off = static_cast<int64_t>(b) * A.seq_stride + static_cast<int64_t>(head) * A.head_stride +
                      static_cast<int64_t>(u) * N * D;
  if (is_v)
    encode_tile<D, N, 1, VB, 0, true, KB, VB, SB>(A, static_cast<const unsigned char*>(A.x[1]) + 2 * off, b, head, u,
                                                     A.tile_start[b] + u, nullptr, smem);
  else
    encode_tile<D, N, 1, KB, 0, false, KB, VB, SB>(A, static_cast<const unsigned char*>(A.x[0]) + 2 * off, b, head, u,
                                                      A.tile_start[b] + u, nullptr, smem);
}


// Fused append + commit (one launch per decode step): x[0] / x[1] hold each
// (sequence, KV head)'s newest K / V token, at position seq_lens[b] - 1. A
// token that does not complete a tile goes to its row of the raw tail; one
// that does completes the tile in the tail's rows 0..N-2 and the tile is
// encoded straight into its pages (the tail then holds nothing). The tail
// rows read here were written by earlier launches.
template <int D, int N>
__global__ void __launch_bounds__(2 * D, D == 128 ? 2 : 1) append_commit_kernel(EncodeArgs A, const int32_t* seq_lens,
                                                              int32_t max_seq_len, unsigned char* tail_k,
                                                              unsigned char* tail_v) {
  extern __shared__ __align__(128) unsigned char smem[];
  pdl_launch_dependents();
  const bool is_v = blockIdx.z == 1;
  const int head = blockIdx.x, b = blockIdx.y;
  const int L = seq_lens[b];
  if (L <= 0 || L > max_seq_len) {  // nothing appended (0) or an invalid length
    if (L != 0 && threadIdx.x == 0 && !is_v && head == 0) set_error(A.err, KVARN_DEVERR_SEQ_LEN);
    return;
  }
  const int64_t hs = static_cast<int64_t>(b) * A.num_kv_heads + head;
  // 16-bit elements (fp16 or bf16)
  const unsigned char* tok = static_cast<const unsigned char*>(A.x[is_v]) + 2 * hs * D;
  unsigned char* tail = (is_v ? tail_v : tail_k) + 2 * hs * N * D;
  if (L % N != 0) {
    const int row = (L - 1) % N;
    for (int i = threadIdx.x; i < D / 8; i += blockDim.x)
      reinterpret_cast<uint4*>(tail + 2 * static_cast<int64_t>(row) * D)[i] = reinterpret_cast<const uint4*>(tok)[i];
    return;
  }
  if (is_v)
    encode_tile<D, N, 1, 2, 0, true>(A, tail, b, head, 0, L / N - 1, tok, smem);
  else
    encode_tile<D, N, 1, 4, 0, false>(A, tail, b, head, 0, L / N - 1, tok, smem);
}

// ------------------------------------------------------------- launchers
template <int D, int N, int KB = 4, int VB = 2, int SB = 4>
cudaError_t launch_dense(const EncodeArgs& A, cudaStream_t st) {
  constexpr bool gen = !(KB == 4 && VB == 2);
  constexpr int smem = gen ? EncShape<D, N, 1, true>::SMEM : EncShape<D, N, 1>::SMEM;
  auto kern = encode_dense_kernel<D, N, KB, VB, SB>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  dim3 grid(A.chunk_tiles, A.num_kv_heads, 2 * A.num_seqs);
  kern<<<grid, 2 * D, smem, st>>>(A);
  return cudaGetLastError();
}

// The dense encode kernels of one (K width, V width, scale bytes)
// combination (head_dim 128); each combination compiles in its own
// translation unit.
template <int KB, int VB, int SB>
cudaError_t launch_encode_widths(const EncodeArgs& A, int N, bool bf16, cudaStream_t st);

#define KVARN_DECLARE_ENC_WIDTHS(KB, VB) \
  template <>                            \
  cudaError_t launch_encode_widths<KB, VB, 2>(const EncodeArgs& A, int N, bool bf16, cudaStream_t st);
KVARN_WIDTH_PAIRS(KVARN_DECLARE_ENC_WIDTHS)
#define KVARN_DECLARE_ENC_WIDTHS_S32(KB, VB) \
  template <>                                \
  cudaError_t launch_encode_widths<KB, VB, 4>(const EncodeArgs& A, int N, bool bf16, cudaStream_t st);
KVARN_WIDTH_PAIRS_S32(KVARN_DECLARE_ENC_WIDTHS_S32)
#undef KVARN_DECLARE_ENC_WIDTHS_S32
template <int KB, int VB, int SB>
cudaError_t launch_encode_widths256(const EncodeArgs& A, int N, bool bf16, cudaStream_t st);
#define KVARN_DECLARE_ENC_WIDTHS_256(KB, VB) \
  template <>                                \
  cudaError_t launch_encode_widths256<KB, VB, 2>(const EncodeArgs& A, int N, bool bf16, cudaStream_t st);
KVARN_WIDTH_PAIRS_256(KVARN_DECLARE_ENC_WIDTHS_256)
#undef KVARN_DECLARE_ENC_WIDTHS_256
#undef KVARN_DECLARE_ENC_WIDTHS

#define KVARN_ENCODE_WIDTHS(KB, VB, SB)                                                                \
  template <>                                                                                          \
  cudaError_t launch_encode_widths<KB, VB, SB>(const EncodeArgs& A, int N, bool /*bf16*/, cudaStream_t st) { \
    if (N == 128)                                                                                      \
      return launch_dense<128, 128, KB, VB, SB>(A, st);                                 \
    if (N == 64)                                                                                       \
      return launch_dense<128, 64, KB, VB, SB>(A, st);                                  \
    return cudaErrorInvalidValue;                                                                      \
  }

#define KVARN_ENCODE_WIDTHS_256(KB, VB)                                                                 \
  template <>                                                                                         \
  cudaError_t launch_encode_widths256<KB, VB, 2>(const EncodeArgs& A, int N, bool /*bf16*/, cudaStream_t st) { \
    if (N == 128)                                                                                     \
      return launch_dense<256, 128, KB, VB, 2>(A, st);                                 \
    if (N == 64)                                                                                      \
      return launch_dense<256, 64, KB, VB, 2>(A, st);                                  \
    return cudaErrorInvalidValue;                                                                     \
  }

}  // namespace kvarn

// KVarN decode attention over the compressed paged cache, sm_103a.
//
// Paged, split-K, GQA-grouped decode that streams the packed codes and
// scales straight from HBM and dequantises them in registers; no fp16 K or V
// buffer is ever formed (turbo-attn page, "Inline dequant"). Scores are
// taken in the rotated basis: the query is rotated once per CTA and the
// output un-rotated once in the merge (turbo-attn page, "How it works").
//
// Kernel 1 (decode_dense_kernel): persistent CTAs, each taking an equal
// contiguous range of the flattened list of committed tiles of all
// (sequence, KV head, row group) units (stream-K) and writing one partial
// per unit its range touches; a segment's tiles go round-robin to the W
// warps (warp pairs at head_dim 256). The CTAs also take the raw-record
// chunks (sink and tail rows) round-robin, before their tiles. A warp keeps one
// shared-memory slot for the K parts and one for the V parts of its tile's
// pages, filled by one-dimensional bulk copies (completion counted on an
// mbarrier); an L2 prefetch of later tiles measured slower (its lines were
// partly evicted and read twice) and is not used. The K slot
// is refilled with the next tile while P V runs, the V slot while the next
// Q K runs. Per tile and warp:
//   q~ = (kappa q H) * c_K, split into fp16 hi + lo rows of the mma A tile
//        (rows 0-7 hi, 8-15 lo: the G <= 8 query heads of the group leave
//        half of the m16 tile free, so the split costs no extra mma);
//   S  = q~ . (K codes / 8)^T with mma.sync m16n8k16 (the codes as exact fp16
//        multiples of 1/8, one hardware e2m3 -> fp16 conversion per operand
//        register after one mask per four registers);
//   s  = 8 a_K * S + b_K * sum(q~)              (row scales folded back in);
//   online softmax in base 2;
//   u  = (p * a_V)(V codes / 2) with the same hi/lo A tile (e2m1 -> fp16);
//   acc = acc * alpha + c_V * (2 u + sum p b_V).
// The warps of a CTA merge in shared memory and write one partial
// (max, sum, unnormalised output) per segment; the raw partials (original
// basis) sit in the slots after the tile partials, and each row's count of
// tile partials is written beside them.
// Kernel 2 (merge_kernel): log-sum-exp merge of the partials, inverse
// Hadamard transform of the rotated part, plus the tail part.
#pragma once

#include <cuda.h>
#include <math.h>

#include <algorithm>

#include "kvarn_common.cuh"
#include "kvarn_launch.h"
#include "kvarn_merge.cuh"

namespace kvarn {

constexpr float kLog2e = 1.4426950408889634f;

// CTAs per SM the 4-warp decode kernel is register-limited to (3 caps it at
// 168 registers per thread, 2 at 255).
#ifndef KVARN_DECODE_MIN_CTAS
#define KVARN_DECODE_MIN_CTAS 3
#endif

// Floats per k-chunk block of the rotated query rows in shared memory: the
// block's 128 (8 rows x 4 lane columns x 4 channels) plus 4 of padding, so
// that the scalar stores that build the rows (one lane per k-chunk, a block
// apart) fall in different banks.
constexpr int kQFragStride = 132;

// Floats per row of the merge scratch: m, l, two pads, then D values; a
// stride of 8 modulo the 32 banks keeps the row-wise float2 / float4 stores
// of a warp on distinct banks.
template <int D> constexpr int merge_stride() { return D + 8; }

// HV warps share a tile (HV = 2 at head_dim 256: each warp owns half of the
// channels of Q K and of P V, and the pair adds its partial scores).
template <int D> constexpr int halves_for() { return D == 256 ? 2 : 1; }

// Codecs of the decode skeleton: the KVarN pages, the affine comparison
// codec (per-token groups of 64 channels with an fp16 scale and offset each,
// original basis), or none: the uncompressed fp16 pages (K and V in fragment
// order, original basis; tiles of 32 tokens, the last one partial).
constexpr int kCodecKvarn = 0, kCodecAffine = 1, kCodecRaw = 2;

template <int D, int N, int W, int KB = 4, int VB = 2, int SB = 4, int CD = kCodecKvarn>
struct DecShape {
  static constexpr int HV = halves_for<D>();
  static constexpr int UNITS = W / HV;  // tiles in flight per CTA
  static constexpr DensePage PG{D, N, KB, VB, SB};
  static constexpr AffinePage AG{D, KB, VB};
  static constexpr bool AFF = CD == kCodecAffine;
  static constexpr bool RAW = CD == kCodecRaw;
  static constexpr int PPT = N / kPageTokens;
  static constexpr int RAW_PART = 2 * kPageTokens * D;  // fp16 K (or V) of a page
  static constexpr int PB = RAW ? 2 * RAW_PART : AFF ? AG.bytes() : PG.bytes();
  static constexpr int KP = RAW ? RAW_PART : AFF ? AG.k_part() : PG.k_part();
  static constexpr int VP = RAW ? RAW_PART : AFF ? AG.v_part() : PG.v_part();
  static constexpr int GR = D / 64;  // affine groups per token
  static constexpr int KSLOT = PPT * KP;
  static constexpr int VSLOT = PPT * VP;
  static constexpr int WARP_SMEM = KSLOT + VSLOT;
  static constexpr int NB = N / 8;
  static constexpr int KC = D / 16;
  static constexpr int NC = D / 8;
  static constexpr int CPP = PG.cols();
  static constexpr int KCH = D / 64;  // groups of four k-chunks (eight K fragments) per page
  static constexpr int VHC = D / 64;  // groups of eight channel blocks (eight V fragments) per page
  // code planes (width, fragments per word, words per unit, region offset)
  static constexpr int KW0 = plane_w0(KB), KW1 = plane_w1(KB), VW0 = plane_w0(VB), VW1 = plane_w1(VB);
  static constexpr int KF0 = 8 / KW0, KF1 = KW1 ? 8 / KW1 : 8, VF0 = 8 / VW0, VF1 = VW1 ? 8 / VW1 : 8;
  static constexpr int KU0 = D * KW0 / 64 < 4 ? D * KW0 / 64 : 4;
  static constexpr int KU1 = KW1 ? (D * KW1 / 64 < 4 ? D * KW1 / 64 : 4) : 1;
  static constexpr int KR1 = 2 * D * KW0, VR1 = 2 * D * VW0;
  // operand values are code_kappa(bits) * (code - code_center(bits))
  static constexpr float KINV = 1.f / code_kappa(KB), VINV = 1.f / code_kappa(VB);
  static constexpr float KCENTER = static_cast<float>(code_center(KB)), VCENTER = static_cast<float>(code_center(VB));
  static constexpr int RING = UNITS * WARP_SMEM;
  static constexpr int XS = 2 * (N / 8) + 2;  // exchanged per lane: partial scores, two timeout flags
  static constexpr int XBUF = HV == 2 ? UNITS * 2 * 32 * XS * 4 : 0;
  static constexpr int OFF_BARS = RING, OFF_QROT = RING + UNITS * 2 * 8;
  static constexpr int OFF_XBUF = OFF_QROT + (D / 16) * kQFragStride * 4;
  // raw-record scratch, taken from the page slots (which no copy touches
  // before the tile loop starts) where it fits. While a CTA scores its raw
  // records: each warp's weight block (32 records x 8 rows) and, at head_dim
  // 128 where they fit in the slots, its staged key rows (32 rows, each padded
  // by 16 bytes so that the lanes' reads of their own rows do not collide);
  // elsewhere a lane reads its key row from global memory. Afterwards, at
  // the same place, the warps' partials for the merge (a barrier between).
  // The channel-major query rows (8 x D floats) take the query-row region.
  static constexpr int RAW_MRG = W * 8 * merge_stride<D>() * 4;
  static constexpr int RAW_PB = W * 32 * 8 * 4;
  static constexpr int RAW_KROW = 2 * D + 16;
  static constexpr int RAW_KST = HV == 1 && !RAW && RAW_PB + W * 32 * RAW_KROW <= RING ? W * 32 * RAW_KROW : 0;
  static constexpr int RAW_P1 = RAW_PB + RAW_KST;
  static constexpr bool MRG_IN = RAW_MRG <= RING;
  static constexpr int END0 = OFF_XBUF + XBUF;
  static constexpr int OFF_RAW_MRG = MRG_IN ? 0 : END0;
  static constexpr int OFF_RAW_PB = RAW_P1 <= RING ? 0 : XBUF >= RAW_P1 ? OFF_XBUF : END0;
  static constexpr int OFF_RAW_KST = OFF_RAW_PB + RAW_PB;
  static constexpr int SMEM = END0 + (MRG_IN ? 0 : RAW_MRG) > OFF_RAW_PB + RAW_P1 ? END0 + (MRG_IN ? 0 : RAW_MRG)
                                                                                    : OFF_RAW_PB + RAW_P1;
  static_assert(UNITS * 8 * merge_stride<D>() * 4 <= RING, "tile merge scratch must fit in the slots");
  static_assert(8 * D * 4 <= (D / 16) * kQFragStride * 4 && W * 40 * 4 <= (D / 16) * kQFragStride * 4,
                "raw-record query rows and weight exchange must fit in the query-row region");
  static_assert(OFF_RAW_PB % 16 == 0 && OFF_RAW_KST % 16 == 0 && RAW_KROW % 16 == 0, "raw scratch alignment");
  static_assert(W % HV == 0, "whole warp pairs");
  static_assert(KP % 16 == 0 && VP % 16 == 0, "page parts must keep 16-byte alignment");
  static constexpr bool GATHER = parts_gather(D, N, KP, VP, KB, VB);
  static_assert(!AFF || HV == 1, "the affine codec is compiled at head_dim 128");
  static_assert(!RAW || (N == 32 && !GATHER), "fp16 pages: tiles of two pages, copied by cp.async");
  // first-box widths of the K and V parts (the whole part unless split)
  static constexpr int KS = GATHER ? gather_split(KP, 2 * D * KB) : KP;
  static constexpr int VS = GATHER ? gather_split(VP, 2 * D * VB) : VP;
  static_assert(!GATHER || (KSLOT % 128 == 0 && WARP_SMEM % 128 == 0), "gather destinations stay 128-byte aligned");
};

struct DecArgs {
  // 2-D tensor maps over the cache (one row per (page, KV head), 8-byte
  // elements) with boxes of a page's K part and of its V part: the TMA
  // gathers of the shapes dense_gather() selects (unused otherwise)
  CUtensorMap tmk, tmk2, tmv, tmv2;  // second boxes of split parts
  const void* q;  // [B][Q][Hq][D]
  float kappa;    // sm_scale * log2(e)
  const uint8_t* cache;
  int32_t Hq, Hkv, G;
  int32_t Q;           // query tokens per sequence (speculative verify: the last Q tokens)
  int32_t tail_cap;    // tail rows per (sequence, KV head)
  int32_t sink_tiles;  // raw sink records: tokens [0, sink_tiles N) are rows of sink_k / sink_v
  int32_t recent;      // raw recent records: the newest `recent` accepted tokens stay in the tail
  const void* sink_k;
  const void* sink_v;
  int64_t num_pages;
  const int32_t* bt;
  int32_t bt_stride;
  const int32_t* seq_lens;
  int32_t max_seq_len;
  const void* tail_k;
  const void* tail_v;
  float* ws;
  int32_t* counts;     // per output row: tile partial slots written for it (slots [0, count))
  int32_t num_seqs;
  int32_t X;           // work units per sequence: KV heads x row groups
  int32_t min_tiles;   // fewest compressed tiles a CTA takes (bounds the slots a unit needs)
  int32_t tile_slots;  // partial slots reserved for compressed tiles; raw slots follow them
  int32_t raw_splits;  // raw slots (chunks of raw_chunk raw tokens)
  int32_t raw_chunk;   // raw tokens per raw split
  int32_t slots;       // tile_slots + raw_splits
  uint32_t* err;
  int32_t partial_tiles;  // uncompressed pages: a sequence's last tile may be partial (tokens past len masked)
  long long wait_limit;   // clock cycles a page copy is waited for before the kernel gives up
  int32_t bf16;           // storage dtype of q and of the raw records: 0 fp16, 1 bf16
  int32_t withhold;       // diagnostic: every copy is announced this many bytes larger (its phase never completes)
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

// E consecutive fp16 or bf16 elements (the storage dtype chosen at run time:
// the branch is uniform over the grid).
template <int E>
__device__ __forceinline__ void load_vec_rt(const void* p, bool bf16, float* out) {
  if (bf16)
    load_vec<__nv_bfloat16, E>(static_cast<const __nv_bfloat16*>(p), out);
  else
    load_vec<__half, E>(static_cast<const __half*>(p), out);
}

__device__ __forceinline__ void write_empty(float* part, int D, int lane) {
  if (lane == 0) {
    part[0] = -INFINITY;
    part[1] = 0.f;
  }
  for (int j = lane; j < D; j += 32) part[4 + j] = 0.f;
}

// Rows of a CTA: up to eight (query head, query token) pairs, pair p = 8 rg + r
// with head p % G and query token p / G, so that one mma row tile serves G Q
// <= 8 pairs at the cost of one.
struct RowMap {
  int rg, n;  // row group, rows used in it
  __device__ RowMap(const DecArgs& A, int rg_) : rg(rg_), n(min(8, A.G * A.Q - 8 * rg_)) {}
  __device__ int head(const DecArgs& A, int r) const { return (8 * rg + r) % A.G; }
  __device__ int query(const DecArgs& A, int r) const { return (8 * rg + r) / A.G; }
};

// The rotated, scaled query rows in shared memory, in mma fragment order:
// for k-chunk kc, row g and lane column t the four channels 16 kc + 2 t,
// +1, +8, +9 are one 16-byte word, and a warp's 32 words for one k-chunk are
// contiguous (one conflict-free 128-bit load per lane); k-chunk blocks are
// kQFragStride floats apart.
__device__ __forceinline__ int q_frag(int kc, int g, int t) { return kc * kQFragStride + (g * 4 + t) * 4; }

// Partial slot of (sequence b, query token j, query head hq).
__device__ __forceinline__ float* part_of(const DecArgs& A, int D, int b, int j, int hq, int slot) {
  return A.ws + (static_cast<int64_t>((b * A.Q + j) * A.Hq + hq) * A.slots + slot) * kPStride(D);
}

// Tokens visible to query token j of a sequence of len tokens (causal among
// the Q tokens under verification), and the committed prefix shared by all.
__device__ __forceinline__ int visible_len(int len, int Q, int j) { return max(0, len - Q + 1 + j); }

// ------------------------------------------------------------- raw records
// E consecutive fp16 or bf16 elements as raw bits (converted at use, so that a
// prefetched row holds half the registers of its floats).
template <int E>
struct RawRow {
  uint32_t w[E / 2];
};
template <int E>
__device__ __forceinline__ RawRow<E> raw_load(const void* p) {
  RawRow<E> r;
  if constexpr (E == 4) {
    const uint2 u = __ldg(reinterpret_cast<const uint2*>(p));
    r.w[0] = u.x;
    r.w[1] = u.y;
  } else {
    static_assert(E % 8 == 0, "vector width");
#pragma unroll
    for (int k = 0; k < E / 8; ++k) {
      const uint4 u = __ldg(reinterpret_cast<const uint4*>(p) + k);
      r.w[4 * k] = u.x;
      r.w[4 * k + 1] = u.y;
      r.w[4 * k + 2] = u.z;
      r.w[4 * k + 3] = u.w;
    }
  }
  return r;
}
// The same from shared memory.
template <int E>
__device__ __forceinline__ RawRow<E> raw_shared(const unsigned char* p) {
  RawRow<E> r;
  if constexpr (E == 4) {
    const uint2 u = *reinterpret_cast<const uint2*>(p);
    r.w[0] = u.x;
    r.w[1] = u.y;
  } else {
    static_assert(E % 8 == 0, "vector width");
#pragma unroll
    for (int k = 0; k < E / 8; ++k) {
      const uint4 u = reinterpret_cast<const uint4*>(p)[k];
      r.w[4 * k] = u.x;
      r.w[4 * k + 1] = u.y;
      r.w[4 * k + 2] = u.z;
      r.w[4 * k + 3] = u.w;
    }
  }
  return r;
}
template <int E>
__device__ __forceinline__ void raw_floats(const RawRow<E>& r, bool bf16, float* out) {
#pragma unroll
  for (int k = 0; k < E / 2; ++k) {
    float2 f;
    if (bf16)
      f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&r.w[k]));
    else
      f = __half22float2(*reinterpret_cast<const __half2*>(&r.w[k]));
    out[2 * k] = f.x;
    out[2 * k + 1] = f.y;
  }
}

// Raw (sink and tail) records of a unit: dense attention in the original
// basis, in fp32 on the CUDA cores. Row r of the unit (a (head, query token)
// pair) attends to the raw tokens at positions below its visible length: the
// sink rows [0, min(sink, visible)) and the tail rows for tokens [committed,
// visible). All rows of the unit share one raw list, the sink rows of the
// longest row then its tail rows, masked per row by position; raw split
// `chunk` covers list entries [chunk * raw_chunk, +raw_chunk), cut into W
// consecutive pieces, one per warp. Each warp leaves the (max, sum,
// unnormalised output) of its piece per row in the merge scratch `mrg`
// (8 rows of merge_stride<D>() floats per warp), and the pieces are merged
// per row into the split's partial.
//
// The list of a split: row r's query token, query head and visible length in
// lane r (r < R.n), the list bounds, and where its records start.
struct RawSplit {
  int qj_l = 0, hq_l = 0, vis_l = 0;
  int n_sink, c0, c1, committed, slot;
  int64_t sink0, tail0;
  bool miss;
  __device__ RawSplit(const DecArgs& A, const RowMap& R, int N, int b, int kvh, int len, int sink, int committed_,
                      int chunk) {
    const int lane = threadIdx.x & 31;
    if (lane < R.n) {
      qj_l = R.query(A, lane);
      hq_l = kvh * A.G + R.head(A, lane);
      vis_l = visible_len(len, A.Q, qj_l);
    }
    // the longest row's list bounds everything read
    int vis_max = vis_l;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) vis_max = max(vis_max, __shfl_xor_sync(0xffffffffu, vis_max, o));
    committed = committed_;
    n_sink = min(sink, vis_max);
    const int n_tail = max(0, vis_max - committed);
    c0 = chunk * A.raw_chunk;
    c1 = min(n_sink + n_tail, c0 + A.raw_chunk);
    miss = (c1 > max(c0, n_sink) && (A.tail_k == nullptr || A.tail_v == nullptr)) ||
           (min(c1, n_sink) > c0 && (A.sink_k == nullptr || A.sink_v == nullptr));
    slot = A.tile_slots + chunk;
    sink0 = (static_cast<int64_t>(b) * A.Hkv + kvh) * (A.sink_tiles * N);
    tail0 = (static_cast<int64_t>(b) * A.Hkv + kvh) * A.tail_cap;
  }
  __device__ int qj(int r) const { return __shfl_sync(0xffffffffu, qj_l, r); }
  __device__ int hq(int r) const { return __shfl_sync(0xffffffffu, hq_l, r); }
  __device__ int position(int i) const { return i < n_sink ? i : committed + (i - n_sink); }
  // record row of list entry i (keys or values)
  __device__ const char* row(const DecArgs& A, int D, int i, bool v) const {
    const void* base = i < n_sink ? (v ? A.sink_v : A.sink_k) : (v ? A.tail_v : A.tail_k);
    return static_cast<const char*>(base) + 2 * D * (i < n_sink ? sink0 + i : tail0 + (i - n_sink));
  }
};

// Scoring with the channels split over the lanes (head_dim 256, and where the
// key rows of a block cannot be staged): a lane holds D / 32 channels of the
// rows of a pass (all eight at head_dim 128, four at 256: two passes over
// the records, which keeps the kernel's register budget of the tile loop).
// Per step of four records a lane forms its channels' products for the
// rows x 4 (row, record) pairs, and a reduce-scatter over the warp leaves
// lane l with the whole score of pair l mod (4 x rows); online softmax per
// row over groups of four lanes, the weights and rescales to every lane
// through 160 bytes of shared memory (`pxbuf`); the next four records load
// while the current ones are scored.
template <int D, int N, int W>
__device__ void raw_pieces_by_channel(const DecArgs& A, const RawSplit& L, float* mw, float* pxbuf, int b,
                                      const RowMap& R, int w0, int w1) {
  constexpr int E = D / 32, U = 4, RP = D == 256 ? 4 : 8, PAIRS = RP * U;
  constexpr int MS = merge_stride<D>();
  const int lane = threadIdx.x & 31;
  const int my_r = (lane & (PAIRS - 1)) >> 2, my_u = lane & 3;  // pair of the lane after the reduce-scatter
  for (int r0 = 0; r0 < R.n; r0 += RP) {
    // this lane's channels of the pass's query rows, kappa-scaled (zero past R.n)
    float q[RP][E];
#pragma unroll
    for (int r = 0; r < RP; ++r) {
      const int qj = L.qj(r0 + r), hq = L.hq(r0 + r);
      if (r0 + r < R.n) {
        const int64_t qoff = (static_cast<int64_t>(b * A.Q + qj) * A.Hq + hq) * D + lane * E;
        load_vec_rt<E>(static_cast<const char*>(A.q) + 2 * qoff, A.bf16, q[r]);
#pragma unroll
        for (int e = 0; e < E; ++e) q[r][e] *= A.kappa;
      } else {
#pragma unroll
        for (int e = 0; e < E; ++e) q[r][e] = 0.f;
      }
    }
    const int my_vis = __shfl_sync(0xffffffffu, L.vis_l, r0 + my_r);
    float acc[RP][E];
#pragma unroll
    for (int r = 0; r < RP; ++r)
#pragma unroll
      for (int e = 0; e < E; ++e) acc[r][e] = 0.f;
    float m = -INFINITY, l = 0.f;  // row r0 + my_r (the same in every lane of the row)
    RawRow<E> kb[U], vb[U];
    auto fetch = [&](int i0) {
#pragma unroll
      for (int u = 0; u < U; ++u) {
        if (i0 + u < w1) {
          kb[u] = raw_load<E>(L.row(A, D, i0 + u, false) + 2 * lane * E);
          vb[u] = raw_load<E>(L.row(A, D, i0 + u, true) + 2 * lane * E);
        } else {
#pragma unroll
          for (int k = 0; k < E / 2; ++k) kb[u].w[k] = vb[u].w[k] = 0u;
        }
      }
    };
    if (w0 < w1) fetch(w0);
    for (int i0 = w0; i0 < w1; i0 += U) {
      RawRow<E> kc[U], vc[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        kc[u] = kb[u];
        vc[u] = vb[u];
      }
      if (i0 + U < w1) fetch(i0 + U);  // the next step's records load during this one
      // partial products of pair (r, u) over this lane's channels
      float v[PAIRS];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        float kf[E];
        raw_floats<E>(kc[u], A.bf16, kf);
#pragma unroll
        for (int r = 0; r < RP; ++r) {
          float d = 0.f;
#pragma unroll
          for (int e = 0; e < E; ++e) d = fmaf(q[r][e], kf[e], d);
          v[4 * r + u] = d;
        }
      }
      // whole sums over the lanes above the pair count, then a
      // reduce-scatter: at the stage of offset o a lane keeps the half of
      // its values that its bit o selects and adds its partner's copy of it
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1) {
        if (o >= PAIRS) {
#pragma unroll
          for (int i = 0; i < PAIRS; ++i) v[i] += __shfl_xor_sync(0xffffffffu, v[i], o);
        } else {
          const bool up = (lane & o) != 0;
#pragma unroll
          for (int i = 0; i < o; ++i) {
            const float keep = up ? v[i + o] : v[i], give = up ? v[i] : v[i + o];
            v[i] = keep + __shfl_xor_sync(0xffffffffu, give, o);
          }
        }
      }
      const int i = i0 + my_u;
      const float s = (i < w1 && L.position(i) < my_vis) ? v[0] : -INFINITY;
      const float mx = fmaxf(fmaxf(s, __shfl_xor_sync(0xffffffffu, s, 1)),
                             fmaxf(__shfl_xor_sync(0xffffffffu, s, 2), __shfl_xor_sync(0xffffffffu, s, 3)));
      const float m_new = fmaxf(m, mx);
      const float alpha = m_new == -INFINITY ? 1.f : exp2f(m - m_new);
      const float p = s == -INFINITY ? 0.f : exp2f(s - m_new);
      l = fmaf(l, alpha, warp_sum_xor(p, 1, 4));
      m = m_new;
      // weights and rescales of every row to every lane (lanes holding the
      // same pair store the same value)
      pxbuf[lane & (PAIRS - 1)] = p;
      if (my_u == 0) pxbuf[32 + my_r] = alpha;
      __syncwarp();
      float vf[U][E];
#pragma unroll
      for (int u = 0; u < U; ++u) raw_floats<E>(vc[u], A.bf16, vf[u]);
#pragma unroll
      for (int r = 0; r < RP; ++r) {
        const float4 pr = *reinterpret_cast<const float4*>(pxbuf + 4 * r);
        const float al = pxbuf[32 + r];
#pragma unroll
        for (int e = 0; e < E; ++e) {
          float a = acc[r][e] * al;
          a = fmaf(pr.x, vf[0][e], a);
          a = fmaf(pr.y, vf[1][e], a);
          a = fmaf(pr.z, vf[2][e], a);
          acc[r][e] = fmaf(pr.w, vf[3][e], a);
        }
      }
      __syncwarp();
    }
    // this warp's piece of the pass's rows into the merge scratch
    if (my_u == 0 && lane < PAIRS) {
      mw[(r0 + my_r) * MS] = m;
      mw[(r0 + my_r) * MS + 1] = l;
    }
#pragma unroll
    for (int r = 0; r < RP; ++r)
#pragma unroll
      for (int e = 0; e < E; e += 4)
        *reinterpret_cast<float4*>(mw + (r0 + r) * MS + 4 + lane * E + e) =
            make_float4(acc[r][e], acc[r][e + 1], acc[r][e + 2], acc[r][e + 3]);
  }
}

// Scoring with one record per lane (head_dim 128 where a block's key rows fit
// in the page slots). A warp takes its piece in blocks of 32 records:
//  - the block's key rows are copied into shared memory coalesced (`kst`,
//    rows padded by 16 bytes) and each lane reads its own record's row back;
//    it forms the dot products with all eight rows, whose kappa-scaled query
//    channels come channel-major from shared memory (`qs`: qs[8 d + r], one
//    broadcast load per four rows), so no score needs a cross-lane sum;
//  - softmax: per row, the block maximum over the lanes, the rescale of the
//    running state, base-2 weights; each lane keeps its own partial of the
//    row sums (one warp sum per row at the end);
//  - P.V: the block's value rows are copied into the staging rows once the
//    keys are read (the copy runs while the weights are formed), the weights
//    go through shared memory (`pw`, 1 KB per warp), and the lane owns D / 32
//    channels of every row's accumulator and walks the block's records.
template <int D, int N, int W>
__device__ void raw_pieces_by_record(const DecArgs& A, const RawSplit& L, float* mw, const float* qs, float* pw,
                                     unsigned char* kw, int w0, int w1) {
  constexpr int E = D / 32, KROW = 2 * D + 16, MS = merge_stride<D>();
  const int lane = threadIdx.x & 31;
  int vis[8];
#pragma unroll
  for (int r = 0; r < 8; ++r) vis[r] = __shfl_sync(0xffffffffu, L.vis_l, r);
  float acc[8][E], m[8], l[8];
#pragma unroll
  for (int r = 0; r < 8; ++r) {
    m[r] = -INFINITY;
    l[r] = 0.f;
#pragma unroll
    for (int e = 0; e < E; ++e) acc[r][e] = 0.f;
  }
  // P.V of record j of the block from its value row, staged in shared memory
  auto pv = [&](int j) {
    float vf[E];
    raw_floats<E>(raw_shared<E>(kw + j * KROW + 2 * lane * E), A.bf16, vf);
    const float4 pa = *reinterpret_cast<const float4*>(pw + j * 8);
    const float4 pb = *reinterpret_cast<const float4*>(pw + j * 8 + 4);
    const float p8[8] = {pa.x, pa.y, pa.z, pa.w, pb.x, pb.y, pb.z, pb.w};
#pragma unroll
    for (int r = 0; r < 8; ++r)
#pragma unroll
      for (int e = 0; e < E; ++e) acc[r][e] = fmaf(p8[r], vf[e], acc[r][e]);
  };
  for (int blk = w0; blk < w1; blk += 32) {
    const int nrec = min(32, w1 - blk);
    // the block's key (then value) rows, coalesced: 16-byte piece lane + 32 t
    // is piece (lane + 32 t) % (D / 8) of row (lane + 32 t) / (D / 8)
    auto stage_rows = [&](bool v) {
#pragma unroll 4
      for (int t = 0; t < D / 8; ++t) {
        const int q = lane + 32 * t, row = q / (D / 8), col = q % (D / 8);
        if (row < nrec) cp_async16(kw + row * KROW + 16 * col, L.row(A, D, blk + row, v) + 16 * col);
      }
    };
    stage_rows(false);
    cp_async_wait_all();
    __syncwarp();
    const int i = blk + lane;
    const bool valid = i < w1;
    float s[8];
#pragma unroll
    for (int r = 0; r < 8; ++r) s[r] = 0.f;
    if (valid) {
#pragma unroll 8
      for (int c = 0; c < D / 8; ++c) {
        RawRow<8> k8;
        const uint4 u = *reinterpret_cast<const uint4*>(kw + lane * KROW + 16 * c);
        k8.w[0] = u.x;
        k8.w[1] = u.y;
        k8.w[2] = u.z;
        k8.w[3] = u.w;
        float kf[8];
        raw_floats<8>(k8, A.bf16, kf);
#pragma unroll
        for (int dd = 0; dd < 8; ++dd) {
          const float4 qa = *reinterpret_cast<const float4*>(qs + (8 * c + dd) * 8);
          const float4 qb = *reinterpret_cast<const float4*>(qs + (8 * c + dd) * 8 + 4);
          s[0] = fmaf(qa.x, kf[dd], s[0]);
          s[1] = fmaf(qa.y, kf[dd], s[1]);
          s[2] = fmaf(qa.z, kf[dd], s[2]);
          s[3] = fmaf(qa.w, kf[dd], s[3]);
          s[4] = fmaf(qb.x, kf[dd], s[4]);
          s[5] = fmaf(qb.y, kf[dd], s[5]);
          s[6] = fmaf(qb.z, kf[dd], s[6]);
          s[7] = fmaf(qb.w, kf[dd], s[7]);
        }
      }
    }
    // every lane is done with its key row: the value rows take their place
    // while the weights are formed
    __syncwarp();
    stage_rows(true);
    const int pos = L.position(i);
#pragma unroll
    for (int r = 0; r < 8; ++r) {
      const float sr = valid && pos < vis[r] ? s[r] : -INFINITY;
      float bm = sr;
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1) bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, o));
      const float mn = fmaxf(m[r], bm);
      const float al = mn == -INFINITY ? 1.f : exp2f(m[r] - mn);
      const float p = sr == -INFINITY ? 0.f : exp2f(sr - mn);
      l[r] = fmaf(l[r], al, p);
      m[r] = mn;
#pragma unroll
      for (int e = 0; e < E; ++e) acc[r][e] *= al;
      s[r] = p;
    }
    // the block's weights to every lane
    *reinterpret_cast<float4*>(pw + lane * 8) = make_float4(s[0], s[1], s[2], s[3]);
    *reinterpret_cast<float4*>(pw + lane * 8 + 4) = make_float4(s[4], s[5], s[6], s[7]);
    cp_async_wait_all();
    __syncwarp();
#pragma unroll 4
    for (int j = 0; j < nrec; ++j) pv(j);
    __syncwarp();  // pw and the staged rows are rewritten by the next block
  }
#pragma unroll
  for (int r = 0; r < 8; ++r) l[r] = warp_sum_xor(l[r], 1, 32);
  // this warp's piece into the merge scratch, which the other warps' weight
  // blocks and key rows may occupy until they are done
  __syncthreads();
  if (lane == 0) {
#pragma unroll
    for (int r = 0; r < 8; ++r) {
      mw[r * MS] = m[r];
      mw[r * MS + 1] = l[r];
    }
  }
#pragma unroll
  for (int r = 0; r < 8; ++r)
#pragma unroll
    for (int e = 0; e < E; e += 4)
      *reinterpret_cast<float4*>(mw + r * MS + 4 + lane * E + e) =
          make_float4(acc[r][e], acc[r][e + 1], acc[r][e + 2], acc[r][e + 3]);
}

// The raw partials of split `chunk` of a unit. KST: scoring by record with
// the key rows staged in shared memory (`kst`, `pbuf` the weight blocks, `qs`
// the channel-major query rows), else by channel (`pxbuf`).
template <int D, int N, int W, bool KST>
__device__ void tail_partials(const DecArgs& A, unsigned char* mrg_smem, float* qrows, float* pbuf, unsigned char* kst,
                              int b, int kvh, const RowMap& R, int len, int sink, int committed, int chunk) {
  constexpr int MS = merge_stride<D>();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const RawSplit L(A, R, N, b, kvh, len, sink, committed, chunk);
  if (L.c1 <= L.c0 || L.miss) {
    if (L.miss && threadIdx.x == 0) set_error(A.err, KVARN_DEVERR_NO_TAIL);
    for (int r = warp; r < R.n; r += W) write_empty(part_of(A, D, b, L.qj(r), L.hq(r), L.slot), D, lane);
    return;
  }
  // this warp's piece of the split
  const int per = KST ? (L.c1 - L.c0 + W - 1) / W : (L.c1 - L.c0 + W * 4 - 1) / (W * 4) * 4;
  const int w0 = L.c0 + warp * per, w1 = min(L.c1, w0 + per);
  float* mrg = reinterpret_cast<float*>(mrg_smem);
  float* mw = mrg + warp * 8 * MS;
  if constexpr (KST) {
    // query rows, kappa-scaled, channel-major (zero past R.n): row r by warp r % W
    for (int r = warp; r < 8; r += W) {
      const int qj = L.qj(r), hq = L.hq(r);
      const unsigned short* qrow =
          static_cast<const unsigned short*>(A.q) + (static_cast<int64_t>(b * A.Q + qj) * A.Hq + hq) * D;
#pragma unroll
      for (int d = lane; d < D; d += 32) {
        float v = 0.f;
        if (r < R.n) {
          const unsigned short h = __ldg(qrow + d);
          v = (A.bf16 ? __bfloat162float(__ushort_as_bfloat16(h)) : __half2float(__ushort_as_half(h))) * A.kappa;
        }
        qrows[d * 8 + r] = v;
      }
    }
    __syncthreads();
    raw_pieces_by_record<D, N, W>(A, L, mw, qrows, pbuf + warp * 256, kst + warp * 32 * (2 * D + 16), w0, w1);
  } else {
    raw_pieces_by_channel<D, N, W>(A, L, mw, qrows + warp * 40, b, R, w0, w1);
  }
  // ---- merge the warps' pieces, row r by warp r % W
  __syncthreads();
  for (int r = warp; r < R.n; r += W) {
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < W; ++w) M = fmaxf(M, mrg[(w * 8 + r) * MS]);
    float sc[W], Lr = 0.f;
#pragma unroll
    for (int w = 0; w < W; ++w) {
      sc[w] = M == -INFINITY ? 0.f : exp2f(mrg[(w * 8 + r) * MS] - M);
      Lr = fmaf(mrg[(w * 8 + r) * MS + 1], sc[w], Lr);
    }
    float* part = part_of(A, D, b, L.qj(r), L.hq(r), L.slot);
#pragma unroll
    for (int j = lane; j < D; j += 32) {
      float a = 0.f;
#pragma unroll
      for (int w = 0; w < W; ++w) a = fmaf(mrg[(w * 8 + r) * MS + 4 + j], sc[w], a);
      part[4 + j] = a;
    }
    if (lane == 0) {
      part[0] = M;
      part[1] = Lr;
    }
  }
  __syncthreads();  // the scratch and the query rows are read before the next item writes them
}

// Resident CTAs per SM the kernel is compiled for: 3 x 4 warps at head_dim
// 128 (168 registers); 4 x 2 warps at 256 (a warp pair, up to 255 registers:
// at 5 CTAs the pair's 204 registers spill).
#ifndef KVARN_DECODE_MIN_CTAS_256
#define KVARN_DECODE_MIN_CTAS_256 4
#endif
// The affine codec keeps a score accumulator per channel group and builds
// its value weights per group: 2 CTAs of 4 warps (up to 255 registers; at 3
// CTAs it spills).
template <int D, int W, int CD = 0> constexpr int decode_min_ctas() {
  return W == 4 ? (CD == 1 ? 2 : KVARN_DECODE_MIN_CTAS) : D == 256 ? KVARN_DECODE_MIN_CTAS_256 : 1;
}

// ---------------------------------------------------------- work mapping
// The compressed tiles of all (sequence, unit) pairs form one flattened
// list: sequence-major, then unit x = row group * Hkv + KV head, then tile.
// CTA c of C takes the contiguous range [c T / C, (c + 1) T / C) of the T
// tiles (stream-K), so every CTA gets the same number of tiles to within one
// whatever the sequence lengths; a unit cut by range ends gets one partial
// per CTA, merged afterwards.

// Length of sequence b, checked against max_seq_len (flagged and clamped).
__device__ __forceinline__ int checked_len(const DecArgs& A, int b) {
  int len = A.seq_lens[b];
  if (len < 0 || len > A.max_seq_len) {
    set_error(A.err, KVARN_DEVERR_SEQ_LEN);
    len = len < 0 ? 0 : A.max_seq_len;
  }
  return len;
}

// First token past the committed tiles: only tokens up to the first query
// token are accepted, so only the tiles they fill can be committed; of those,
// the raw sink records come first and the newest `recent` accepted tokens
// stay raw. Compressed tiles are [sink_tiles, committed / N).
__device__ __forceinline__ int committed_end(const DecArgs& A, int N, int len) {
  if (A.partial_tiles) return (len + N - 1) / N * N;  // every token is in the pages
  return max(A.sink_tiles * N, (max(0, visible_len(len, A.Q, 0) - A.recent) / N) * N);
}

__device__ __forceinline__ int seq_tiles(const DecArgs& A, int N, int b) {
  return committed_end(A, N, checked_len(A, b)) / N - A.sink_tiles;
}

// Inclusive warp prefix sum.
__device__ __forceinline__ int64_t warp_incl_scan(int64_t v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int64_t y = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += y;
  }
  return v;
}

// Flattened tiles of sequences [0, b_end) (every lane of the warp returns it).
__device__ __forceinline__ int64_t tiles_before(const DecArgs& A, int N, int b_end) {
  const int lane = threadIdx.x & 31;
  int64_t base = 0;
  for (int b0 = 0; b0 < b_end; b0 += 32) {
    const int bb = b0 + lane;
    const int64_t n = bb < b_end ? static_cast<int64_t>(seq_tiles(A, N, bb)) * A.X : 0;
    base += __shfl_sync(0xffffffffu, warp_incl_scan(n), 31);
  }
  return base;
}

struct TilePos {
  int b, x, tile, n;  // sequence, unit, tile within the unit's compressed tiles, the unit's tiles
  int64_t u0;         // the unit's first flattened tile
};

// Position of flattened tile `cur` (< the total); warp-cooperative.
__device__ __forceinline__ TilePos locate_tile(const DecArgs& A, int N, int64_t cur) {
  const int lane = threadIdx.x & 31;
  int64_t base = 0;
  TilePos P{-1, 0, 0, 0, 0};
  for (int b0 = 0; b0 < A.num_seqs; b0 += 32) {
    const int bb = b0 + lane;
    const int n = bb < A.num_seqs ? seq_tiles(A, N, bb) : 0;
    const int64_t incl = warp_incl_scan(static_cast<int64_t>(n) * A.X);
    const unsigned hit = __ballot_sync(0xffffffffu, base + incl > cur);
    if (hit) {
      const int l = __ffs(hit) - 1;
      P.b = b0 + l;
      P.n = __shfl_sync(0xffffffffu, n, l);
      const int64_t before = base + __shfl_sync(0xffffffffu, incl, l) - static_cast<int64_t>(P.n) * A.X;
      const int64_t within = cur - before;
      P.x = static_cast<int>(within / P.n);
      P.tile = static_cast<int>(within % P.n);
      P.u0 = before + static_cast<int64_t>(P.x) * P.n;
      return P;
    }
    base += __shfl_sync(0xffffffffu, incl, 31);
  }
  return P;
}

// CTA ranges are cut on multiples of g tiles (the tiles a CTA has in
// flight), so that a segment inside a range splits evenly over the warps
// whenever the unit lengths are multiples of g: with T tiles in G =
// ceil(T / g) groups, CTA c takes groups [c G / C, (c + 1) G / C).
__device__ __forceinline__ int64_t cta_range_start(int c, int C, int64_t total, int g) {
  const int64_t G = (total + g - 1) / g;
  return min(total, static_cast<int64_t>(g) * (c * G / C));
}

// The CTA whose range holds flattened tile t.
__device__ __forceinline__ int cta_of_tile(int64_t t, int C, int64_t total, int g) {
  const int64_t G = (total + g - 1) / g;
  return static_cast<int>(((t / g + 1) * C - 1) / G);
}

// ------------------------------------------------------------ one segment
// Tiles [t0, t1) of unit x of sequence b: rotated query rows, the tile loop
// of every warp, the merge of the CTA's warps, and the partial into `slot`.
// ph: this warp's mbarrier bookkeeping, which persists across segments:
// K and V slot phases waited (bits 0 and 8) and copies started (bits 16 and
// 24), each counted mod 256 (only parities are read). `dead`: a copy timed
// out earlier; the segment then only writes empty partials. Returns false
// when a copy timed out (in this segment or before).
template <int D, int N, int W, int KB, int VB, int SB, int CD>
__device__ __forceinline__ bool dense_segment(const DecArgs& A, unsigned char* smem, int b, int x, int t0, int t1,
                                              int slot, uint32_t& ph,
                                              bool dead) {
  using S = DecShape<D, N, W, KB, VB, SB, CD>;
  constexpr bool AFF = S::AFF, RAW = S::RAW;
  constexpr bool PLAIN_Q = AFF || RAW;  // original basis, no column scale on the query
  constexpr DensePage PG = S::PG;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g = lane >> 2, t = lane & 3;
  const int kvh = x % A.Hkv;
  const RowMap R(A, x / A.Hkv);

  constexpr int HV = S::HV, UNITS = S::UNITS;
  const int half = HV == 2 ? (warp & 1) : 0, unit = warp / HV;
  const bool leader = half == 0;  // writes the unit's results
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S::OFF_BARS);
  float* qrot = reinterpret_cast<float*>(smem + S::OFF_QROT);
  float* xbuf = reinterpret_cast<float*>(smem + S::OFF_XBUF);
  unsigned char* kslot = smem + unit * S::WARP_SMEM;
  unsigned char* vslot = kslot + S::KSLOT;
  uint64_t* barK = bars + 2 * unit;
  uint64_t* barV = barK + 1;
  // the two warps of a unit meet at named barrier 1 + unit
  auto pair_sync = [&]() {
    if constexpr (HV == 2 && UNITS == 1) asm volatile("bar.sync 1, 64;" ::: "memory");
    else if constexpr (HV == 2) asm volatile("bar.sync %0, 64;" ::"r"(1 + unit) : "memory");
  };

  const int first = t0 + unit;
  const int n_my = !dead && first < t1 ? (t1 - first + UNITS - 1) / UNITS : 0;
  const int32_t* bt = A.bt + static_cast<int64_t>(b) * A.bt_stride;
  // physical page `lane` (lanes < PPT) of this unit's i-th tile; the load is
  // issued a tile ahead and checked only where the copy needs it, so that
  // no instruction waits on it early
  // uncompressed pages: the sequence's tokens, the last tile partial
  const int len_b = RAW ? checked_len(A, b) : 0;
  auto tile_valid = [&](int i) -> int { return RAW ? len_b - (first + i * UNITS) * N : N; };
  auto page_load = [&](int i) -> int {
    if (RAW && lane * kPageTokens >= tile_valid(i)) return -1;  // past the sequence: not loaded
    return lane < S::PPT ? bt[(first + i * UNITS) * S::PPT + lane] : 0;
  };
  auto page_check = [&](int phys) -> int {
    if (RAW && phys == -1) return -1;
    if (phys < 0 || phys >= A.num_pages) {
      set_error(A.err, KVARN_DEVERR_PAGE_RANGE);
      phys = 0;
    }
    return phys;
  };
  auto page_at = [&](int phys) { return A.cache + (static_cast<int64_t>(phys) * A.Hkv + kvh) * S::PB; };
  // The unit's HV warps copy the tile's page parts into the slot 16 bytes a
  // thread at a time (cp.async on the load/store pipe: sixteen bulk copies
  // a tile serialised on the SM's copy unit cost a sixth of the tile loop);
  // each thread then arrives on the slot's barrier once its copies land.
  // Page p's physical id sits in lane p (page ids are read by lanes < PPT).
  // Byte `off` of page p's part (part size P, first box Sp) in its slot: per
  // group of four pages, the four first boxes, then the four second boxes.
  auto part_at = [](const unsigned char* slot, int p, int off, int P, int Sp) -> const unsigned char* {
    if constexpr (S::GATHER) {
      const unsigned char* grp = slot + (p / 4) * 4 * P;
      return off < Sp ? grp + (p % 4) * Sp + off : grp + 4 * Sp + (p % 4) * (P - Sp) + (off - Sp);
    } else {
      return slot + p * P + off;
    }
  };
  auto kp = [&](int p, int off) { return part_at(kslot, p, off, S::KP, S::KS); };
  auto vp = [&](int p, int off) { return part_at(vslot, p, off, S::VP, S::VS); };
  auto issue_part = [&](int phys, unsigned char* slot, int part_off, int part_bytes, int box1, uint64_t* bar,
                        const CUtensorMap* tm, const CUtensorMap* tm2) {
    if constexpr (S::GATHER) {
      // one TMA gather per four pages (two for a split part), from the
      // unit's lane 0 (rows phys * Hkv + kvh)
      fence_proxy_async_smem();  // the warp's reads of the slot precede the async writes
      int row[S::PPT];
#pragma unroll
      for (int p = 0; p < S::PPT; ++p) row[p] = __shfl_sync(0xffffffffu, phys, p) * A.Hkv + kvh;
      __syncwarp();
      if (leader && lane == 0) {
        mbar_arrive_expect_tx(bar, S::PPT * part_bytes + A.withhold);
#pragma unroll
        for (int q4 = 0; q4 < S::PPT / 4; ++q4) {
          unsigned char* dst = slot + 4 * q4 * part_bytes;
          tma_gather4(dst, tm, part_off / 8, row[4 * q4], row[4 * q4 + 1], row[4 * q4 + 2], row[4 * q4 + 3], bar);
          if (box1 < part_bytes)
            tma_gather4(dst + 4 * box1, tm2, (part_off + box1) / 8, row[4 * q4], row[4 * q4 + 1], row[4 * q4 + 2],
                        row[4 * q4 + 3], bar);
        }
      }
    } else {
      __syncwarp();  // every lane's reads of the slot precede the copies
      const int tid = half * 32 + lane;
#pragma unroll
      for (int p = 0; p < S::PPT; ++p) {
        const int pid = __shfl_sync(0xffffffffu, phys, p);
        if (RAW && pid < 0) continue;  // a page past the sequence is not read
        const unsigned char* src = page_at(pid) + part_off;
        unsigned char* dst = slot + p * part_bytes;
#pragma unroll
        for (int c = tid; c < part_bytes / 16; c += 32 * HV) cp_async16(dst + 16 * c, src + 16 * c);
      }
      if (A.withhold == 0 || tid != 0) cp_async_arrive(bar);  // a withheld arrival: the phase never completes
    }
  };
  auto issue_k = [&](int phys) {
    ph += 1u << 16;
    issue_part(phys, kslot, 0, S::KP, S::KS, barK, &A.tmk, &A.tmk2);
  };
  auto issue_v = [&](int phys) {
    ph += 1u << 24;
    issue_part(phys, vslot, S::KP, S::VP, S::VS, barV, &A.tmv, &A.tmv2);
  };

  if (n_my > 0) {
    const int phys = page_check(page_load(0));
    issue_k(phys);
    issue_v(phys);
  }

  // ---- rotated, scaled query rows of the row group (unused rows are zero)
  for (int h = warp; h < 8; h += W) {
    constexpr int E = D / 32;
    float v[E];
    if (h < R.n) {
      const int hq = kvh * A.G + R.head(A, h), j = R.query(A, h);
      const int64_t qoff = (static_cast<int64_t>(b * A.Q + j) * A.Hq + hq) * D + lane * E;
      load_vec_rt<E>(static_cast<const char*>(A.q) + 2 * qoff, A.bf16, v);
      if constexpr (!PLAIN_Q) warp_fwht<E>(v);  // the affine and fp16 pages are in the original basis
      const float sc = PLAIN_Q ? A.kappa : A.kappa / sqrtf(static_cast<float>(D));
#pragma unroll
      for (int e = 0; e < E; ++e) v[e] *= sc;
    } else {
#pragma unroll
      for (int e = 0; e < E; ++e) v[e] = 0.f;
    }
#pragma unroll
    for (int e = 0; e < E; ++e) {
      const int ch = lane * E + e, w = ch % 16;
      qrot[q_frag(ch / 16, h, (w % 8) / 2) + (w % 2) + 2 * (w / 8)] = v[e];
    }
  }
  __syncthreads();

  constexpr int KCW = S::KC / HV, NCW = S::NC / HV;  // this warp's k-chunks and channel blocks
  float m = -INFINITY, lsum = 0.f;
  float2 acc[NCW];
#pragma unroll
  for (int nc = 0; nc < NCW; ++nc) acc[nc] = f2(0.f);
  float* xmine = xbuf + (unit * 2 + half) * 32 * S::XS;
  const float* xother = xbuf + (unit * 2 + (half ^ 1)) * 32 * S::XS;

  bool timed_out = false;
  for (int i = 0; i < n_my; ++i) {
    // the next tile's page ids, loaded a tile ahead of their copies
    int phys_next = i + 1 < n_my ? page_load(i + 1) : 0;
    // a warp of a pair that gives up on a copy tells its partner at the next
    // pair barrier and both leave together
    bool late = !mbar_wait_bounded(barK, ph & 1, A.wait_limit);
    ph += 1u;
    if constexpr (HV == 1) {
      if (late) {
        timed_out = true;
        break;
      }
    }
    // -- q~ = q' * c_K as fp16 hi/lo A fragments (this warp's channels);
    //    the affine pages take q' as it is
    uint32_t Aq[KCW][4];
    float2 qs2[KCW];
#pragma unroll
    for (int kcl = 0; kcl < KCW; ++kcl) {
      const int kc = half * KCW + kcl;
      const int ch0 = 16 * kc + 2 * t;
      const float4 qv = *reinterpret_cast<const float4*>(qrot + q_frag(kc, g, t));
      float2 x01 = make_float2(qv.x, qv.y), x89 = make_float2(qv.z, qv.w);
      if constexpr (!PLAIN_Q) {
        const unsigned char* cp = kp(ch0 / S::CPP, PG.k_col() + (ch0 % S::CPP) * SB);
        x01 = f2mul(x01, load_scale2<SB>(cp));
        x89 = f2mul(x89, load_scale2<SB>(cp + 8 * SB));
      }
      qs2[kcl] = f2add(x01, x89);
      split_hi_lo2(x01, Aq[kcl][0], Aq[kcl][1]);
      split_hi_lo2(x89, Aq[kcl][2], Aq[kcl][3]);
    }
    float2 qsum = f2(0.f);
    float qg[S::GR];  // affine: sum of the query over each 64-channel group
    if constexpr (AFF) {
#pragma unroll
      for (int gr = 0; gr < S::GR; ++gr) {
        float2 a = qs2[4 * gr];
#pragma unroll
        for (int k = 1; k < 4; ++k) a = f2add(a, qs2[4 * gr + k]);
        qg[gr] = warp_sum_xor(a.x + a.y, 1, 4);
      }
    } else if constexpr (!RAW) {
      const float2 q2 = tree_reduce(qs2, [](float2 a, float2 b) { return f2add(a, b); });
      qsum = f2(warp_sum_xor(q2.x + q2.y, 1, 4));
    }
    const int valid = tile_valid(i);  // tokens of this tile below the length (N but for fp16 pages)

    // -- S = q~ . (kappa_K codes)^T, two pages (four 8-token blocks) at a
    //    time so that four independent accumulator chains hide the mma
    //    latency. Per group of four k-chunks a lane's fragments (2 kc + e,
    //    e the token block) are KW consecutive words of each code plane.
    float2 s[S::NB];
    // the affine scores keep one accumulator per 64-channel group (one group
    // of four k-chunks), each scaled by its own per-token scale
    constexpr int DG = AFF ? S::KCH : 1;
    if constexpr (RAW) {
      // the fp16 rows: row 8 e + g of a page, lane chunk t holding channels
      // 16 kc + {2t, 2t + 1, 2t + 8, 2t + 9} in k-chunk order (8 bytes each)
#pragma unroll
      for (int p = 0; p < S::PPT; ++p) {
        float d[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const unsigned char* kr = kp(p, (8 * e + g) * 2 * D + t * (D / 2) + 8 * half * KCW);
#pragma unroll
          for (int j = 0; j < KCW / 2; ++j) {
            const uint4 kw = *reinterpret_cast<const uint4*>(kr + 16 * j);
            mma_f16(d[e], Aq[2 * j][0], Aq[2 * j][1], Aq[2 * j][2], Aq[2 * j][3], kw.x, kw.y);
            mma_f16(d[e], Aq[2 * j + 1][0], Aq[2 * j + 1][1], Aq[2 * j + 1][2], Aq[2 * j + 1][3], kw.z, kw.w);
          }
        }
#pragma unroll
        for (int e = 0; e < 2; ++e) s[2 * p + e] = f2add(make_float2(d[e][0], d[e][1]), make_float2(d[e][2], d[e][3]));
      }
    }
#pragma unroll
    for (int p0 = 0; p0 < S::PPT && !RAW; p0 += 2) {
      float d[DG][2][2][4];
#pragma unroll
      for (int dg = 0; dg < DG; ++dg)
#pragma unroll
        for (int pi = 0; pi < 2; ++pi)
#pragma unroll
          for (int e = 0; e < 2; ++e) d[dg][pi][e][0] = d[dg][pi][e][1] = d[dg][pi][e][2] = d[dg][pi][e][3] = 0.f;
#pragma unroll
      for (int chl = 0; chl < S::KCH / HV; ++chl) {
        const int ch = half * (S::KCH / HV) + chl;
        uint32_t x0[2][S::KW0], x1[2][S::KW1 ? S::KW1 : 1];
#pragma unroll
        for (int pi = 0; pi < 2; ++pi) {
          load_words<S::KW0>(kp(p0 + pi, 4 * S::KU0 * (32 * ((ch * S::KW0) / S::KU0) + lane) + 4 * ((ch * S::KW0) % S::KU0)),
                             x0[pi]);
          if constexpr (S::KW1 != 0)
            load_words<S::KW1>(kp(p0 + pi, S::KR1 + 4 * S::KU1 * (32 * ((ch * S::KW1) / S::KU1) + lane) +
                                               4 * ((ch * S::KW1) % S::KU1)),
                               x1[pi]);
        }
        static_for<0, 8>([&](auto fgc) {
          constexpr int fg = decltype(fgc)::value;  // fragment 2 w4 + e of the group
          const int kc = 4 * chl + fg / 2;          // this warp's k-chunk
#pragma unroll
          for (int pi = 0; pi < 2; ++pi) {
            uint32_t b0, b1;
            code_pair<KB, fg % S::KF0, fg % S::KF1>(x0[pi][fg / S::KF0], x1[pi][(fg / S::KF1) % (S::KW1 ? S::KW1 : 1)],
                                                    b0, b1);
            mma_f16(d[AFF ? chl : 0][pi][fg % 2], Aq[kc][0], Aq[kc][1], Aq[kc][2], Aq[kc][3], b0, b1);
          }
        });
      }
      if constexpr (AFF) {
        // s = sum over groups of kappa_K sc_g S_g + (of_g + center sc_g) Q_g,
        // the records of tokens 8 e + 2 t and + 1 (scales, then offsets)
        static_assert(S::GR == 2, "two groups per token record");
#pragma unroll
        for (int pi = 0; pi < 2; ++pi)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const uint4 rec = *reinterpret_cast<const uint4*>(kp(p0 + pi, S::AG.k_sc() + 8 * (8 * e + 2 * t)));
            const float2 sa = __half22float2(u32_as_h2(rec.x)), oa = __half22float2(u32_as_h2(rec.y));
            const float2 sb = __half22float2(u32_as_h2(rec.z)), ob = __half22float2(u32_as_h2(rec.w));
            float2 v = f2(0.f);
#pragma unroll
            for (int gr = 0; gr < 2; ++gr) {
              const float2 sc = gr ? make_float2(sa.y, sb.y) : make_float2(sa.x, sb.x);
              const float2 of = gr ? make_float2(oa.y, ob.y) : make_float2(oa.x, ob.x);
              const float2 Sg = f2add(make_float2(d[gr][pi][e][0], d[gr][pi][e][1]),
                                      make_float2(d[gr][pi][e][2], d[gr][pi][e][3]));
              v = f2fma(f2mul(sc, f2(S::KINV)), Sg, v);
              v = f2fma(f2fma(f2(S::KCENTER), sc, of), f2(qg[gr]), v);
            }
            s[2 * (p0 + pi) + e] = v;
          }
      } else {
#pragma unroll
        for (int pi = 0; pi < 2; ++pi)
#pragma unroll
          for (int e = 0; e < 2; ++e)
            s[2 * (p0 + pi) + e] =
                f2add(make_float2(d[0][pi][e][0], d[0][pi][e][1]), make_float2(d[0][pi][e][2], d[0][pi][e][3]));
      }
    }

    // -- row-scale fold (linear, so a warp of a pair folds its partial
    //    scores with its own sum of q~ and the pair adds them in a fixed
    //    order, leaving both with the same scores), then the online softmax
    //    in base 2. The K slot is read for the last time here.
    if constexpr (!PLAIN_Q) {
#pragma unroll
      for (int nb = 0; nb < S::NB; ++nb) {
        const int idx = (nb & 1) * 8 + 2 * t;
        const float2 ka = load_scale2<SB>(kp(nb >> 1, PG.k_a() + idx * SB));
        const float2 kb = load_scale2<SB>(kp(nb >> 1, PG.k_b() + idx * SB));
        const float2 kb_c = S::KCENTER != 0.f ? f2fma(f2(S::KCENTER), ka, kb) : kb;
        s[nb] = f2fma(f2mul(ka, f2(S::KINV)), s[nb], f2mul(kb_c, qsum));
      }
    }
    if constexpr (HV == 2) {
#pragma unroll
      for (int nb = 0; nb < S::NB; ++nb) {
        xmine[(2 * nb) * 32 + lane] = s[nb].x;
        xmine[(2 * nb + 1) * 32 + lane] = s[nb].y;
      }
      xmine[(S::XS - 2) * 32 + lane] = late ? 1.f : 0.f;
      pair_sync();
      late = late || xother[(S::XS - 2) * 32 + lane] != 0.f;
      late = __any_sync(0xffffffffu, late);
#pragma unroll
      for (int nb = 0; nb < S::NB; ++nb) {
        const float2 o = make_float2(xother[(2 * nb) * 32 + lane], xother[(2 * nb + 1) * 32 + lane]);
        s[nb] = half ? f2add(o, s[nb]) : f2add(s[nb], o);
      }
      if (late) {
        timed_out = true;
        break;
      }
    }
    if constexpr (RAW) {  // tokens past the length (a partial last tile) take no weight
#pragma unroll
      for (int nb = 0; nb < S::NB; ++nb) {
        const int tok = 8 * nb + 2 * t;
        s[nb] = make_float2(tok < valid ? s[nb].x : -INFINITY, tok + 1 < valid ? s[nb].y : -INFINITY);
      }
    }
    float mts[S::NB];
#pragma unroll
    for (int nb = 0; nb < S::NB; ++nb) mts[nb] = fmaxf(s[nb].x, s[nb].y);
    float mt = tree_reduce(mts, [](float a, float b) { return fmaxf(a, b); });
    mt = warp_max_xor(mt, 1, 4);
    const float m_new = fmaxf(m, mt);
    const float alpha = fast_exp2(m - m_new);
    float2 ps2[S::NB];
#pragma unroll
    for (int nb = 0; nb < S::NB; ++nb) {
      const float2 z = f2add(s[nb], f2(-m_new));
      s[nb] = make_float2(fast_exp2(z.x), fast_exp2(z.y));
      ps2[nb] = s[nb];
    }
    const float2 pt = tree_reduce(ps2, [](float2 a, float2 b) { return f2add(a, b); });
    lsum = fmaf(lsum, alpha, pt.x + pt.y);
    m = m_new;

    // the K slot is free: start the next tile's K part
    if (i + 1 < n_my) {
      phys_next = page_check(phys_next);
      issue_k(phys_next);
    }

    late = !mbar_wait_bounded(barV, (ph >> 8) & 1, A.wait_limit);
    ph += 1u << 8;
    if constexpr (HV == 1) {
      if (late) {
        timed_out = true;
        break;
      }
    }

    // -- P V: weights p * a_V as hi/lo A fragments, one k16 chunk per page
    //    (affine: p * the group's scale, built per group below)
    uint32_t Ap[S::PPT][4];
    float2 be2[S::PPT];
    float2 beta = f2(0.f);
    if constexpr (RAW) {
#pragma unroll
      for (int pp = 0; pp < S::PPT; ++pp) {
        split_hi_lo2(s[2 * pp], Ap[pp][0], Ap[pp][1]);
        split_hi_lo2(s[2 * pp + 1], Ap[pp][2], Ap[pp][3]);
      }
    } else if constexpr (!AFF) {
#pragma unroll
    for (int pp = 0; pp < S::PPT; ++pp) {
      const float2 va0 = load_scale2<SB>(vp(pp, PG.v_a() - S::KP + (2 * t) * SB));
      const float2 va1 = load_scale2<SB>(vp(pp, PG.v_a() - S::KP + (8 + 2 * t) * SB));
      const float2 vb0 = load_scale2<SB>(vp(pp, PG.v_b() - S::KP + (2 * t) * SB));
      const float2 vb1 = load_scale2<SB>(vp(pp, PG.v_b() - S::KP + (8 + 2 * t) * SB));
      be2[pp] = f2fma(s[2 * pp], S::VCENTER != 0.f ? f2fma(f2(S::VCENTER), va0, vb0) : vb0,
                      f2mul(s[2 * pp + 1], S::VCENTER != 0.f ? f2fma(f2(S::VCENTER), va1, vb1) : vb1));
      split_hi_lo2(f2mul(s[2 * pp], va0), Ap[pp][0], Ap[pp][1]);
      split_hi_lo2(f2mul(s[2 * pp + 1], va1), Ap[pp][2], Ap[pp][3]);
    }
      const float2 bt2 = tree_reduce(be2, [](float2 a, float2 b) { return f2add(a, b); });
      beta = f2(warp_sum_xor(bt2.x + bt2.y, 1, 4));
    }

#pragma unroll
    for (int nc = 0; nc < NCW; ++nc) acc[nc] = f2mul(acc[nc], f2(alpha));
    // channel blocks in groups of eight: the group's fragments are one
    // unit (VW consecutive words) of each code plane
#pragma unroll
    for (int hql = 0; hql < S::VHC / HV; ++hql) {
      const int hq = half * (S::VHC / HV) + hql;
      if constexpr (AFF) {
        // group hq (channels [64 hq, +64)): weights p * sc_hq and the offset
        // term sum p (of_hq + center sc_hq), records of tokens 2t, 2t + 1
        // and 8 + 2t, 9 + 2t of each page
#pragma unroll
        for (int pp = 0; pp < S::PPT; ++pp) {
          const uint4 r0 = *reinterpret_cast<const uint4*>(vp(pp, S::AG.v_sc() + 8 * (2 * t)));
          const uint4 r1 = *reinterpret_cast<const uint4*>(vp(pp, S::AG.v_sc() + 8 * (8 + 2 * t)));
          auto pick = [&](uint32_t a, uint32_t b2) {
            const float2 fa = __half22float2(u32_as_h2(a)), fb = __half22float2(u32_as_h2(b2));
            return hq ? make_float2(fa.y, fb.y) : make_float2(fa.x, fb.x);
          };
          const float2 sc0 = pick(r0.x, r0.z), of0 = pick(r0.y, r0.w);
          const float2 sc1 = pick(r1.x, r1.z), of1 = pick(r1.y, r1.w);
          be2[pp] = f2fma(s[2 * pp], f2fma(f2(S::VCENTER), sc0, of0),
                          f2mul(s[2 * pp + 1], f2fma(f2(S::VCENTER), sc1, of1)));
          split_hi_lo2(f2mul(s[2 * pp], sc0), Ap[pp][0], Ap[pp][1]);
          split_hi_lo2(f2mul(s[2 * pp + 1], sc1), Ap[pp][2], Ap[pp][3]);
        }
        const float2 bt2 = tree_reduce(be2, [](float2 a, float2 b) { return f2add(a, b); });
        beta = f2(warp_sum_xor(bt2.x + bt2.y, 1, 4));
      }
      float u[8][4];
#pragma unroll
      for (int k = 0; k < 8; ++k) u[k][0] = u[k][1] = u[k][2] = u[k][3] = 0.f;
      if constexpr (RAW) {
        // lane chunk 4 g + t of a page's V rows: per 8-channel block nc,
        // channel 8 nc + g at tokens (2t, 2t + 1) then (2t + 8, 2t + 9);
        // rows past the length may hold any bits and are cleared, so that
        // their zero weight never meets an inf or nan
#pragma unroll
        for (int pp = 0; pp < S::PPT; ++pp) {
          const int tb = pp * kPageTokens + 2 * t;
          const uint32_t m01 = (tb < valid ? 0x0000FFFFu : 0u) | (tb + 1 < valid ? 0xFFFF0000u : 0u);
          const uint32_t m89 = (tb + 8 < valid ? 0x0000FFFFu : 0u) | (tb + 9 < valid ? 0xFFFF0000u : 0u);
          const unsigned char* vr = vp(pp, (4 * g + t) * D + 64 * hq);
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const uint4 vw = *reinterpret_cast<const uint4*>(vr + 16 * j);
            mma_f16(u[2 * j], Ap[pp][0], Ap[pp][1], Ap[pp][2], Ap[pp][3], vw.x & m01, vw.y & m89);
            mma_f16(u[2 * j + 1], Ap[pp][0], Ap[pp][1], Ap[pp][2], Ap[pp][3], vw.z & m01, vw.w & m89);
          }
        }
      }
#pragma unroll
      for (int pp = 0; pp < S::PPT && !RAW; ++pp) {
        uint32_t x0[S::VW0], x1[S::VW1 ? S::VW1 : 1];
        load_words<S::VW0>(vp(pp, 4 * S::VW0 * (32 * hq + lane)), x0);
        if constexpr (S::VW1 != 0) load_words<S::VW1>(vp(pp, S::VR1 + 4 * S::VW1 * (32 * hq + lane)), x1);
        static_for<0, 8>([&](auto kc_) {
          constexpr int k = decltype(kc_)::value;
          uint32_t b0, b1;
          code_pair<VB, k % S::VF0, k % S::VF1>(x0[k / S::VF0], x1[(k / S::VF1) % (S::VW1 ? S::VW1 : 1)], b0, b1);
          mma_f16(u[k], Ap[pp][0], Ap[pp][1], Ap[pp][2], Ap[pp][3], b0, b1);
        });
      }
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const int nc = 8 * hq + k, ncl = 8 * hql + k;
        const int ch = 8 * nc + 2 * t;
        const float2 uk = f2add(make_float2(u[k][0], u[k][1]), make_float2(u[k][2], u[k][3]));
        if constexpr (RAW) {
          acc[ncl] = f2add(uk, acc[ncl]);
        } else if constexpr (AFF) {
          acc[ncl] = f2add(f2fma(uk, f2(S::VINV), beta), acc[ncl]);
        } else {
          const float2 cv = load_scale2<SB>(vp(ch / S::CPP, PG.v_col() - S::KP + (ch % S::CPP) * SB));
          acc[ncl] = f2fma(cv, f2fma(uk, f2(S::VINV), beta), acc[ncl]);
        }
      }
    }
    if constexpr (HV == 2) {  // both warps are done with the V slot
      xmine[(S::XS - 1) * 32 + lane] = late ? 1.f : 0.f;
      pair_sync();
      late = __any_sync(0xffffffffu, late || xother[(S::XS - 1) * 32 + lane] != 0.f);
      if (late) {
        timed_out = true;
        break;
      }
    }
    if (i + 1 < n_my) issue_v(phys_next);
  }
  if (timed_out) {
    if (leader && lane == 0) set_error(A.err, KVARN_DEVERR_TIMEOUT);
    cp_async_wait_all();  // this thread's copies have landed (a hardware wait, like a load's)
    // wait (bounded) for the last copy of each slot this warp started (a
    // parity whose phase precedes the barrier's first completes at once); no
    // copy is started after a time-out
    mbar_wait_bounded(barK, ((ph >> 16) - 1) & 1, 100000000LL);
    mbar_wait_bounded(barV, ((ph >> 24) - 1) & 1, 100000000LL);
  }
  lsum = warp_sum_xor(lsum, 1, 4);

  // ---- merge the units of the CTA (scratch aliases the slots)
  const bool any_late = __syncthreads_or(timed_out);
  float* mrg = reinterpret_cast<float*>(smem);
  constexpr int MS = merge_stride<D>();
  float* mw = mrg + unit * 8 * MS;
  if (t == 0 && leader) {
    mw[g * MS] = n_my > 0 ? m : -INFINITY;
    mw[g * MS + 1] = n_my > 0 ? lsum : 0.f;
  }
#pragma unroll
  for (int ncl = 0; ncl < NCW; ++ncl) {
    const int nc = half * NCW + ncl;
    *reinterpret_cast<float2*>(mw + g * MS + 4 + 8 * nc + 2 * t) = acc[ncl];
  }
  __syncthreads();
  for (int idx = threadIdx.x; idx < R.n * D; idx += W * 32) {
    const int gg = idx / D, j = idx % D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < UNITS; ++w) M = fmaxf(M, mrg[(w * 8 + gg) * MS]);
    float a = 0.f, L = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < UNITS; ++w) {
        const float* r = mrg + (w * 8 + gg) * MS;
        const float sc = exp2f(r[0] - M);
        a = fmaf(r[4 + j], sc, a);
        L = fmaf(r[1], sc, L);
      }
    }
    float* part = part_of(A, D, b, R.query(A, gg), kvh * A.G + R.head(A, gg), slot);
    part[4 + j] = a;
    if (j == 0) {
      part[0] = M;
      part[1] = L;
    }
  }
  // the scratch is read before the next segment's copies land in the slots
  __syncthreads();
  return !any_late;
}

template <int D, int N, int W, int KB = 4, int VB = 2, int SB = 4, int CD = kCodecKvarn>
__global__ void __launch_bounds__(W * 32, (decode_min_ctas<D, W, CD>())) decode_dense_kernel(const __grid_constant__ DecArgs A) {
  using S = DecShape<D, N, W, KB, VB, SB, CD>;
  extern __shared__ __align__(128) unsigned char smem[];
  pdl_launch_dependents();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  {
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S::OFF_BARS);
    if (warp % S::HV == 0 && lane == 0) {
      // one arrival per copying thread (cp.async), or lane 0's (TMA gathers)
      mbar_init(bars + 2 * (warp / S::HV), S::GATHER ? 1 : 32 * S::HV);
      mbar_init(bars + 2 * (warp / S::HV) + 1, S::GATHER ? 1 : 32 * S::HV);
    }
    fence_mbar_init();
  }
  // launched as a programmatic dependent of the kernel before it (a commit,
  // or whatever wrote the queries, lengths or tails): nothing in global
  // memory is read before that kernel has completed
  pdl_wait_primary();

  // ---- raw records: items r = blockIdx.x, + gridDim.x, ... of (sequence,
  //      unit, raw chunk)
  const int64_t units = static_cast<int64_t>(A.num_seqs) * A.X;
  for (int64_t r = blockIdx.x; r < units * A.raw_splits; r += gridDim.x) {
    const int chunk = static_cast<int>(r % A.raw_splits);
    const int64_t u = r / A.raw_splits;
    const int b = static_cast<int>(u / A.X), x = static_cast<int>(u % A.X);
    const int len = checked_len(A, b);
    if constexpr (S::RAW) {
      // the uncompressed pages hold every token: the raw splits stay empty
      const RowMap R(A, x / A.Hkv);
      for (int rr = warp; rr < R.n; rr += W)
        write_empty(part_of(A, D, b, R.query(A, rr), (x % A.Hkv) * A.G + R.head(A, rr), A.tile_slots + chunk), D,
                    lane);
    } else {
      tail_partials<D, N, W, (S::RAW_KST > 0)>(A, smem + S::OFF_RAW_MRG, reinterpret_cast<float*>(smem + S::OFF_QROT),
                                               reinterpret_cast<float*>(smem + S::OFF_RAW_PB), smem + S::OFF_RAW_KST, b,
                                               x % A.Hkv, RowMap(A, x / A.Hkv), len, A.sink_tiles * N,
                                               committed_end(A, N, len), chunk);
    }
  }

  const int64_t total = tiles_before(A, N, A.num_seqs);
  const int64_t by_tiles = total / A.min_tiles > 1 ? total / A.min_tiles : 1;
  const int C = static_cast<int>(by_tiles < gridDim.x ? by_tiles : gridDim.x);

  // ---- tile-partial counts of units u = blockIdx.x, + gridDim.x, ...
  if (warp == 0) {
    for (int64_t u = blockIdx.x; u < units; u += gridDim.x) {
      const int b = static_cast<int>(u / A.X), x = static_cast<int>(u % A.X);
      const int n = seq_tiles(A, N, b);
      int count = 0;
      if (n > 0) {
        const int64_t u0 = tiles_before(A, N, b) + static_cast<int64_t>(x) * n;
        count = cta_of_tile(u0 + n - 1, C, total, S::UNITS) - cta_of_tile(u0, C, total, S::UNITS) + 1;
      }
      const RowMap R(A, x / A.Hkv);
      if (lane < R.n)
        A.counts[(b * A.Q + R.query(A, lane)) * A.Hq + (x % A.Hkv) * A.G + R.head(A, lane)] = count;
    }
  }
  __syncthreads();  // mbarrier initialisation visible to every warp
  if (total == 0 || static_cast<int>(blockIdx.x) >= C) return;

  // ---- this CTA's tiles, one segment per unit they touch. The position is
  //      kept in shared memory (no register holds it across a segment),
  //      double-buffered: the next position is written to the entry nobody
  //      reads in this pass, and read after the segment's closing barrier.
  __shared__ int64_t pos[3];  // current tile (two entries), end of the range
  if (threadIdx.x == 0) {
    pos[0] = cta_range_start(blockIdx.x, C, total, S::UNITS);
    pos[2] = cta_range_start(blockIdx.x + 1, C, total, S::UNITS);
  }
  __syncthreads();
  uint32_t ph = 0;
  bool dead = false;
  for (int k = 0;; k ^= 1) {
    const int64_t cur = pos[k], stop = pos[2];
    if (cur >= stop) break;
    const TilePos P = locate_tile(A, N, cur);
    if (P.b < 0) break;  // unreachable: cur < total
    const int64_t seg_end = min(stop, P.u0 + P.n);
    const int slot = static_cast<int>(blockIdx.x) - cta_of_tile(P.u0, C, total, S::UNITS);
    const int t0 = A.sink_tiles + P.tile;
    const int t1 = t0 + static_cast<int>(seg_end - cur);
    if (threadIdx.x == 0) pos[k ^ 1] = seg_end;
    dead = !dense_segment<D, N, W, KB, VB, SB, CD>(A, smem, P.b, P.x, t0, t1, slot, ph, dead) || dead;
  }
}

template <int D, int N, int W, int KB, int VB, int SB, int CD = kCodecKvarn>
cudaError_t run_dense(const DecArgs& A, int ctas, cudaStream_t st) {
  using S = DecShape<D, N, W, KB, VB, SB, CD>;
  auto kern = decode_dense_kernel<D, N, W, KB, VB, SB, CD>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, S::SMEM);
  if (e != cudaSuccess) return e;
  // a programmatic dependent of the kernel before it on the stream: the
  // grid is scheduled while that kernel's last CTAs run and waits for its
  // completion before the first global read
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(ctas);
  cfg.blockDim = dim3(W * 32);
  cfg.dynamicSmemBytes = S::SMEM;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, A);
}

// CTAs of one decode kernel resident per SM (registers and shared memory).
template <int D, int N, int W, int KB, int VB, int SB, int CD = kCodecKvarn>
int resident_dense() {
  using S = DecShape<D, N, W, KB, VB, SB, CD>;
  auto kern = decode_dense_kernel<D, N, W, KB, VB, SB, CD>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, S::SMEM) != cudaSuccess) return 1;
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, W * 32, S::SMEM) != cudaSuccess || n < 1) return 1;
  return n;
}

// Warps per CTA of the head_dim-128 decode of these widths: 4, or 2 where a
// 4-warp CTA's page slots would take more than half an SM's shared memory
// (8-bit codes at 128-token tiles: 137 KB, one CTA of 4 warps per SM; 2-warp
// CTAs fit three to an SM).
template <int D, int N, int KB, int VB, int SB, int CD = kCodecKvarn>
constexpr int width_warps() {
  return DecShape<D, N, 4, KB, VB, SB, CD>::SMEM > 116 * 1024 ? 2 : 4;
}

// The decode kernels of one (K width, V width, scale bytes) combination and
// their residency (which sizes the persistent grid: the page parts of wider
// codes take more shared memory); each combination is compiled in its own
// translation unit.
template <int KB, int VB, int SB>
cudaError_t run_dense_widths(const DecArgs& A, int D, int N, bool bf16, int ctas, cudaStream_t st);
template <int KB, int VB, int SB>
int resident_widths(int D, int N);

#define KVARN_DECLARE_WIDTHS(KB, VB, SB)                                                             \
  template <>                                                                                       \
  cudaError_t run_dense_widths<KB, VB, SB>(const DecArgs& A, int D, int N, bool bf16, int ctas,    \
                                           cudaStream_t st);                                        \
  template <>                                                                                       \
  int resident_widths<KB, VB, SB>(int D, int N);
#define KVARN_DECLARE_WIDTHS_S16(KB, VB) KVARN_DECLARE_WIDTHS(KB, VB, 2)
#define KVARN_DECLARE_WIDTHS_S32(KB, VB) KVARN_DECLARE_WIDTHS(KB, VB, 4)
KVARN_WIDTH_PAIRS(KVARN_DECLARE_WIDTHS_S16)
KVARN_WIDTH_PAIRS_S32(KVARN_DECLARE_WIDTHS_S32)
#undef KVARN_DECLARE_WIDTHS_S16
#undef KVARN_DECLARE_WIDTHS_S32
#undef KVARN_DECLARE_WIDTHS

// The same at head_dim 256 (warp pairs share a tile).
template <int KB, int VB, int SB>
cudaError_t run_dense_widths256(const DecArgs& A, int N, bool bf16, int ctas, cudaStream_t st);
template <int KB, int VB, int SB>
int resident_widths256(int N);

#define KVARN_DECLARE_WIDTHS_256(KB, VB)                                                           \
  template <>                                                                                     \
  cudaError_t run_dense_widths256<KB, VB, 2>(const DecArgs& A, int N, bool bf16, int ctas, cudaStream_t st); \
  template <>                                                                                     \
  int resident_widths256<KB, VB, 2>(int N);
KVARN_WIDTH_PAIRS_256(KVARN_DECLARE_WIDTHS_256)
#undef KVARN_DECLARE_WIDTHS_256

// The decode over uncompressed fp16 pages (the same kernel with no codec;
// 32-token tiles, 4 warps at head_dim 128, warp pairs at 256), compiled in
// kvarn_fp16.cu.
template <int D>
cudaError_t run_raw(const DecArgs& A, int ctas, cudaStream_t st);
template <int D>
int resident_raw();

// The affine comparison decode of one code width (keys and values alike,
// head_dim 128, 128-token tiles), compiled in kvarn_affine_dec.cu.
#define KVARN_AFFINE_WIDTHS(X) X(2) X(3) X(4) X(6) X(8)
template <int KB>
cudaError_t run_affine_widths(const DecArgs& A, bool bf16, int ctas, cudaStream_t st);
template <int KB>
int resident_affine();
#define KVARN_DECLARE_AFFINE(K)                                                                  \
  template <>                                                                                   \
  cudaError_t run_affine_widths<K>(const DecArgs& A, bool bf16, int ctas, cudaStream_t st);     \
  template <>                                                                                   \
  int resident_affine<K>();
KVARN_AFFINE_WIDTHS(KVARN_DECLARE_AFFINE)
#undef KVARN_DECLARE_AFFINE

#define KVARN_DECODE_WIDTHS(KB, VB, SB)                                                                   \
  template <>                                                                                           \
  cudaError_t run_dense_widths<KB, VB, SB>(const DecArgs& A, int D, int N, bool /*bf16*/, int ctas,    \
                                           cudaStream_t st) {                                           \
    constexpr int W1 = width_warps<128, 128, KB, VB, SB>(), W2 = width_warps<128, 64, KB, VB, SB>();    \
    if (D == 128 && N == 128)                                                                           \
      return run_dense<128, 128, W1, KB, VB, SB>(A, ctas, st);                       \
    if (D == 128 && N == 64)                                                                            \
      return run_dense<128, 64, W2, KB, VB, SB>(A, ctas, st);                        \
    return cudaErrorInvalidValue;                                                                       \
  }                                                                                                     \
  template <>                                                                                           \
  int resident_widths<KB, VB, SB>(int D, int N) {                                                       \
    if (D == 128 && N == 128) return resident_dense<128, 128, width_warps<128, 128, KB, VB, SB>(), KB, VB, SB>(); \
    if (D == 128 && N == 64) return resident_dense<128, 64, width_warps<128, 64, KB, VB, SB>(), KB, VB, SB>();   \
    return 1;                                                                                           \
  }

#define KVARN_DECODE_WIDTHS_256(KB, VB)                                                                \
  template <>                                                                                          \
  cudaError_t run_dense_widths256<KB, VB, 2>(const DecArgs& A, int N, bool /*bf16*/, int ctas, cudaStream_t st) { \
    if (N == 128)                                                                                      \
      return run_dense<256, 128, 2, KB, VB, 2>(A, ctas, st);                            \
    if (N == 64)                                                                                       \
      return run_dense<256, 64, 2, KB, VB, 2>(A, ctas, st);                             \
    return cudaErrorInvalidValue;                                                                      \
  }                                                                                                    \
  template <>                                                                                          \
  int resident_widths256<KB, VB, 2>(int N) {                                                           \
    return N == 128 ? resident_dense<256, 128, 2, KB, VB, 2>()                                 \
                    : resident_dense<256, 64, 2, KB, VB, 2>();                                 \
  }

}  // namespace kvarn

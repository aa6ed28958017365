// KVarN decode attention: split planning and launch (kernels in
// kvarn_decode_kernel.cuh; the k4v2 preset with fp32 scales is instantiated
// here, the other code widths in kvarn_decode_k*{lo,hi}.cu and
// kvarn_decode_d256{a,b}.cu).
#include <cudaTypedefs.h>

#include <atomic>

#include "kvarn_decode_kernel.cuh"

namespace kvarn {

// Clock cycles the dense decode kernels wait for a page copy before they
// give up (flag KVARN_DEVERR_TIMEOUT and return); 0: the default, about a
// second. Read when a call launches.
static std::atomic<long long> g_copy_wait_limit{0};
static std::atomic<int> g_copy_withhold{0};
constexpr long long kDefaultCopyWait = 2000000000LL;

void set_copy_wait_test(long long cycles, int withhold) {
  g_copy_wait_limit.store(cycles, std::memory_order_relaxed);
  g_copy_withhold.store(withhold, std::memory_order_relaxed);
}

// ------------------------------------------------------------- planning
int device_sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
    return 148;
  return n;
}

int dense_decode_warps(int32_t D) { return D == 256 ? 2 : 4; }

DensePlan plan_dense_stream(int32_t num_seqs, int32_t units_per_seq, int32_t max_tiles, int32_t D, int32_t N,
                            int32_t raw_max, int32_t kb, int32_t vb, int32_t sb, int32_t ctas_per_sm) {
  DensePlan p{};
  // tiles a CTA has in flight: one per warp, one per warp pair at head_dim 256
  const int in_flight = D == 256 ? dense_decode_warps(D) / 2 : dense_decode_warps(D);
  const int64_t resident = static_cast<int64_t>(device_sm_count()) *
                           (ctas_per_sm > 0 ? ctas_per_sm : dense_decode_ctas_per_sm(D, N, kb, vb, sb));
  const int64_t units = static_cast<int64_t>(num_seqs) * units_per_seq;
  const int64_t most = units * std::max(0, max_tiles);
  // four tiles in flight per CTA slot at least, fewer (down to one round)
  // when the whole batch is too small to fill the GPU; a multiple of the
  // tiles in flight, the granularity of the CTA ranges
  const int64_t want = std::max<int64_t>(in_flight, std::min<int64_t>(4 * in_flight, most / resident));
  p.min_tiles = static_cast<int32_t>((want + in_flight - 1) / in_flight * in_flight);
  p.tile_slots = max_tiles > 0 ? 1 + (max_tiles - 1 + p.min_tiles - 1) / p.min_tiles : 0;
  // raw tokens per split: the size with the shortest estimated raw phase,
  // (splits per CTA slot, rounded up) x (tokens of a split + about 96 tokens'
  // worth of fixed cost per split: its query rows, barriers and merge).
  // Larger splits cost less each but can leave a few CTAs with two of them.
  p.raw_chunk = kRawChunk;
  {
    int64_t best = -1;
    for (int32_t ch = kRawChunk; ch <= 16 * kRawChunk; ch *= 2) {
      const int64_t splits = raw_max > ch ? (raw_max + ch - 1) / ch : 1;
      const int64_t rounds = (units * splits + resident - 1) / resident;
      const int64_t cost = rounds * (std::min<int64_t>(ch, std::max(0, raw_max)) + 96);
      if (best < 0 || cost < best) {
        best = cost;
        p.raw_chunk = ch;
      }
      if (splits == 1) break;
    }
  }
  p.raw_splits = raw_max > p.raw_chunk ? (raw_max + p.raw_chunk - 1) / p.raw_chunk : 1;
  p.slots = p.tile_slots + p.raw_splits;
  const int64_t tile_ctas = (most + p.min_tiles - 1) / p.min_tiles;
  const int64_t raw_items = units * p.raw_splits;
  p.ctas = static_cast<int32_t>(std::max<int64_t>(1, std::min(resident, std::max(tile_ctas, raw_items))));
  return p;
}

int64_t dense_stream_workspace_bytes(int64_t rows, int32_t D, const DensePlan& plan) {
  return rows * plan.slots * kPStride(D) * 4 + (rows * 4 + 15) / 16 * 16;
}

// CTAs of the compressed decode kernel of these widths that fit on one SM at
// once (same for fp16 and bf16 queries, which share the register and smem
// footprint); computed once per combination.
int dense_decode_ctas_per_sm(int32_t D, int32_t N, int32_t kb, int32_t vb, int32_t sb) {
  // one entry per combination, filled by whichever host thread asks first
  // (threads racing on an empty entry compute the same value)
  static std::atomic<int> cache[2][2][9][9][2] = {};
  const int di = D == 256, ni = N == 64, si = sb == 2;
  if (kb < 0 || kb > 8 || vb < 0 || vb > 8) return 1;
  const int known = cache[di][ni][kb][vb][si].load(std::memory_order_relaxed);
  if (known) return known;
  int c = 0;
  {
    if (kb == 4 && vb == 2 && sb == 4) {
      if (D == 128 && N == 128) c = resident_dense<128, 128, 4, 4, 2, 4>();
      else if (D == 128) c = resident_dense<128, 64, 4, 4, 2, 4>();
      else if (N == 128) c = resident_dense<256, 128, 2, 4, 2, 4>();
      else c = resident_dense<256, 64, 2, 4, 2, 4>();
    } else if (D == 128 && sb == 2) {
      switch (16 * kb + vb) {
#define KVARN_RES_CASE(K, V) \
  case 16 * K + V: c = resident_widths<K, V, 2>(D, N); break;
        KVARN_WIDTH_PAIRS(KVARN_RES_CASE)
#undef KVARN_RES_CASE
        default: c = 1; break;
      }
    } else if (D == 128 && sb == 4) {
      switch (16 * kb + vb) {
#define KVARN_RES_CASE(K, V) \
  case 16 * K + V: c = resident_widths<K, V, 4>(D, N); break;
        KVARN_WIDTH_PAIRS_S32(KVARN_RES_CASE)
#undef KVARN_RES_CASE
        default: c = 1; break;
      }
    } else if (D == 256 && sb == 2) {
      switch (16 * kb + vb) {
#define KVARN_RES_CASE(K, V) \
  case 16 * K + V: c = resident_widths256<K, V, 2>(N); break;
        KVARN_WIDTH_PAIRS_256(KVARN_RES_CASE)
#undef KVARN_RES_CASE
        default: c = 1; break;
      }
    } else {
      c = 1;
    }
  }
  cache[di][ni][kb][vb][si].store(c, std::memory_order_relaxed);
  return c;
}

// cuTensorMapEncodeTiled of the driver, found once through the runtime.
static PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  // a function-local static: initialised once, thread-safe
  static const PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    return static_cast<PFN_cuTensorMapEncodeTiled_v12000>(nullptr);
  }();
  return fn;
}

// The cache as rows of 8-byte elements, one row per (page, KV head); the box
// is one row high and `box_bytes` wide (a page's K or V part, or one of its
// two pieces).
static cudaError_t cache_tensor_map(CUtensorMap* map, const void* cache, int64_t rows, int page_bytes,
                                    int box_bytes) {
  auto enc = tensor_map_encoder();
  if (!enc) return cudaErrorNotSupported;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(page_bytes / 8), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(page_bytes)};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(box_bytes / 8), 1u};
  const cuuint32_t estr[2] = {1u, 1u};
  const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT64, 2, const_cast<void*>(cache), dims, strides, box, estr,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t launch_decode_dense(const DecodeParams& p, const DensePlan& plan, cudaStream_t st) {
  if (p.num_seqs == 0) return cudaSuccess;
  DecArgs A{};
  {
    const int kb = p.k_bits ? p.k_bits : 4, vb = p.v_bits ? p.v_bits : 2, sb = p.scale_bytes ? p.scale_bytes : 4;
    const bool aff = p.codec == 1;
    const int kpart = aff ? AffinePage(p.D, kb, vb).k_part() : DensePage(p.D, p.N, kb, vb, sb).k_part();
    const int vpart = aff ? AffinePage(p.D, kb, vb).v_part() : DensePage(p.D, p.N, kb, vb, sb).v_part();
    if (p.codec != 2 && parts_gather(p.D, p.N, kpart, vpart, kb, vb)) {
      const int page = kpart + vpart;
      const int64_t rows = static_cast<int64_t>(p.num_pages) * p.num_kv_heads;
      // a part wider than one box is gathered as two (split where its
      // codes' first half ends); the second map is unused otherwise
      const int ks = gather_split(kpart, 2 * p.D * kb), vs = gather_split(vpart, 2 * p.D * vb);
      cudaError_t e = cache_tensor_map(&A.tmk, p.cache, rows, page, ks);
      if (e == cudaSuccess) e = cache_tensor_map(&A.tmv, p.cache, rows, page, vs);
      if (e == cudaSuccess && ks < kpart) e = cache_tensor_map(&A.tmk2, p.cache, rows, page, kpart - ks);
      if (e == cudaSuccess && vs < vpart) e = cache_tensor_map(&A.tmv2, p.cache, rows, page, vpart - vs);
      if (e != cudaSuccess) return e;
    }
  }
  A.q = p.q;
  A.kappa = p.sm_scale * kLog2e;
  A.cache = p.cache;
  A.Hq = p.num_q_heads;
  A.Hkv = p.num_kv_heads;
  A.G = p.num_q_heads / p.num_kv_heads;
  A.Q = p.num_queries > 0 ? p.num_queries : 1;
  A.tail_cap = p.tail_cap > 0 ? p.tail_cap : p.N;
  A.sink_tiles = p.sink_tokens / p.N;
  A.recent = p.recent_tokens;
  A.sink_k = p.sink_k;
  A.sink_v = p.sink_v;
  A.num_pages = p.num_pages;
  A.bt = p.block_table;
  A.bt_stride = p.bt_stride;
  A.seq_lens = p.seq_lens;
  A.max_seq_len = p.max_seq_len;
  A.tail_k = p.tail_k;
  A.tail_v = p.tail_v;
  A.ws = static_cast<float*>(p.workspace);
  const int64_t rows = static_cast<int64_t>(p.num_seqs) * A.Q * p.num_q_heads;
  A.counts = reinterpret_cast<int32_t*>(A.ws + rows * plan.slots * kPStride(p.D));
  A.num_seqs = p.num_seqs;
  A.X = p.num_kv_heads * row_groups(A.G, A.Q);
  A.min_tiles = plan.min_tiles;
  A.tile_slots = plan.tile_slots;
  A.raw_splits = plan.raw_splits;
  A.raw_chunk = plan.raw_chunk;
  A.slots = plan.slots;
  A.err = p.err;
  A.bf16 = p.bf16 ? 1 : 0;
  A.partial_tiles = p.codec == 2;
  {
    const long long w = g_copy_wait_limit.load(std::memory_order_relaxed);
    A.wait_limit = w > 0 ? w : kDefaultCopyWait;
    A.withhold = g_copy_withhold.load(std::memory_order_relaxed);
  }
  cudaError_t e = cudaErrorInvalidValue;
  const int kb = p.k_bits ? p.k_bits : 4, vb = p.v_bits ? p.v_bits : 2, sb = p.scale_bytes ? p.scale_bytes : 4;
  if (p.codec == 2) {  // the uncompressed fp16 pages (tiles of 32 tokens)
    e = p.D == 128 ? run_raw<128>(A, plan.ctas, st) : p.D == 256 ? run_raw<256>(A, plan.ctas, st)
                                                                  : cudaErrorInvalidValue;
    if (e != cudaSuccess) return e;
    return p.D == 128 ? launch_merge<128, false>(A.ws, A.slots, rows, A.counts, 0, A.tile_slots, p.out, p.lse, st)
                      : launch_merge<256, false>(A.ws, A.slots, rows, A.counts, 0, A.tile_slots, p.out, p.lse, st);
  }
  if (p.codec == 1) {
    if (p.D != 128 || p.N != 128 || kb != vb) return cudaErrorInvalidValue;
    switch (kb) {
#define KVARN_AFF_CASE(K) \
  case K: e = run_affine_widths<K>(A, p.bf16, plan.ctas, st); break;
      KVARN_AFFINE_WIDTHS(KVARN_AFF_CASE)
#undef KVARN_AFF_CASE
      default: break;
    }
    if (e != cudaSuccess) return e;
    return launch_merge<128, false>(A.ws, A.slots, rows, A.counts, 0, A.tile_slots, p.out, p.lse, st);
  }
  if (kb == 4 && vb == 2 && sb == 4) {
#define KV_DISPATCH(DD, NN, WW)                                                              \
  if (p.D == DD && p.N == NN)                                                                \
    e = run_dense<DD, NN, WW, 4, 2, 4>(A, plan.ctas, st);
    KV_DISPATCH(128, 128, 4)
    KV_DISPATCH(128, 64, 4)
    KV_DISPATCH(256, 128, 2)
    KV_DISPATCH(256, 64, 2)
#undef KV_DISPATCH
  } else if (sb == 2 && p.D == 256) {
    switch (16 * kb + vb) {
#define KVARN_RUN_CASE(K, V) \
  case 16 * K + V: e = run_dense_widths256<K, V, 2>(A, p.N, p.bf16, plan.ctas, st); break;
      KVARN_WIDTH_PAIRS_256(KVARN_RUN_CASE)
#undef KVARN_RUN_CASE
      default: break;
    }
  } else if (sb == 2) {
    switch (16 * kb + vb) {
#define KVARN_RUN_CASE(K, V) \
  case 16 * K + V: e = run_dense_widths<K, V, 2>(A, p.D, p.N, p.bf16, plan.ctas, st); break;
      KVARN_WIDTH_PAIRS(KVARN_RUN_CASE)
#undef KVARN_RUN_CASE
      default: break;
    }
  } else if (sb == 4 && p.D == 128) {
    switch (16 * kb + vb) {
#define KVARN_RUN_CASE(K, V) \
  case 16 * K + V: e = run_dense_widths<K, V, 4>(A, p.D, p.N, p.bf16, plan.ctas, st); break;
      KVARN_WIDTH_PAIRS_S32(KVARN_RUN_CASE)
#undef KVARN_RUN_CASE
      default: break;
    }
  }
  if (e != cudaSuccess) return e;
  return p.D == 128 ? launch_merge<128>(A.ws, A.slots, rows, A.counts, 0, A.tile_slots, p.out, p.lse, st)
                    : launch_merge<256>(A.ws, A.slots, rows, A.counts, 0, A.tile_slots, p.out, p.lse, st);
}

}  // namespace kvarn

// extern "C" boundary of libkvarn: argument validation on the host, then the
// launches. Declarations and the contract of every call are in kvarn.h.
#include <cuda_runtime.h>

#include <algorithm>

#include "../../include/kvarn.h"
#include "kvarn_common.cuh"
#include "kvarn_launch.h"

using namespace kvarn;

namespace {

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int32_t from_cuda(cudaError_t e) { return e == cudaSuccess ? KVARN_OK : KVARN_ECUDA; }

// Dense layout with a compiled codec variant.
int32_t check_dense(const kvarn_layout* L) {
  if (!L) return KVARN_EINVAL;
  if (L->page_tokens != kPageTokens) return KVARN_EUNSUPPORTED;
  if (L->head_dim != 128 && L->head_dim != 256) return KVARN_EUNSUPPORTED;
  if (L->tile_tokens != 128 && L->tile_tokens != 64) return KVARN_EUNSUPPORTED;
  if (L->scale_dtype != 0 && L->scale_dtype != 1) return KVARN_EUNSUPPORTED;
  if (!widths_supported(L->head_dim, L->k_bits, L->v_bits, L->scale_dtype == 1 ? 2 : 4))
    return KVARN_EUNSUPPORTED;
  if (L->norm_iters < 1 || L->norm_iters > 8) return KVARN_EUNSUPPORTED;
  if (L->rope_dim != 0) return KVARN_EINVAL;
  if (L->kv_dtype != 0 && L->kv_dtype != 1) return KVARN_EUNSUPPORTED;
  if (L->num_kv_heads < 1 || L->num_pages < 0) return KVARN_EINVAL;
  return KVARN_OK;
}

int32_t check_latent(const kvarn_layout* L) {
  if (!L) return KVARN_EINVAL;
  if (L->page_tokens != kPageTokens || L->head_dim != 512 || L->tile_tokens != 128 ||
      L->k_bits != 4 || L->v_bits != 0 || L->rope_dim != 64 || L->num_kv_heads != 1)
    return KVARN_EUNSUPPORTED;
  if (L->norm_iters < 1 || L->norm_iters > 8) return KVARN_EUNSUPPORTED;
  if (L->kv_dtype != 0 && L->kv_dtype != 1) return KVARN_EUNSUPPORTED;
  if (L->num_pages < 0) return KVARN_EINVAL;
  return KVARN_OK;
}

bool is_latent(const kvarn_layout* L) { return L && L->head_dim == 512 && L->rope_dim > 0; }

// Layout of the affine comparison codec: head_dim 128, 128-token tiles of
// 16-token pages, equal key and value widths from {2, 3, 4, 6, 8}.
int32_t check_affine(const kvarn_layout* L) {
  if (!L) return KVARN_EINVAL;
  if (L->page_tokens != kPageTokens || L->head_dim != 128 || L->tile_tokens != 128 || L->rope_dim != 0)
    return KVARN_EUNSUPPORTED;
  if (L->k_bits != L->v_bits || !affine_width_compiled(L->k_bits)) return KVARN_EUNSUPPORTED;
  if (L->kv_dtype != 0 && L->kv_dtype != 1) return KVARN_EUNSUPPORTED;
  if (L->num_kv_heads < 1 || L->num_pages < 0) return KVARN_EINVAL;
  return KVARN_OK;
}

}  // namespace

extern "C" {

int32_t kvarn_version(void) { return 100; }

const char* kvarn_status_string(int32_t s) {
  switch (s) {
    case KVARN_OK: return "ok";
    case KVARN_EINVAL: return "invalid argument";
    case KVARN_EUNSUPPORTED: return "unsupported shape or width";
    case KVARN_EALIGN: return "misaligned pointer or stride";
    case KVARN_ECUDA: return "CUDA runtime error";
    case KVARN_EWORKSPACE: return "workspace too small";
    default: return "unknown status";
  }
}

int32_t kvarn_layout_check(const kvarn_layout* L) {
  return is_latent(L) ? check_latent(L) : check_dense(L);
}

int64_t kvarn_page_bytes(const kvarn_layout* L) {
  if (kvarn_layout_check(L) != KVARN_OK) return -1;
  if (is_latent(L)) return LatentPage(L->head_dim, L->rope_dim, L->tile_tokens).bytes();
  return DensePage(L->head_dim, L->tile_tokens, L->k_bits, L->v_bits, L->scale_dtype == 1 ? 2 : 4).bytes();
}

// The k4v2 preset with fp32 scales: the page format of the append, fp16
// bypass and no-allocation paths.
static bool is_preset(const kvarn_layout* L) {
  return L->k_bits == 4 && L->v_bits == 2 && L->scale_dtype == 0;
}

static int32_t encode_tiles(const void* k, const void* v, int64_t seq_stride, int64_t head_stride,
                            int32_t num_seqs, int32_t chunk_tokens, const int32_t* tile_start,
                            const int32_t* block_table, int32_t bt_stride, const kvarn_layout* L,
                            void* cache, float* stages, uint32_t* error_flags, kvarn_stream_t stream,
                            bool affine = false) {
  int32_t s = affine ? check_affine(L) : check_dense(L);
  if (s != KVARN_OK) return s;
  if (num_seqs < 0 || chunk_tokens < 0 || chunk_tokens % L->tile_tokens) return KVARN_EINVAL;
  if (num_seqs == 0 || chunk_tokens == 0) return KVARN_OK;
  if (!k || !v || !tile_start || !block_table || !cache || !error_flags) return KVARN_EINVAL;
  if (seq_stride < 0 || head_stride < 0 || bt_stride < 1) return KVARN_EINVAL;
  if (!aligned(k, 16) || !aligned(v, 16) || seq_stride % 8 || head_stride % 8) return KVARN_EALIGN;
  if (!aligned(cache, 128) || !aligned(error_flags, 4)) return KVARN_EALIGN;
  EncodeParams p{};
  p.k = k;
  p.v = v;
  p.seq_stride = seq_stride;
  p.head_stride = head_stride;
  p.num_seqs = num_seqs;
  p.chunk_tokens = chunk_tokens;
  p.tile_start = tile_start;
  p.block_table = block_table;
  p.bt_stride = bt_stride;
  p.cache = cache;
  p.num_pages = L->num_pages;
  p.num_kv_heads = L->num_kv_heads;
  p.D = L->head_dim;
  p.N = L->tile_tokens;
  p.norm_iters = L->norm_iters;
  p.bf16 = L->kv_dtype == 1;
  p.err = error_flags;
  p.k_bits = L->k_bits;
  p.v_bits = L->v_bits;
  p.scale_bytes = L->scale_dtype == 1 ? 2 : 4;
  p.stages = stages;
  if (affine) return from_cuda(launch_encode_affine(p, reinterpret_cast<cudaStream_t>(stream)));
  return from_cuda(launch_encode_dense(p, reinterpret_cast<cudaStream_t>(stream)));
}

int32_t kvarn_encode_tiles(const void* k, const void* v, int64_t seq_stride, int64_t head_stride,
                           int32_t num_seqs, int32_t chunk_tokens, const int32_t* tile_start,
                           const int32_t* block_table, int32_t bt_stride,
                           const kvarn_layout* L, void* cache, uint32_t* error_flags,
                           kvarn_stream_t stream) {
  return encode_tiles(k, v, seq_stride, head_stride, num_seqs, chunk_tokens, tile_start, block_table,
                      bt_stride, L, cache, nullptr, error_flags, stream);
}

int64_t kvarn_encode_stage_floats(const kvarn_layout* L, int32_t num_seqs, int32_t chunk_tokens) {
  if (check_dense(L) != KVARN_OK || num_seqs < 0 || chunk_tokens < 0 || chunk_tokens % L->tile_tokens)
    return -1;
  return static_cast<int64_t>(num_seqs) * L->num_kv_heads * (chunk_tokens / L->tile_tokens) * 2 *
         stage_floats(L->head_dim, L->tile_tokens);
}

int32_t kvarn_encode_tiles_staged(const void* k, const void* v, int64_t seq_stride, int64_t head_stride,
                                  int32_t num_seqs, int32_t chunk_tokens, const int32_t* tile_start,
                                  const int32_t* block_table, int32_t bt_stride,
                                  const kvarn_layout* L, void* cache, float* stages,
                                  uint32_t* error_flags, kvarn_stream_t stream) {
  if (!stages) return KVARN_EINVAL;
  if (!aligned(stages, 16)) return KVARN_EALIGN;
  return encode_tiles(k, v, seq_stride, head_stride, num_seqs, chunk_tokens, tile_start, block_table,
                      bt_stride, L, cache, stages, error_flags, stream);
}

// max_seq_len here: the accepted length bound (sizes the tile splits); raw_max:
// raw (sink + tail) tokens a row may see (sizes the raw splits).
static DensePlan dense_plan(const kvarn_layout* L, int32_t num_seqs, int32_t num_q_heads,
                            int32_t num_queries, int32_t max_seq_len, int32_t raw_max, bool affine = false) {
  const int32_t G = num_q_heads / L->num_kv_heads;
  if (affine)
    return plan_dense_stream(num_seqs, L->num_kv_heads * row_groups(G, num_queries), max_seq_len / L->tile_tokens,
                             L->head_dim, L->tile_tokens, raw_max, L->k_bits, L->v_bits, 2,
                             affine_decode_ctas_per_sm(L->k_bits));
  return plan_dense_stream(num_seqs, L->num_kv_heads * row_groups(G, num_queries), max_seq_len / L->tile_tokens,
                           L->head_dim, L->tile_tokens, raw_max, L->k_bits ? L->k_bits : 4, L->v_bits ? L->v_bits : 2,
                           L->scale_dtype == 1 ? 2 : 4);
}

// Plan of the decode over uncompressed fp16 pages: 32-token tiles, the last
// one partial, no raw records.
static DensePlan fp16_plan(const kvarn_layout* L, int32_t num_seqs, int32_t num_q_heads, int32_t max_seq_len) {
  const int32_t G = num_q_heads / L->num_kv_heads;
  return plan_dense_stream(num_seqs, L->num_kv_heads * row_groups(G, 1), (max_seq_len + 31) / 32, L->head_dim, 32, 0,
                           4, 2, 4, raw_decode_ctas_per_sm(L->head_dim));
}

static int64_t dense_ws(const kvarn_layout* L, int32_t num_seqs, int32_t num_q_heads, int32_t num_queries,
                        const DensePlan& plan) {
  return dense_stream_workspace_bytes(static_cast<int64_t>(num_seqs) * num_q_heads * num_queries, L->head_dim, plan);
}

// Raw tokens a row can see: at most the sequence, and at most the sink, the
// newest records, a partial tile and the tokens under verification.
static int32_t raw_bound(const kvarn_layout* L, int32_t max_seq_len, int32_t num_queries, int32_t sink,
                         int32_t recent) {
  const int64_t r = static_cast<int64_t>(sink) + recent + L->tile_tokens + num_queries - 2;
  return static_cast<int32_t>(std::min<int64_t>(std::max(0, max_seq_len), std::max<int64_t>(0, r)));
}

int32_t kvarn_append(const void* k, const void* v, const int32_t* seq_lens, int32_t max_seq_len,
                     void* tail_k, void* tail_v, int32_t num_seqs, const int32_t* block_table,
                     int32_t bt_stride, const kvarn_layout* L, void* cache, uint32_t* error_flags,
                     kvarn_stream_t stream) {
  int32_t s = check_dense(L);
  if (s != KVARN_OK) return s;
  if (!is_preset(L)) return KVARN_EUNSUPPORTED;
  if (num_seqs < 0 || max_seq_len < 0) return KVARN_EINVAL;
  if (num_seqs == 0) return KVARN_OK;
  if (!k || !v || !seq_lens || !tail_k || !tail_v || !block_table || !cache || !error_flags || bt_stride < 1)
    return KVARN_EINVAL;
  if (bt_stride < (max_seq_len / L->tile_tokens) * (L->tile_tokens / kPageTokens)) return KVARN_EINVAL;
  if (!aligned(k, 16) || !aligned(v, 16) || !aligned(tail_k, 16) || !aligned(tail_v, 16)) return KVARN_EALIGN;
  if (!aligned(cache, 128) || !aligned(error_flags, 4)) return KVARN_EALIGN;
  AppendParams p{};
  p.k = k;
  p.v = v;
  p.seq_lens = seq_lens;
  p.max_seq_len = max_seq_len;
  p.tail_k = tail_k;
  p.tail_v = tail_v;
  p.num_seqs = num_seqs;
  p.block_table = block_table;
  p.bt_stride = bt_stride;
  p.cache = cache;
  p.num_pages = L->num_pages;
  p.num_kv_heads = L->num_kv_heads;
  p.D = L->head_dim;
  p.N = L->tile_tokens;
  p.norm_iters = L->norm_iters;
  p.bf16 = L->kv_dtype == 1;
  p.err = error_flags;
  return from_cuda(launch_append_commit(p, reinterpret_cast<cudaStream_t>(stream)));
}

int64_t kvarn_decode_workspace_bytes(const kvarn_layout* L, int32_t num_seqs, int32_t num_q_heads,
                                     int32_t max_seq_len) {
  if (kvarn_layout_check(L) != KVARN_OK || num_seqs < 0 || num_q_heads < 1 || max_seq_len < 0)
    return -1;
  if (is_latent(L)) return mla_workspace_bytes(num_seqs, num_q_heads, plan_mla(num_seqs, max_seq_len));
  if (num_q_heads % L->num_kv_heads) return -1;
  const DensePlan plan = dense_plan(L, num_seqs, num_q_heads, 1, max_seq_len, raw_bound(L, max_seq_len, 1, 0, 0));
  int64_t ws16 = 0;
  if (L->head_dim == 128 || L->head_dim == 256)
    ws16 = dense_stream_workspace_bytes(static_cast<int64_t>(num_seqs) * num_q_heads, L->head_dim,
                                        fp16_plan(L, num_seqs, num_q_heads, max_seq_len));
  return std::max(dense_ws(L, num_seqs, num_q_heads, 1, plan), ws16);
}

int64_t kvarn_decode_window_workspace_bytes(const kvarn_layout* L, int32_t num_seqs, int32_t num_q_heads,
                                            int32_t num_queries, int32_t max_seq_len, int32_t sink_tokens,
                                            int32_t recent_tokens) {
  if (kvarn_layout_check(L) != KVARN_OK || is_latent(L) || num_seqs < 0 || num_q_heads < 1 ||
      max_seq_len < 0 || num_queries < 1 || num_queries > KVARN_MAX_VERIFY_QUERIES ||
      num_q_heads % L->num_kv_heads || sink_tokens < 0 || recent_tokens < 0)
    return -1;
  const DensePlan plan =
      dense_plan(L, num_seqs, num_q_heads, num_queries, std::max(0, max_seq_len - num_queries + 1),
                 raw_bound(L, max_seq_len, num_queries, sink_tokens, recent_tokens));
  return dense_ws(L, num_seqs, num_q_heads, num_queries, plan);
}

int64_t kvarn_decode_verify_workspace_bytes(const kvarn_layout* L, int32_t num_seqs, int32_t num_q_heads,
                                            int32_t num_queries, int32_t max_seq_len) {
  return kvarn_decode_window_workspace_bytes(L, num_seqs, num_q_heads, num_queries, max_seq_len, 0, 0);
}

static int32_t check_decode_common(const kvarn_layout* L, int32_t num_q_heads,
                                   const int32_t* block_table, int32_t bt_stride,
                                   const int32_t* seq_lens, int32_t max_seq_len, int32_t num_seqs,
                                   float* out, void* workspace, uint32_t* error_flags) {
  if (num_seqs < 0 || max_seq_len < 0 || num_q_heads < 1) return KVARN_EINVAL;
  if (num_seqs == 0) return KVARN_OK;
  if (!block_table || !seq_lens || !out || !workspace || !error_flags) return KVARN_EINVAL;
  if (num_q_heads % L->num_kv_heads) return KVARN_EINVAL;
  if (!aligned(out, 16) || !aligned(workspace, 16)) return KVARN_EALIGN;
  (void)bt_stride;
  return KVARN_OK;
}

static int32_t decode_dense_common(const void* q, int32_t num_q_heads, int32_t num_queries, float sm_scale,
                                   const void* cache, const kvarn_layout* L, const int32_t* block_table,
                                   int32_t bt_stride, const int32_t* seq_lens, int32_t max_seq_len,
                                   const void* tail_k, const void* tail_v, int32_t tail_cap,
                                   int32_t sink_tokens, const void* sink_k, const void* sink_v,
                                   int32_t recent_tokens, int32_t num_seqs, float* out, float* lse,
                                   void* workspace, int64_t workspace_bytes, uint32_t* error_flags,
                                   kvarn_stream_t stream, bool affine = false) {
  int32_t s = affine ? check_affine(L) : check_dense(L);
  if (s != KVARN_OK) return s;
  s = check_decode_common(L, num_q_heads, block_table, bt_stride, seq_lens, max_seq_len, num_seqs,
                          out, workspace, error_flags);
  if (s != KVARN_OK || num_seqs == 0) return s;
  if (!q || !cache) return KVARN_EINVAL;
  if (num_q_heads / L->num_kv_heads > 8) return KVARN_EUNSUPPORTED;
  // committed tiles: those filled by the accepted tokens [0, len - Q + 1),
  // less the newest recent_tokens, never before the sink
  const int32_t accepted = std::max(0, max_seq_len - num_queries + 1);
  const int32_t end = std::max(sink_tokens, (std::max(0, accepted - recent_tokens) / L->tile_tokens) *
                                                L->tile_tokens);
  const int32_t committed_pages = end > sink_tokens ? end / kPageTokens : 0;
  if (bt_stride < committed_pages) return KVARN_EINVAL;
  if (!aligned(q, 16) || !aligned(cache, 128)) return KVARN_EALIGN;
  if ((tail_k && !aligned(tail_k, 16)) || (tail_v && !aligned(tail_v, 16))) return KVARN_EALIGN;
  if ((sink_k && !aligned(sink_k, 16)) || (sink_v && !aligned(sink_v, 16))) return KVARN_EALIGN;
  const DensePlan plan = dense_plan(L, num_seqs, num_q_heads, num_queries, accepted,
                                    raw_bound(L, max_seq_len, num_queries, sink_tokens, recent_tokens), affine);
  if (workspace_bytes < dense_ws(L, num_seqs, num_q_heads, num_queries, plan)) return KVARN_EWORKSPACE;
  DecodeParams p{};
  p.q = q;
  p.num_q_heads = num_q_heads;
  p.sm_scale = sm_scale;
  p.cache = static_cast<const uint8_t*>(cache);
  p.D = L->head_dim;
  p.N = L->tile_tokens;
  p.num_kv_heads = L->num_kv_heads;
  p.num_pages = L->num_pages;
  p.block_table = block_table;
  p.bt_stride = bt_stride;
  p.seq_lens = seq_lens;
  p.max_seq_len = max_seq_len;
  p.tail_k = tail_k;
  p.tail_v = tail_v;
  p.num_seqs = num_seqs;
  p.out = out;
  p.lse = lse;
  p.workspace = workspace;
  p.err = error_flags;
  p.bf16 = L->kv_dtype == 1;
  p.num_queries = num_queries;
  p.tail_cap = tail_cap;
  p.sink_tokens = sink_tokens;
  p.sink_k = sink_k;
  p.sink_v = sink_v;
  p.recent_tokens = recent_tokens;
  p.k_bits = L->k_bits;
  p.v_bits = L->v_bits;
  p.scale_bytes = affine ? 2 : (L->scale_dtype == 1 ? 2 : 4);
  p.codec = affine ? 1 : 0;
  return from_cuda(launch_decode_dense(p, plan, reinterpret_cast<cudaStream_t>(stream)));
}

int32_t kvarn_decode(const void* q, int32_t num_q_heads, float sm_scale, const void* cache,
                     const kvarn_layout* L, const int32_t* block_table, int32_t bt_stride,
                     const int32_t* seq_lens, int32_t max_seq_len, const void* tail_k,
                     const void* tail_v, int32_t num_seqs, float* out, float* lse,
                     void* workspace, int64_t workspace_bytes, uint32_t* error_flags,
                     kvarn_stream_t stream) {
  if (!L) return KVARN_EINVAL;
  return decode_dense_common(q, num_q_heads, 1, sm_scale, cache, L, block_table, bt_stride, seq_lens,
                             max_seq_len, tail_k, tail_v, L->tile_tokens, 0, nullptr, nullptr, 0, num_seqs,
                             out, lse, workspace, workspace_bytes, error_flags, stream);
}

int32_t kvarn_decode_verify(const void* q, int32_t num_q_heads, int32_t num_queries, float sm_scale,
                            const void* cache, const kvarn_layout* L, const int32_t* block_table,
                            int32_t bt_stride, const int32_t* seq_lens, int32_t max_seq_len,
                            const void* tail_k, const void* tail_v, int32_t tail_capacity,
                            int32_t num_seqs, float* out, float* lse, void* workspace,
                            int64_t workspace_bytes, uint32_t* error_flags, kvarn_stream_t stream) {
  if (!L) return KVARN_EINVAL;
  if (num_queries < 1 || num_queries > KVARN_MAX_VERIFY_QUERIES) return KVARN_EUNSUPPORTED;
  if (tail_capacity < L->tile_tokens + num_queries - 2 || tail_capacity < 1) return KVARN_EINVAL;
  return decode_dense_common(q, num_q_heads, num_queries, sm_scale, cache, L, block_table, bt_stride,
                             seq_lens, max_seq_len, tail_k, tail_v, tail_capacity, 0, nullptr, nullptr, 0,
                             num_seqs, out, lse, workspace, workspace_bytes, error_flags, stream);
}

int32_t kvarn_decode_window(const void* q, int32_t num_q_heads, int32_t num_queries, float sm_scale,
                            const void* cache, const kvarn_layout* L, const int32_t* block_table,
                            int32_t bt_stride, const int32_t* seq_lens, int32_t max_seq_len,
                            int32_t sink_tokens, const void* sink_k, const void* sink_v,
                            int32_t recent_tokens, const void* tail_k, const void* tail_v,
                            int32_t tail_capacity, int32_t num_seqs, float* out, float* lse,
                            void* workspace, int64_t workspace_bytes, uint32_t* error_flags,
                            kvarn_stream_t stream) {
  if (!L) return KVARN_EINVAL;
  if (num_queries < 1 || num_queries > KVARN_MAX_VERIFY_QUERIES) return KVARN_EUNSUPPORTED;
  if (L->tile_tokens < 1 || sink_tokens < 0 || sink_tokens % L->tile_tokens || recent_tokens < 0)
    return KVARN_EINVAL;
  if (tail_capacity < 1 || static_cast<int64_t>(tail_capacity) <
                               static_cast<int64_t>(recent_tokens) + L->tile_tokens + num_queries - 2)
    return KVARN_EINVAL;
  return decode_dense_common(q, num_q_heads, num_queries, sm_scale, cache, L, block_table, bt_stride,
                             seq_lens, max_seq_len, tail_k, tail_v, tail_capacity, sink_tokens, sink_k,
                             sink_v, recent_tokens, num_seqs, out, lse, workspace, workspace_bytes,
                             error_flags, stream);
}

int64_t kvarn_fp16_page_bytes(const kvarn_layout* L) {
  if (!L || (L->head_dim != 128 && L->head_dim != 256) || L->page_tokens != kPageTokens) return -1;
  return 4LL * kPageTokens * L->head_dim;
}

int32_t kvarn_store_fp16(const void* k, const void* v, int64_t seq_stride, int64_t head_stride,
                         int32_t num_seqs, int32_t token0, int32_t count,
                         const int32_t* block_table, int32_t bt_stride, const kvarn_layout* L,
                         void* cache, uint32_t* error_flags, kvarn_stream_t stream) {
  if (kvarn_fp16_page_bytes(L) < 0) return KVARN_EUNSUPPORTED;
  if (L->kv_dtype != 0) return KVARN_EUNSUPPORTED;
  if (num_seqs < 0 || token0 < 0 || count < 0 || token0 % kPageTokens || count % kPageTokens)
    return KVARN_EINVAL;
  if (num_seqs == 0 || count == 0) return KVARN_OK;
  if (!k || !v || !block_table || !cache || !error_flags || bt_stride < 1 || L->num_kv_heads < 1)
    return KVARN_EINVAL;
  if (!aligned(cache, 128) || !aligned(k, 4) || !aligned(v, 4)) return KVARN_EALIGN;
  StoreFp16Params p{};
  p.k = k;
  p.v = v;
  p.seq_stride = seq_stride;
  p.head_stride = head_stride;
  p.num_seqs = num_seqs;
  p.token0 = token0;
  p.count = count;
  p.block_table = block_table;
  p.bt_stride = bt_stride;
  p.cache = cache;
  p.num_pages = L->num_pages;
  p.num_kv_heads = L->num_kv_heads;
  p.D = L->head_dim;
  p.err = error_flags;
  return from_cuda(launch_store_fp16(p, reinterpret_cast<cudaStream_t>(stream)));
}

int32_t kvarn_decode_fp16(const void* q, int32_t num_q_heads, float sm_scale, const void* cache,
                          const kvarn_layout* L, const int32_t* block_table, int32_t bt_stride,
                          const int32_t* seq_lens, int32_t max_seq_len, int32_t num_seqs,
                          float* out, float* lse, void* workspace, int64_t workspace_bytes,
                          uint32_t* error_flags, kvarn_stream_t stream) {
  if (kvarn_fp16_page_bytes(L) < 0 || L->kv_dtype != 0) return KVARN_EUNSUPPORTED;
  if (L->num_kv_heads < 1 || L->num_pages < 0) return KVARN_EINVAL;
  int32_t s = check_decode_common(L, num_q_heads, block_table, bt_stride, seq_lens, max_seq_len,
                                  num_seqs, out, workspace, error_flags);
  if (s != KVARN_OK || num_seqs == 0) return s;
  if (!q || !cache) return KVARN_EINVAL;
  if (num_q_heads / L->num_kv_heads > 8) return KVARN_EUNSUPPORTED;
  if (bt_stride < (max_seq_len + kPageTokens - 1) / kPageTokens) return KVARN_EINVAL;
  if (!aligned(q, 16) || !aligned(cache, 128)) return KVARN_EALIGN;
  const DensePlan plan = fp16_plan(L, num_seqs, num_q_heads, max_seq_len);
  if (workspace_bytes < dense_stream_workspace_bytes(static_cast<int64_t>(num_seqs) * num_q_heads, L->head_dim, plan))
    return KVARN_EWORKSPACE;
  DecodeParams p{};
  p.q = q;
  p.num_q_heads = num_q_heads;
  p.sm_scale = sm_scale;
  p.cache = static_cast<const uint8_t*>(cache);
  p.D = L->head_dim;
  p.N = 32;
  p.num_kv_heads = L->num_kv_heads;
  p.num_pages = L->num_pages;
  p.block_table = block_table;
  p.bt_stride = bt_stride;
  p.seq_lens = seq_lens;
  p.max_seq_len = max_seq_len;
  p.num_seqs = num_seqs;
  p.out = out;
  p.lse = lse;
  p.workspace = workspace;
  p.err = error_flags;
  p.num_queries = 1;
  p.tail_cap = 32;
  p.codec = 2;
  return from_cuda(launch_decode_dense(p, plan, reinterpret_cast<cudaStream_t>(stream)));
}

int32_t kvarn_encode_latent(const void* latent, int64_t seq_stride, const void* rope,
                            int64_t rope_seq_stride, int32_t num_seqs, int32_t chunk_tokens,
                            const int32_t* tile_start, const int32_t* block_table,
                            int32_t bt_stride, const kvarn_layout* L, void* cache,
                            uint32_t* error_flags, kvarn_stream_t stream) {
  int32_t s = check_latent(L);
  if (s != KVARN_OK) return s;
  if (num_seqs < 0 || chunk_tokens < 0 || chunk_tokens % L->tile_tokens) return KVARN_EINVAL;
  if (num_seqs == 0 || chunk_tokens == 0) return KVARN_OK;
  if (!latent || !rope || !tile_start || !block_table || !cache || !error_flags || bt_stride < 1)
    return KVARN_EINVAL;
  if (seq_stride < 0 || rope_seq_stride < 0) return KVARN_EINVAL;
  if (!aligned(latent, 16) || !aligned(rope, 16) || seq_stride % 8 || rope_seq_stride % 8)
    return KVARN_EALIGN;
  if (!aligned(cache, 128)) return KVARN_EALIGN;
  EncodeLatentParams p{};
  p.latent = latent;
  p.seq_stride = seq_stride;
  p.rope = rope;
  p.rope_seq_stride = rope_seq_stride;
  p.num_seqs = num_seqs;
  p.chunk_tokens = chunk_tokens;
  p.tile_start = tile_start;
  p.block_table = block_table;
  p.bt_stride = bt_stride;
  p.cache = cache;
  p.num_pages = L->num_pages;
  p.norm_iters = L->norm_iters;
  p.bf16 = L->kv_dtype == 1;
  p.err = error_flags;
  return from_cuda(launch_encode_latent(p, reinterpret_cast<cudaStream_t>(stream)));
}

int32_t kvarn_decode_mla(const void* q_latent, const void* q_rope, int32_t num_heads,
                         float sm_scale, const void* cache, const kvarn_layout* L,
                         const int32_t* block_table, int32_t bt_stride, const int32_t* seq_lens,
                         int32_t max_seq_len, const void* tail_latent, const void* tail_rope,
                         int32_t num_seqs, float* out, float* lse, void* workspace,
                         int64_t workspace_bytes, uint32_t* error_flags, kvarn_stream_t stream) {
  int32_t s = check_latent(L);
  if (s != KVARN_OK) return s;
  s = check_decode_common(L, num_heads, block_table, bt_stride, seq_lens, max_seq_len, num_seqs, out,
                          workspace, error_flags);
  if (s != KVARN_OK || num_seqs == 0) return s;
  if (!q_latent || !q_rope || !cache) return KVARN_EINVAL;
  if (num_heads % 16 || num_heads > 128) return KVARN_EUNSUPPORTED;
  if (bt_stride < (max_seq_len / L->tile_tokens) * (L->tile_tokens / kPageTokens)) return KVARN_EINVAL;
  if (!aligned(q_latent, 16) || !aligned(q_rope, 16) || !aligned(cache, 128)) return KVARN_EALIGN;
  if ((tail_latent && !aligned(tail_latent, 16)) || (tail_rope && !aligned(tail_rope, 16)))
    return KVARN_EALIGN;
  const SplitPlan plan = plan_mla(num_seqs, max_seq_len);
  if (workspace_bytes < mla_workspace_bytes(num_seqs, num_heads, plan)) return KVARN_EWORKSPACE;
  DecodeParams p{};
  p.q = q_latent;
  p.q_rope = q_rope;
  p.num_q_heads = num_heads;
  p.sm_scale = sm_scale;
  p.cache = static_cast<const uint8_t*>(cache);
  p.D = 512;
  p.N = L->tile_tokens;
  p.num_kv_heads = 1;
  p.num_pages = L->num_pages;
  p.block_table = block_table;
  p.bt_stride = bt_stride;
  p.seq_lens = seq_lens;
  p.max_seq_len = max_seq_len;
  p.tail_k = tail_latent;
  p.tail_v = tail_rope;
  p.num_seqs = num_seqs;
  p.out = out;
  p.lse = lse;
  p.workspace = workspace;
  p.err = error_flags;
  p.bf16 = L->kv_dtype == 1;
  return from_cuda(launch_decode_mla(p, plan, reinterpret_cast<cudaStream_t>(stream)));
}

int64_t kvarn_affine_page_bytes(const kvarn_layout* L) {
  if (check_affine(L) != KVARN_OK) return -1;
  return AffinePage(L->head_dim, L->k_bits, L->v_bits).bytes();
}

int32_t kvarn_affine_encode_tiles(const void* k, const void* v, int64_t seq_stride, int64_t head_stride,
                                  int32_t num_seqs, int32_t chunk_tokens, const int32_t* tile_start,
                                  const int32_t* block_table, int32_t bt_stride, const kvarn_layout* L,
                                  void* cache, uint32_t* error_flags, kvarn_stream_t stream) {
  return encode_tiles(k, v, seq_stride, head_stride, num_seqs, chunk_tokens, tile_start, block_table, bt_stride, L,
                      cache, nullptr, error_flags, stream, true);
}

int64_t kvarn_affine_decode_workspace_bytes(const kvarn_layout* L, int32_t num_seqs, int32_t num_q_heads,
                                            int32_t max_seq_len) {
  if (check_affine(L) != KVARN_OK || num_seqs < 0 || num_q_heads < 1 || max_seq_len < 0 ||
      num_q_heads % L->num_kv_heads)
    return -1;
  const DensePlan plan =
      dense_plan(L, num_seqs, num_q_heads, 1, max_seq_len, raw_bound(L, max_seq_len, 1, 0, 0), true);
  return dense_ws(L, num_seqs, num_q_heads, 1, plan);
}

int32_t kvarn_affine_decode(const void* q, int32_t num_q_heads, float sm_scale, const void* cache,
                            const kvarn_layout* L, const int32_t* block_table, int32_t bt_stride,
                            const int32_t* seq_lens, int32_t max_seq_len, const void* tail_k,
                            const void* tail_v, int32_t num_seqs, float* out, float* lse, void* workspace,
                            int64_t workspace_bytes, uint32_t* error_flags, kvarn_stream_t stream) {
  if (!L) return KVARN_EINVAL;
  return decode_dense_common(q, num_q_heads, 1, sm_scale, cache, L, block_table, bt_stride, seq_lens,
                             max_seq_len, tail_k, tail_v, L->tile_tokens, 0, nullptr, nullptr, 0, num_seqs,
                             out, lse, workspace, workspace_bytes, error_flags, stream, true);
}

int32_t kvarn_set_copy_wait_test(int64_t cycles, int32_t withhold) {
  if (cycles < 0 || (withhold != 0 && withhold != 1)) return KVARN_EINVAL;
  set_copy_wait_test(cycles, withhold ? 16 : 0);
  return KVARN_OK;
}

int32_t kvarn_read_error_flags(const uint32_t* error_flags, uint32_t* host_out,
                               kvarn_stream_t stream) {
  if (!error_flags || !host_out) return KVARN_EINVAL;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (cudaMemcpyAsync(host_out, error_flags, 4, cudaMemcpyDeviceToHost, st) != cudaSuccess)
    return KVARN_ECUDA;
  return from_cuda(cudaStreamSynchronize(st));
}

}  // extern "C"

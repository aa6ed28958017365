// Internal launch parameters shared by the C-ABI layer and the kernels.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace kvarn {

struct EncodeParams {
  const void* k;
  const void* v;
  int64_t seq_stride, head_stride;
  int32_t num_seqs, chunk_tokens;
  const int32_t* tile_start;
  const int32_t* block_table;
  int32_t bt_stride;
  void* cache;
  int64_t num_pages;
  int32_t num_kv_heads, D, N, norm_iters;
  bool bf16;
  uint32_t* err;
  int32_t k_bits, v_bits, scale_bytes;  // 4, 2, 4 for the k4v2 preset with fp32 scales
  float* stages;  // optional fp32 stage records of the encoded tiles (null: none)
};

// Code widths and scale sizes with compiled kernels: every pair of a key
// width and a value width from {2, 3, 4, 5, 6, 8} (the gmlx page sets the
// two widths separately), with fp16 or fp32 scales at head_dim 128 and with
// fp16 scales at head_dim 256, where (4, 2) also takes fp32 scales.
inline bool width_compiled(int32_t b) { return b == 2 || b == 3 || b == 4 || b == 5 || b == 6 || b == 8; }
inline bool widths_supported(int32_t D, int32_t kb, int32_t vb, int32_t sb) {
  if (kb == 4 && vb == 2 && sb == 4) return true;
  if (!width_compiled(kb) || !width_compiled(vb)) return false;
  if (D == 256) return sb == 2;
  return D == 128 && (sb == 2 || sb == 4);
}

// X(KB, VB) for every compiled (key width, value width) pair with fp16
// scales; the key used by the dispatch switches is 16 KB + VB.
#define KVARN_WIDTH_ROW(X, K) X(K, 2) X(K, 3) X(K, 4) X(K, 5) X(K, 6) X(K, 8)
#define KVARN_WIDTH_PAIRS(X)                                                         \
  KVARN_WIDTH_ROW(X, 2) KVARN_WIDTH_ROW(X, 3) KVARN_WIDTH_ROW(X, 4) KVARN_WIDTH_ROW(X, 5) \
  KVARN_WIDTH_ROW(X, 6) KVARN_WIDTH_ROW(X, 8)
// X(KB, VB) for the pairs compiled at head_dim 256 (fp16 scales): all.
#define KVARN_WIDTH_PAIRS_256(X) KVARN_WIDTH_PAIRS(X)
// X(KB, VB) for the pairs compiled with fp32 scales at head_dim 128 besides
// the preset (4, 2), which has its own instantiation.
#define KVARN_WIDTH_ROW_NO42(X, K) X(K, 3) X(K, 4) X(K, 5) X(K, 6) X(K, 8)
#define KVARN_WIDTH_PAIRS_S32(X)                                                              \
  KVARN_WIDTH_ROW(X, 2) KVARN_WIDTH_ROW(X, 3) KVARN_WIDTH_ROW_NO42(X, 4) KVARN_WIDTH_ROW(X, 5) \
  KVARN_WIDTH_ROW(X, 6) KVARN_WIDTH_ROW(X, 8)

struct AppendParams {
  const void* k;  // newest token per (sequence, KV head): [B][Hkv][D]
  const void* v;
  const int32_t* seq_lens;  // lengths including the newest token
  int32_t max_seq_len;
  void* tail_k;  // [B][Hkv][N][D]
  void* tail_v;
  int32_t num_seqs;
  const int32_t* block_table;
  int32_t bt_stride;
  void* cache;
  int64_t num_pages;
  int32_t num_kv_heads, D, N, norm_iters;
  bool bf16;
  uint32_t* err;
};
cudaError_t launch_append_commit(const AppendParams& p, cudaStream_t st);

struct EncodeLatentParams {
  const void* latent;
  int64_t seq_stride;
  const void* rope;
  int64_t rope_seq_stride;
  int32_t num_seqs, chunk_tokens;
  const int32_t* tile_start;
  const int32_t* block_table;
  int32_t bt_stride;
  void* cache;
  int64_t num_pages;
  int32_t norm_iters;
  bool bf16;
  uint32_t* err;
};

struct DecodeParams {
  const void* q;            // [B][Hq][D] (dense) or q_latent [B][H][Dl] (MLA)
  const void* q_rope;       // MLA only
  int32_t num_q_heads;
  float sm_scale;
  const uint8_t* cache;
  int32_t D, N, num_kv_heads;
  int64_t num_pages;
  const int32_t* block_table;
  int32_t bt_stride;
  const int32_t* seq_lens;
  int32_t max_seq_len;
  const void* tail_k;       // tail_latent for MLA
  const void* tail_v;       // tail_rope for MLA
  int32_t num_seqs;
  float* out;
  float* lse;
  void* workspace;
  uint32_t* err;
  bool bf16;
  int32_t num_queries;  // dense: query tokens per sequence (0 or 1: plain decode)
  int32_t tail_cap;     // dense: tail rows per (sequence, KV head) (0: N)
  int32_t sink_tokens;  // dense: raw sink records (a multiple of N; 0: none)
  int32_t recent_tokens;  // dense: newest accepted tokens kept raw (0: none)
  const void* sink_k;   // dense: [B][Hkv][sink_tokens][D]
  const void* sink_v;
  int32_t k_bits, v_bits, scale_bytes;  // dense code widths and scale size (0: the k4v2 preset, fp32)
  int32_t codec;        // dense: 0 the KVarN pages, 1 the affine comparison pages
};

// (query head, query token) row groups of eight per KV head.
inline int32_t row_groups(int32_t G, int32_t Q) { return (G * Q + 7) / 8; }

// Split-K plan: tiles per split and the number of splits (+1 slot for the
// tail partial). Depends only on the arguments and the device's SM count.
struct SplitPlan {
  int32_t tiles_per_split;
  int32_t nsplit;  // splits over committed tiles
  int32_t slots;   // nsplit + 1 (the tail)
};

constexpr int32_t kRawChunk = 128;  // smallest split of the raw (sink and tail) records of the dense decode

// Plan of the compressed decode: `ctas` persistent CTAs share the flattened
// list of compressed tiles (stream-K), each taking at least `min_tiles` of
// them, so a unit of n tiles writes at most 1 + ceil((n - 1) / min_tiles)
// tile partials; raw partials (raw_chunk raw tokens each) follow them.
struct DensePlan {
  int32_t ctas;
  int32_t min_tiles;
  int32_t tile_slots;  // partial slots per row reserved for tiles
  int32_t raw_splits;
  int32_t raw_chunk;   // raw tokens per raw split (kRawChunk times a power of two)
  int32_t slots;       // tile_slots + raw_splits
};

// units_per_seq: KV heads x row groups; max_tiles: compressed tiles a unit
// can hold; raw_max: raw tokens a row can see.
DensePlan plan_dense_stream(int32_t num_seqs, int32_t units_per_seq, int32_t max_tiles, int32_t D, int32_t N,
                            int32_t raw_max, int32_t kb = 4, int32_t vb = 2, int32_t sb = 4,
                            int32_t ctas_per_sm = 0);
// Partials of `rows` output rows, then one int32 tile-partial count per row.
int64_t dense_stream_workspace_bytes(int64_t rows, int32_t D, const DensePlan& plan);
int dense_decode_warps(int32_t D);
int dense_decode_ctas_per_sm(int32_t D, int32_t N, int32_t kb = 4, int32_t vb = 2, int32_t sb = 4);
cudaError_t launch_encode_dense(const EncodeParams& p, cudaStream_t st);

// The affine comparison codec (per-token groups of 64 channels, an fp16
// scale and offset per group; head_dim 128, 128-token tiles, equal key and
// value widths): whether a width is compiled, the encoder, and the decode
// kernel's residency (the decode runs through launch_decode_dense with
// DecodeParams::codec = 1).
inline bool affine_width_compiled(int32_t b) { return b == 2 || b == 3 || b == 4 || b == 6 || b == 8; }
cudaError_t launch_encode_affine(const EncodeParams& p, cudaStream_t st);
int affine_decode_ctas_per_sm(int32_t bits);
cudaError_t launch_encode_latent(const EncodeLatentParams& p, cudaStream_t st);
cudaError_t launch_decode_dense(const DecodeParams& p, const DensePlan& plan, cudaStream_t st);

struct StoreFp16Params {
  const void* k;
  const void* v;
  int64_t seq_stride, head_stride;
  int32_t num_seqs, token0, count;
  const int32_t* block_table;
  int32_t bt_stride;
  void* cache;
  int64_t num_pages;
  int32_t num_kv_heads, D;
  uint32_t* err;
};
cudaError_t launch_store_fp16(const StoreFp16Params& p, cudaStream_t st);
// Resident CTAs per SM of the decode over uncompressed fp16 pages (the dense
// decode kernel with no codec: DecodeParams::codec = 2, N = 32).
int raw_decode_ctas_per_sm(int32_t D);

SplitPlan plan_mla(int32_t num_seqs, int32_t max_seq_len);
int64_t mla_workspace_bytes(int32_t num_seqs, int32_t num_heads, const SplitPlan& plan);
cudaError_t launch_decode_mla(const DecodeParams& p, const SplitPlan& plan, cudaStream_t st);

int device_sm_count();
// Diagnostic: clock cycles the dense decode kernels wait for a page copy (0:
// default) and whether each copy is announced larger than it is (so that its
// phase never completes and every wait runs out).
void set_copy_wait_test(long long cycles, int withhold);

}  // namespace kvarn

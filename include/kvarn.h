/*
 * kvarn.h - C ABI of the GB300 (sm_103a) KVarN KV-cache codec and its
 * decode attention.
 *
 * The method ("KVarN ... vLLM KV cache quantization" review, paragraph on the
 * four quantisation stages): every fixed tile of N tokens (128, or 64 for the
 * finer variant) of one KV head is rotated by an orthonormal Hadamard matrix
 * across head_dim, normalised by T alternating column- and row-wise standard
 * deviation passes with the scales kept in log space, then quantised by
 * asymmetric round-to-nearest, 4-bit keys and 2-bit values (the
 * kvarn_k4v2_g128 preset); the scales are folded back in when the cache is
 * read. A tile is committed only when it is full (same review, paragraph on
 * speculative decoding); the tokens of the partial last tile stay fp16 in a
 * tail buffer owned by the caller. The MLA variant quantises the shared
 * compressed latent to int4 (same review, MLA paragraph). The gmlx "KV cache
 * quantization" page ("Which layers quantize") limits head_dim to 128, 256
 * and 512.
 *
 * Conventions for every call:
 *   - All pointers named as device pointers must be device memory of the
 *     current device; the caller owns every buffer. The library allocates
 *     nothing and keeps no state between calls, except the static scratch
 *     array of kvarn_decode_noalloc described with that call.
 *   - Calls are asynchronous on `stream` (0 = legacy default stream) and
 *     keep stream order. The dense decode kernels are launched as
 *     programmatic dependents of the kernel before them on the stream: they
 *     may be scheduled while that kernel finishes, but read nothing before
 *     it has completed, so inputs written by any earlier work on the stream
 *     are seen. Every call takes host sizes and pointers and never
 *     synchronises, so a sequence of calls can be captured in a CUDA graph.
 *   - Argument errors are found on the host and returned at once, before any
 *     launch. Faults found on the device (a block-table entry outside the
 *     cache, a missing tail, a copy that never completed) set bits in the
 *     caller's 32-bit device word `error_flags` (see KVARN_DEVERR_*); read it
 *     with kvarn_read_error_flags. After such a fault the outputs of that
 *     call are unspecified, but no out-of-bounds access is made.
 *   - Device pointers must be 16-byte aligned; the cache 128-byte aligned.
 *
 * Rotated basis. Codes and scales are stored in the rotated basis y = x H,
 * H the Sylvester Hadamard matrix in natural order scaled by 1/sqrt(D)
 * (H = H^T, H H = I). Decode rotates the query once and un-rotates the
 * output once (turbo-attn page, "How it works": scores on rotated KV equal
 * scores on raw KV when the query is rotated by the same matrix).
 *
 * Dense page format (one page = P = 16 tokens of one KV head; bytes):
 *   K codes, 8D bytes, 4-bit. Lane L = 4g + t (g in 0..7, t in 0..3)
 *                      owns one 32-bit word per 16-channel k-chunk kc; its
 *                      byte m = e + 2h holds channel 16kc + 2t + e + 8h of
 *                      token g in the low nibble and of token 8 + g in the
 *                      high nibble. The word of (kc, L) sits at byte
 *                      16(32(kc/4) + L) + 4(kc%4): 16-byte units of four
 *                      k-chunks, the 32 lanes' units contiguous.
 *   V codes, 4D bytes, 2-bit. Lane L = 4g + t owns one word per four
 *                      8-channel blocks nc = 4w + c; byte c of the word is
 *                      channel 8nc + g, its token 2t + e + 8h at bit 2h + 4e
 *                      of the byte. Word w of lane L sits at byte
 *                      8(32(w/2) + L) + 4(w%2).
 *   One mask of a K word leaves four codes in the low 4 bits of its bytes,
 *   which the hardware e2m3 -> fp16 conversion turns into exact operands
 *   (code / 8), two per instruction; one mask of a V word leaves eight codes
 *   as the low 2 bits of nibbles, which the e2m1 -> fp16 conversion turns
 *   into exact operands (code / 2), two per instruction.
 * Other widths (gmlx page, "The two schemes": kvarn widths 2, 3, 4, 5, 6, 8,
 * with separate widths for keys and values): k_bits and v_bits are each any
 * of {2, 3, 4, 5, 6, 8} with head_dim 128 (fp16 or fp32 scales) and with
 * head_dim 256 (fp16 scales; fp32 scales only for k_bits 4, v_bits 2). A
 * b-bit code is stored as planes, 2: [2], 3: [2, 1], 4: [4], 5: [4, 1],
 * 6: [4, 2], 8: [4, 4] (code = plane0 + 2^w0 plane1), each plane region
 * (2*D*w bytes per page, in order) placed by one rule for width w in
 * {1, 2, 4} of which the K codes and V codes above are the w = 4 and w = 2
 * cases: lane L = 4g + t owns words of 8/w fragments; fragment f holds two
 * operand registers h = 0, 1 of two elements e' = 0, 1, element (h, e') at
 * bit 4f + 8e' + 16h (w = 4), 8f + 2h + 4e' (w = 2) or f + 8h + 16e'
 * (w = 1). K: fragment 2kc + e (tokens 8e + g), element (h, e') channel
 * 16kc + 2t + e' + 8h; words in units of U = min(4, D*w/64): word i of
 * lane L at byte 4U(32(i/U) + L) + 4(i%U). V: fragment nc, element (h, e')
 * channel 8nc + g of token 2t + e' + 8h; words in units of w: word i of
 * lane L at byte 4w(32(i/w) + L) + 4(i%w). With fp16 scales a, b and the
 * column slice are 2-byte values; each part is padded to 16 bytes. At 6 bits
 * a page of D = 128, N = 128 takes 3264 bytes, 40% of fp16.
 *
 * The page is a K part followed by a V part, each contiguous so that the
 * decode kernel can fetch and recycle them separately:
 *   K part, KP = 8D + 128 + 4C bytes, C = D*P/N:
 *     [0, 8D)             K codes (above)
 *     [8D, +64)           K a[16] fp32     [8D+64, +64)   K b[16] fp32
 *     [8D+128, +4C)       K column scales c of this page's slice
 *   V part, at KP:
 *     [KP, +4D)           V codes (above)
 *     [KP+4D, +64)        V a[16] fp32     [KP+4D+64, +64) V b[16] fp32
 *     [KP+4D+128, +4C)    V column scales of the slice
 *   page_bytes = 12D + 256 + 8C  (1920 for D = 128, N = 128).
 * The page at logical index l of a sequence holds the column scales of
 * channels [(l mod N/P) * C, +C) of its tile. All words are little-endian.
 * A dequantised rotated value is y[i, j] = c[j] * (a[i] * code[i, j] + b[i]).
 *
 * MLA latent page (latent width Dl = 512, rope width R, 4-bit, K = V):
 *   [0, 8Dl)           latent codes, token-major rows of Dl/2 bytes. A row
 *                      is four lane chunks of Dl/8 bytes; chunk t holds, per
 *                      16-channel k-chunk kc, channels 16kc + {2t, 2t+1,
 *                      2t+8, 2t+9}; its word w serves kc = 2w, 2w+1 and
 *                      nibble n of the word holds channel
 *                      16(2w + (n%4)/2) + 2t + 8(n%2) + n/4. The row's
 *                      16-byte units (unit 4t + q holds words 4q..4q+3 of
 *                      chunk t) sit at unit (4q + t) XOR 4(tau%2).
 *   [8Dl, +2RP)        rope, fp16, token-major (stored unquantised)
 *   then a[16], b[16] fp32, then the column-scale slice (Dl*P/N fp32)
 *   page_bytes = 6528 for Dl = 512, R = 64, N = 128.
 *
 * Cache arrays: dense [num_pages][num_kv_heads][page_bytes] bytes; latent
 * [num_pages][page_bytes]. Logical page l of sequence b is the physical page
 * block_table[b * bt_stride + l].
 */
#ifndef KVARN_H_
#define KVARN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* kvarn_stream_t; /* a cudaStream_t */

typedef enum {
  KVARN_OK = 0,
  KVARN_EINVAL = -1,       /* bad argument (null pointer, size, stride) */
  KVARN_EUNSUPPORTED = -2, /* shape or width with no compiled variant */
  KVARN_EALIGN = -3,       /* pointer or stride not aligned as required */
  KVARN_ECUDA = -4,        /* a CUDA runtime call failed */
  KVARN_EWORKSPACE = -5    /* workspace smaller than required */
} kvarn_status;

/* Bits of the device error word. */
#define KVARN_DEVERR_PAGE_RANGE 0x1u  /* block-table entry outside [0, num_pages) */
#define KVARN_DEVERR_NO_TAIL    0x2u  /* a raw record (tail or sink) is needed but its buffer is NULL */
#define KVARN_DEVERR_TIMEOUT    0x4u  /* a page copy did not complete in time (see kvarn_set_copy_wait_test) */
#define KVARN_DEVERR_SEQ_LEN    0x8u  /* seq_len < 0 or above max_seq_len */

typedef struct {
  int32_t head_dim;     /* D: 128, 256 (dense) or 512 (latent) */
  int32_t tile_tokens;  /* N: 128 or 64 (dense), 128 (latent) */
  int32_t page_tokens;  /* P: 16 */
  int32_t num_kv_heads; /* Hkv (1 for the latent cache) */
  int32_t k_bits;       /* 4 (the k4v2 preset); see below for other widths */
  int32_t v_bits;       /* 2 (the preset); 0 for the latent cache (V = K codes) */
  int32_t norm_iters;   /* T: 1..8 normalisation iterations */
  int32_t rope_dim;     /* 0 (dense) or 64 (latent) */
  int32_t kv_dtype;     /* 0 fp16, 1 bf16: dtype of K/V (latent), q, tails */
  int32_t scale_dtype;  /* 0: fp32 scales a, b, c; 1: fp16 scales (dense only) */
  int64_t num_pages;    /* physical pages in the cache */
} kvarn_layout;

/* Library version (major * 10000 + minor * 100 + patch). */
int32_t kvarn_version(void);

/* Human-readable name of a status code. */
const char* kvarn_status_string(int32_t status);

/* KVARN_OK if the layout names a compiled variant, an error code if not. */
int32_t kvarn_layout_check(const kvarn_layout* layout);

/* Bytes of one page of one KV head (1920 for D = 128, N = 128); -1 if the
 * layout is invalid. */
int64_t kvarn_page_bytes(const kvarn_layout* layout);

/*
 * kvarn_encode_tiles - rotate, normalise, quantise and store whole tiles.
 *
 * KVarN review, four-stage paragraph (the codec) and speculative-decoding
 * paragraph (only full tiles commit). For every sequence b < num_seqs and
 * every tile u < chunk_tokens / N, the N tokens of K and of V starting at
 * token u*N of the chunk are encoded as logical tile tile_start[b] + u of
 * sequence b and written to the N/P pages that the block table names.
 *
 *   k, v         device, kv_dtype, element (b, h, i, d) at
 *                b*seq_stride + h*head_stride + i*D + d  (elements)
 *   seq_stride, head_stride  in elements, multiples of 8
 *   chunk_tokens multiple of N (0 is a no-op)
 *   tile_start   device int32 [num_seqs]; a negative entry skips sequence b
 *                (nothing of it is read or written), so that one call can
 *                commit the tiles that filled in some sequences of a batch
 *   block_table  device int32, row stride bt_stride
 *   cache        device bytes [num_pages][Hkv][page_bytes]
 *   error_flags  device uint32 (bits are OR-ed in; never cleared here)
 * Pages outside the written tiles are not touched. Re-encoding the same
 * input writes the same bytes.
 */
int32_t kvarn_encode_tiles(const void* k, const void* v, int64_t seq_stride, int64_t head_stride,
                           int32_t num_seqs, int32_t chunk_tokens, const int32_t* tile_start,
                           const int32_t* block_table, int32_t bt_stride,
                           const kvarn_layout* layout, void* cache, uint32_t* error_flags,
                           kvarn_stream_t stream);

/*
 * kvarn_encode_tiles_staged - kvarn_encode_tiles that also writes the fp32
 * intermediates of every tile it encodes, so that each stage of the codec
 * (KVarN review, four-stage paragraph) can be checked on its own: the
 * rotation, the normalisation, and the round-to-nearest of the normalised
 * values on their row grids. The pages written are the same bytes as
 * kvarn_encode_tiles writes. A diagnostic call: the stage records are large.
 *
 *   stages  device fp32, kvarn_encode_stage_floats(layout, num_seqs,
 *           chunk_tokens) floats, 16-byte aligned. Record (b, h, u, s)
 *           (s = 0 for K, 1 for V; u the tile within the chunk) starts at
 *           float (((b*Hkv + h)*(chunk_tokens/N) + u)*2 + s) * R,
 *           R = 2*N*D + 3*N + D, and holds, in order:
 *             Y[N][D]   the rotated tile x H (token rows)
 *             Z[N][D]   the tile after the T normalisation iterations
 *             r[N]      row scales (products of the row standard deviations)
 *             lo[N]     row minimum of Z
 *             delta[N]  grid step (max - min) / (2^bits - 1) of the row
 *             c[D]      column scales
 *           The code of element (i, j) is the round-half-to-even of the
 *           exact quotient (Z[i][j] - lo[i]) / delta[i] of these fp32
 *           values (0 where delta is 0), and the stored row scales are the
 *           fp32 products a = r * delta and b = r * lo.
 * Records of sequences skipped by a negative tile_start are not written.
 * Other arguments, results and errors as kvarn_encode_tiles; a NULL `stages`
 * is KVARN_EINVAL.
 */
int64_t kvarn_encode_stage_floats(const kvarn_layout* layout, int32_t num_seqs, int32_t chunk_tokens);

int32_t kvarn_encode_tiles_staged(const void* k, const void* v, int64_t seq_stride, int64_t head_stride,
                                  int32_t num_seqs, int32_t chunk_tokens, const int32_t* tile_start,
                                  const int32_t* block_table, int32_t bt_stride,
                                  const kvarn_layout* layout, void* cache, float* stages,
                                  uint32_t* error_flags, kvarn_stream_t stream);

/*
 * kvarn_append - fused append and commit: one launch per decode step for the
 * whole batch (turbo-attn page, "Compress-on-the-wire": the new token is
 * encoded and written to the packed cache in one kernel; KVarN review,
 * speculative-decoding paragraph: a tile is committed once it is full).
 *
 * For every sequence b with L = seq_lens[b] > 0, the token at position L - 1
 * of every KV head is k / v [b][h]. If L is not a multiple of N, it is stored
 * as row (L - 1) % N of the raw tail. If it is, it completes logical tile
 * L/N - 1, whose other N - 1 tokens are rows 0..N-2 of the tail: the tile is
 * rotated, normalised, quantised and written to its pages exactly as
 * kvarn_encode_tiles would, and the tail holds no token afterwards. A
 * sequence with L = 0 is skipped. The decision is taken on the device, so a
 * captured CUDA graph of the step serves every length.
 *
 *   k, v         device, kv_dtype [num_seqs][Hkv][D]
 *   seq_lens     device int32 [num_seqs], lengths including the new token,
 *                each <= max_seq_len (else KVARN_DEVERR_SEQ_LEN, skipped)
 *   tail_k/v     device, kv_dtype [num_seqs][Hkv][N][D] (read and written)
 *   block_table, bt_stride, layout, cache, error_flags: as kvarn_encode_tiles
 */
int32_t kvarn_append(const void* k, const void* v, const int32_t* seq_lens, int32_t max_seq_len,
                     void* tail_k, void* tail_v, int32_t num_seqs, const int32_t* block_table,
                     int32_t bt_stride, const kvarn_layout* layout, void* cache, uint32_t* error_flags,
                     kvarn_stream_t stream);

/*
 * kvarn_decode_workspace_bytes - scratch needed by kvarn_decode (and by
 * kvarn_decode_fp16 and kvarn_decode_mla with the same arguments): the
 * split-K partials (running max, sum and unnormalised output per split)
 * and, for the compressed decode, one partial count per output row. The
 * call writes every part of it that it reads; nothing needs to start at
 * zero. Returns -1 for invalid arguments.
 */
int64_t kvarn_decode_workspace_bytes(const kvarn_layout* layout, int32_t num_seqs,
                                     int32_t num_q_heads, int32_t max_seq_len);

/*
 * kvarn_decode - one decode query per sequence over the compressed cache.
 *
 * out[b, h] = sum_i softmax_i(sm_scale * q[b, h] . k_i) v_i over the
 * seq_lens[b] tokens of sequence b, where tokens [0, floor(len/N)*N) are the
 * committed tiles, dequantised inline from the pages, and tokens
 * [floor(len/N)*N, len) are rows 0.. of the raw tail buffer. Query head h
 * reads KV head h / (num_q_heads / Hkv) (GQA). Split-K over tiles with a
 * log-sum-exp merge: the committed tiles of all (sequence, KV head) pairs
 * form one list that persistent CTAs share in equal contiguous ranges
 * (stream-K), so the work per CTA does not depend on how the lengths vary.
 *
 *   q            device, kv_dtype [num_seqs][num_q_heads][D]
 *   num_q_heads  a multiple of Hkv, with at most 8 query heads per KV head
 *   cache        as written by kvarn_encode_tiles
 *   seq_lens     device int32 [num_seqs], each in [0, max_seq_len]
 *   max_seq_len  host bound on seq_lens; sizes the grid
 *   tail_k/v     device, kv_dtype [num_seqs][Hkv][N][D], or NULL when every
 *                seq_len is a multiple of N
 *   out          device fp32 [num_seqs][num_q_heads][D]
 *   lse          device fp32 [num_seqs][num_q_heads] (natural log of the
 *                softmax denominator of the scaled scores) or NULL
 *   workspace    device, >= kvarn_decode_workspace_bytes(...)
 * A sequence of length 0 gives out = 0 and lse = -inf.
 */
int32_t kvarn_decode(const void* q, int32_t num_q_heads, float sm_scale, const void* cache,
                     const kvarn_layout* layout, const int32_t* block_table, int32_t bt_stride,
                     const int32_t* seq_lens, int32_t max_seq_len, const void* tail_k,
                     const void* tail_v, int32_t num_seqs, float* out, float* lse,
                     void* workspace, int64_t workspace_bytes, uint32_t* error_flags,
                     kvarn_stream_t stream);

/*
 * kvarn_decode_verify - speculative-decoding verification: num_queries query
 * tokens per sequence, causal among themselves, over the compressed cache.
 *
 * KVarN review, speculative-decoding paragraph: a block is committed only
 * once all its tokens are accepted; gmlx page, "Speed and speculative
 * decoding": a batch verifies up to 4 tokens per row. Sequence b holds
 * L = seq_lens[b] tokens, the last Q = num_queries of them under
 * verification; query token j (0 <= j < Q) is token L - Q + j and attends to
 * tokens [0, L - Q + 1 + j). Tokens up to the first query token are
 * accepted, so the committed tiles are [0, C), C = floor((L - Q + 1)/N)*N,
 * read from the pages, and tokens [C, L) are rows 0.. of the raw tail
 * buffer (at most N + Q - 2 of them). With Q = 1 this is kvarn_decode.
 *
 *   q              device, kv_dtype [num_seqs][Q][num_q_heads][D]
 *   num_queries    1 .. KVARN_MAX_VERIFY_QUERIES
 *   tail_k/v       device, kv_dtype [num_seqs][Hkv][tail_capacity][D], or
 *                  NULL when no query sees a token past C
 *   tail_capacity  rows per (sequence, KV head), >= N + Q - 2
 *   out            device fp32 [num_seqs][Q][num_q_heads][D]
 *   lse            device fp32 [num_seqs][Q][num_q_heads] or NULL
 *   workspace      device, >= kvarn_decode_verify_workspace_bytes(...)
 * Other arguments as for kvarn_decode. A query token that sees no token
 * gives out = 0 and lse = -inf. (query head, query token) pairs share the
 * tensor-core row tile in groups of eight, so up to 8 / (num_q_heads / Hkv)
 * query tokens cost the compute of one.
 */
#define KVARN_MAX_VERIFY_QUERIES 8

int64_t kvarn_decode_verify_workspace_bytes(const kvarn_layout* layout, int32_t num_seqs,
                                            int32_t num_q_heads, int32_t num_queries,
                                            int32_t max_seq_len);

int32_t kvarn_decode_verify(const void* q, int32_t num_q_heads, int32_t num_queries, float sm_scale,
                            const void* cache, const kvarn_layout* layout, const int32_t* block_table,
                            int32_t bt_stride, const int32_t* seq_lens, int32_t max_seq_len,
                            const void* tail_k, const void* tail_v, int32_t tail_capacity,
                            int32_t num_seqs, float* out, float* lse, void* workspace,
                            int64_t workspace_bytes, uint32_t* error_flags, kvarn_stream_t stream);

/*
 * kvarn_decode_window - kvarn_decode_verify with raw sink and recent records
 * (gmlx page, "The two schemes": the first tokens and the newest tokens of a
 * sequence stay fp16 while the records between them are quantised).
 *
 * Sequence b of L = seq_lens[b] tokens, the last Q = num_queries under
 * verification (Q = 1: plain decode): tokens [0, min(S, L)), S =
 * sink_tokens, are rows of the raw sink buffer; the whole tiles [S, C),
 * C = max(S, floor((L - Q + 1 - R) / N) * N), R = recent_tokens, are read
 * from the pages (logical tile t holds tokens [tN, tN + N); tiles below
 * S / N are never read); tokens [C, L) are rows 0.. of the raw tail buffer
 * (at most R + N + Q - 2 of them). Query token j sees [0, L - Q + 1 + j).
 * With S = R = 0 this is kvarn_decode_verify.
 *
 *   sink_tokens    a multiple of N (0: no sink)
 *   sink_k/v       device, kv_dtype [num_seqs][Hkv][sink_tokens][D], or NULL
 *                  when sink_tokens = 0
 *   recent_tokens  >= 0
 *   tail_capacity  rows per (sequence, KV head) of tail_k/v, >= R + N + Q - 2
 *   workspace      >= kvarn_decode_window_workspace_bytes(...) with the same
 *                  num_seqs, num_q_heads, num_queries, max_seq_len,
 *                  sink_tokens and recent_tokens
 * Other arguments as for kvarn_decode_verify. A missing sink or tail buffer
 * that a row needs sets KVARN_DEVERR_NO_TAIL. The raw records are read in
 * splits of 128 to 2048 tokens (chosen from the batch size and the raw
 * length), in parallel with the splits over the pages.
 */
int64_t kvarn_decode_window_workspace_bytes(const kvarn_layout* layout, int32_t num_seqs,
                                            int32_t num_q_heads, int32_t num_queries,
                                            int32_t max_seq_len, int32_t sink_tokens,
                                            int32_t recent_tokens);

int32_t kvarn_decode_window(const void* q, int32_t num_q_heads, int32_t num_queries, float sm_scale,
                            const void* cache, const kvarn_layout* layout, const int32_t* block_table,
                            int32_t bt_stride, const int32_t* seq_lens, int32_t max_seq_len,
                            int32_t sink_tokens, const void* sink_k, const void* sink_v,
                            int32_t recent_tokens, const void* tail_k, const void* tail_v,
                            int32_t tail_capacity, int32_t num_seqs, float* out, float* lse,
                            void* workspace, int64_t workspace_bytes, uint32_t* error_flags,
                            kvarn_stream_t stream);

/*
 * kvarn_fp16_page_bytes / kvarn_store_fp16 / kvarn_decode_fp16 - the same
 * decode skeleton over an uncompressed cache (turbo-attn page, "Also a full
 * bf16 backend": raw KV through the same kernel, so that codec and baseline
 * differ in one variable only).
 *
 * fp16 page format (P = 16 tokens of one KV head, kv_dtype elements):
 *   K: [16][D] placed per token as four lane chunks of D/4 elements, chunk t
 *      holding channels 16kc + {2t, 2t+1, 2t+8, 2t+9} in kc order;
 *   V: lane chunk L = 4g + t (D/2 elements) holding, for every 8-channel block
 *      nc, channel 8nc + g at tokens {2t, 2t+1, 2t+8, 2t+9}.
 *   page_bytes = 4 * 16 * D (K then V).
 * kvarn_store_fp16 writes tokens [token0, token0 + count) of every sequence
 * (token0 and count multiples of 16) into that format; no rotation, no
 * quantisation. kvarn_decode_fp16 reads seq_lens[b] tokens from the pages
 * (the last page may be partial) and takes the same q, out, lse, workspace
 * and error arguments as kvarn_decode; layout->tile_tokens is ignored.
 */
int64_t kvarn_fp16_page_bytes(const kvarn_layout* layout);

int32_t kvarn_store_fp16(const void* k, const void* v, int64_t seq_stride, int64_t head_stride,
                         int32_t num_seqs, int32_t token0, int32_t count,
                         const int32_t* block_table, int32_t bt_stride,
                         const kvarn_layout* layout, void* cache, uint32_t* error_flags,
                         kvarn_stream_t stream);

int32_t kvarn_decode_fp16(const void* q, int32_t num_q_heads, float sm_scale, const void* cache,
                          const kvarn_layout* layout, const int32_t* block_table,
                          int32_t bt_stride, const int32_t* seq_lens, int32_t max_seq_len,
                          int32_t num_seqs, float* out, float* lse, void* workspace,
                          int64_t workspace_bytes, uint32_t* error_flags, kvarn_stream_t stream);

/*
 * kvarn_encode_latent - the MLA variant of kvarn_encode_tiles (KVarN review,
 * MLA paragraph: the compressed latent quantised to int4): the four stages
 * run on every N-token tile of the latent (width head_dim = 512) at k_bits =
 * 4; the rope part (width rope_dim) is stored fp16 beside the codes.
 *
 *   latent  device bf16/fp16 (kv_dtype), element (b, i, d) at
 *           b*seq_stride + i*Dl + d
 *   rope    device fp16, element (b, i, r) at b*rope_seq_stride + i*R + r
 *   cache   device bytes [num_pages][page_bytes]
 * Other arguments as for kvarn_encode_tiles.
 */
int32_t kvarn_encode_latent(const void* latent, int64_t seq_stride, const void* rope,
                            int64_t rope_seq_stride, int32_t num_seqs, int32_t chunk_tokens,
                            const int32_t* tile_start, const int32_t* block_table,
                            int32_t bt_stride, const kvarn_layout* layout, void* cache,
                            uint32_t* error_flags, kvarn_stream_t stream);

/*
 * kvarn_decode_mla - absorbed-MLA decode over the latent cache: query head h
 * scores token i as sm_scale * (q_latent[b, h] . latent_i + q_rope[b, h] .
 * rope_i) and returns out[b, h] = sum_i p_i latent_i (width Dl).
 *
 *   q_latent     device kv_dtype [num_seqs][num_heads][Dl]
 *   q_rope       device kv_dtype [num_seqs][num_heads][R]
 *   tail_latent  device kv_dtype [num_seqs][N][Dl] or NULL
 *   tail_rope    device fp16 [num_seqs][N][R] or NULL
 *   out          device fp32 [num_seqs][num_heads][Dl]
 * num_heads must be a multiple of 16 and at most 128. Other arguments as for
 * kvarn_decode.
 */
int32_t kvarn_decode_mla(const void* q_latent, const void* q_rope, int32_t num_heads,
                         float sm_scale, const void* cache, const kvarn_layout* layout,
                         const int32_t* block_table, int32_t bt_stride, const int32_t* seq_lens,
                         int32_t max_seq_len, const void* tail_latent, const void* tail_rope,
                         int32_t num_seqs, float* out, float* lse, void* workspace,
                         int64_t workspace_bytes, uint32_t* error_flags, kvarn_stream_t stream);

/*
 * kvarn_decode_noalloc - kvarn_decode without a workspace argument. (The
 * pages describing the method have no counterpart of this call; it serves
 * callers that can not allocate device memory: a plugin that its host
 * framework hands only input and output tensors, a process whose device
 * memory a pool allocator owns outright, or a latency-bound path that can
 * not afford the device synchronisation a cudaMalloc may cause.)
 *
 * The split-K partials live in a fixed array of KVARN_NOALLOC_SCRATCH_BYTES
 * of static device memory inside the library, which every GPU that loads
 * the library holds until the process exits. The call allocates nothing
 * (no cudaMalloc, cudaFree or allocating library routine).
 *   - The first call on a device looks up the array's device address (with
 *     that device current) and keeps it for the later calls; make that
 *     first call before any stream capture on the device. A lookup that
 *     fails returns KVARN_ECUDA and is tried again by the next call.
 *   - Every call shares the one array per device and leaves its partials
 *     there; calls whose kernels overlap on the GPU (two streams, two host
 *     threads) race on it. Nothing in it needs to start at zero.
 *   - Returns KVARN_EWORKSPACE, launching nothing, when
 *     kvarn_decode_workspace_bytes(layout, num_seqs, num_q_heads,
 *     max_seq_len) exceeds KVARN_NOALLOC_SCRATCH_BYTES.
 * All other arguments, results and errors are those of kvarn_decode.
 */
#define KVARN_NOALLOC_SCRATCH_BYTES (16LL * 1024 * 1024)

int32_t kvarn_decode_noalloc(const void* q, int32_t num_q_heads, float sm_scale, const void* cache,
                             const kvarn_layout* layout, const int32_t* block_table,
                             int32_t bt_stride, const int32_t* seq_lens, int32_t max_seq_len,
                             const void* tail_k, const void* tail_v, int32_t num_seqs, float* out,
                             float* lse, uint32_t* error_flags, kvarn_stream_t stream);

/*
 * The affine comparison codec (gmlx "KV cache quantization" page, "The two
 * schemes": mlx-lm's affine quantization stores each token's K and V rows as
 * groups of 64 values with N-bit codes and an fp16 scale and offset per
 * group; widths 2, 3, 4, 6, 8). Built on this library's paged cache and
 * decode kernel so that it can be compared with KVarN on the same skeleton,
 * the codec being the only variable: no rotation, no normalisation.
 *
 * Quantisation of a group x[0..63] of one token: offset = fp16(min x), step
 * = fp16((max x - min x) / (2^bits - 1)) (the quotient formed in double and
 * rounded once), code = round-half-to-even of the exact quotient
 * (x - offset) / step of the stored values, clamped to [0, 2^bits - 1]; a
 * zero step gives code 0. A value is read back as offset + step * code.
 *
 * Layout: head_dim 128, tile_tokens 128, page_tokens 16, k_bits = v_bits in
 * {2, 3, 4, 6, 8}; norm_iters and scale_dtype are ignored. The page of one KV
 * head (16 tokens):
 *   K part  K codes in the placement of the dense page's K codes at k_bits
 *           (above), 2*D*k_bits bytes; then per token t, at 2*D*k_bits +
 *           8t, its two group scales then its two group offsets, fp16;
 *           padded to 16 bytes (KP = 2*D*k_bits + 128)
 *   V part  at KP: V codes in the dense page's V placement at v_bits, then
 *           the same token records; padded to 16 bytes
 * (k_bits = 4: 2304 bytes a page, 144 bytes per token and head.)
 *
 * kvarn_affine_encode_tiles takes the arguments of kvarn_encode_tiles (the
 * tiles are whole tiles of the layout, committed as the KVarN tiles are);
 * kvarn_affine_decode those of kvarn_decode, with the raw tail rows scored
 * as there, and a workspace of kvarn_affine_decode_workspace_bytes.
 */
int64_t kvarn_affine_page_bytes(const kvarn_layout* layout);

int32_t kvarn_affine_encode_tiles(const void* k, const void* v, int64_t seq_stride, int64_t head_stride,
                                  int32_t num_seqs, int32_t chunk_tokens, const int32_t* tile_start,
                                  const int32_t* block_table, int32_t bt_stride,
                                  const kvarn_layout* layout, void* cache, uint32_t* error_flags,
                                  kvarn_stream_t stream);

int64_t kvarn_affine_decode_workspace_bytes(const kvarn_layout* layout, int32_t num_seqs,
                                            int32_t num_q_heads, int32_t max_seq_len);

int32_t kvarn_affine_decode(const void* q, int32_t num_q_heads, float sm_scale, const void* cache,
                            const kvarn_layout* layout, const int32_t* block_table, int32_t bt_stride,
                            const int32_t* seq_lens, int32_t max_seq_len, const void* tail_k,
                            const void* tail_v, int32_t num_seqs, float* out, float* lse,
                            void* workspace, int64_t workspace_bytes, uint32_t* error_flags,
                            kvarn_stream_t stream);

/*
 * kvarn_set_copy_wait_test - diagnostic of the dense decode kernels'
 * (kvarn_decode, _verify, _window, _fp16, _noalloc, kvarn_affine_decode)
 * bounded waits for their page copies, so that a test can drive the time-out
 * path without making a copy fail. `cycles`: how long a wait lasts before the
 * kernel gives up (0 restores the default, 2e9 cycles, about a second; a limit
 * below 1e5 cycles is kept by polling instead of the suspending wait).
 * `withhold` = 1: every copy is announced 16 bytes larger than it is (or, for
 * copies by the threads themselves, one thread's arrival is withheld), so
 * that no copy's phase ever completes and every wait runs out, while the
 * copies themselves land as usual. On giving up, a kernel sets
 * KVARN_DEVERR_TIMEOUT in the call's error word, waits a bounded time (about
 * 50 ms) for the copies it started, writes empty partials for the rest of its
 * work and returns: the context stays usable; the call's outputs are
 * unspecified. Process-wide; read when a call launches (a captured CUDA graph
 * keeps the values of its capture). KVARN_EINVAL for a negative count or a
 * withhold other than 0 and 1. The pages describing the method have no
 * counterpart of this call.
 */
int32_t kvarn_set_copy_wait_test(int64_t cycles, int32_t withhold);

/* Copy the device error word to *host_out (synchronises `stream`). */
int32_t kvarn_read_error_flags(const uint32_t* error_flags, uint32_t* host_out,
                               kvarn_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* KVARN_H_ */

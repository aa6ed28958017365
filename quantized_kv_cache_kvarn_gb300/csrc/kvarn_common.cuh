// Device helpers shared by the KVarN kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <type_traits>

#include "../../include/kvarn.h"

namespace kvarn {

constexpr int kPageTokens = 16;

// ---------------------------------------------------------------- layout
// Byte offsets inside one dense page of one KV head (format documented in
// kvarn.h): a K part (codes, a, b, column slice) then a V part (same order).
// KB / VB: code widths; SB: bytes per scale (4: fp32, 2: fp16). C = D*P/N
// column scales per page; parts start and end on 16-byte boundaries.
constexpr int align16(int x) { return (x + 15) / 16 * 16; }

struct DensePage {
  int D, N, KB, VB, SB;
  __host__ __device__ constexpr DensePage(int d, int n, int kb = 4, int vb = 2, int sb = 4)
      : D(d), N(n), KB(kb), VB(vb), SB(sb) {}
  __host__ __device__ constexpr int cols() const { return D * kPageTokens / N; }
  __host__ __device__ constexpr int k_codes() const { return 0; }
  __host__ __device__ constexpr int k_a() const { return 2 * D * KB; }
  __host__ __device__ constexpr int k_b() const { return k_a() + SB * kPageTokens; }
  __host__ __device__ constexpr int k_col() const { return k_b() + SB * kPageTokens; }
  __host__ __device__ constexpr int k_part() const { return align16(k_col() + SB * cols()); }
  __host__ __device__ constexpr int v_codes() const { return k_part(); }
  __host__ __device__ constexpr int v_a() const { return k_part() + 2 * D * VB; }
  __host__ __device__ constexpr int v_b() const { return v_a() + SB * kPageTokens; }
  __host__ __device__ constexpr int v_col() const { return v_b() + SB * kPageTokens; }
  __host__ __device__ constexpr int v_part() const { return align16(2 * D * VB + 2 * SB * kPageTokens + SB * cols()); }
  __host__ __device__ constexpr int bytes() const { return k_part() + v_part(); }
};

// Floats of one dense tile's stage record (the encoder's fp32 intermediates:
// Y and Z, N x D each, then r, lo, delta per token and c per channel).
__host__ __device__ constexpr int64_t stage_floats(int D, int N) {
  return 2LL * N * D + 3LL * N + D;
}

// Dense decode shapes whose page parts are staged by TMA gathers of four
// pages: a 2-D tensor map over the cache with 8-byte elements and one row per
// (page, KV head), boxes one row high and at most 256 elements (2048 bytes)
// wide. A part wider than that is gathered as two boxes split where its
// codes' first half ends (gather_split), so that four pages' first boxes lie
// together and then their second boxes.
__host__ __device__ constexpr int gather_split(int part, int codes_bytes) {
  return part <= 2048 ? part : codes_bytes / 2;
}
__host__ __device__ constexpr bool gather_part_ok(int part, int codes_bytes) {
  return gather_split(part, codes_bytes) <= 2048 && part - gather_split(part, codes_bytes) <= 2048 &&
         gather_split(part, codes_bytes) % 16 == 0 && (4 * part) % 128 == 0 &&
         (4 * gather_split(part, codes_bytes)) % 128 == 0;
}
__host__ __device__ constexpr bool dense_gather(int D, int N, int KB, int VB, int SB) {
  return (D == 128 || D == 256) && (N / kPageTokens) % 4 == 0 &&
         gather_part_ok(DensePage(D, N, KB, VB, SB).k_part(), 2 * D * KB) &&
         gather_part_ok(DensePage(D, N, KB, VB, SB).v_part(), 2 * D * VB);
}

// Page of the affine comparison codec (per token, groups of 64 channels with
// an fp16 scale and offset each, original basis): a K part (K codes in the
// dense page's K plane placement at KB bits, then per token its G = D / 64
// scales and G offsets, fp16: 4G bytes at k_sc() + 4G t) and a V part (V
// codes in the V placement at VB bits, then the same records at v_sc()
// within the part), each padded to 16 bytes.
struct AffinePage {
  int D, KB, VB;
  __host__ __device__ constexpr AffinePage(int d, int kb, int vb) : D(d), KB(kb), VB(vb) {}
  __host__ __device__ constexpr int groups() const { return D / 64; }
  __host__ __device__ constexpr int k_sc() const { return 2 * D * KB; }
  __host__ __device__ constexpr int k_part() const { return align16(k_sc() + 4 * groups() * kPageTokens); }
  __host__ __device__ constexpr int v_sc() const { return 2 * D * VB; }  // within the V part
  __host__ __device__ constexpr int v_part() const { return align16(v_sc() + 4 * groups() * kPageTokens); }
  __host__ __device__ constexpr int bytes() const { return k_part() + v_part(); }
};

// Whether pages with these part sizes are staged by TMA gathers (see
// dense_gather).
__host__ __device__ constexpr bool parts_gather(int D, int N, int kp, int vp, int KB, int VB) {
  return (D == 128 || D == 256) && (N / kPageTokens) % 4 == 0 && gather_part_ok(kp, 2 * D * KB) &&
         gather_part_ok(vp, 2 * D * VB);
}

// Code planes of a b-bit code (low plane first): 2: [2], 3: [2, 1], 4: [4],
// 5: [4, 1], 6: [4, 2], 8: [4, 4]; the code is plane0 + 2^w0 plane1.
__host__ __device__ constexpr int plane_w0(int b) { return b == 2 || b == 3 ? 2 : 4; }
__host__ __device__ constexpr int plane_w1(int b) { return b == 3 || b == 5 ? 1 : b == 6 ? 2 : b == 8 ? 4 : 0; }

// MLA latent page: codes (dense-K placement), fp16 rope, a, b, column slice.
struct LatentPage {
  int D, R, N;
  __host__ __device__ constexpr LatentPage(int d, int r, int n) : D(d), R(r), N(n) {}
  __host__ __device__ constexpr int cols() const { return D * kPageTokens / N; }
  __host__ __device__ constexpr int codes() const { return 0; }
  __host__ __device__ constexpr int rope() const { return 8 * D; }
  __host__ __device__ constexpr int a() const { return 8 * D + 2 * R * kPageTokens; }
  __host__ __device__ constexpr int b() const { return a() + 64; }
  __host__ __device__ constexpr int col() const { return a() + 128; }
  __host__ __device__ constexpr int bytes() const { return col() + 4 * cols(); }
};

// ------------------------------------------------------------- dtype io
template <typename T> __device__ __forceinline__ float to_f32(T x);
template <> __device__ __forceinline__ float to_f32<__half>(__half x) { return __half2float(x); }
template <> __device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 x) {
  return __bfloat162float(x);
}

// Eight consecutive 16-bit elements from a 16-byte aligned address.
template <typename T>
__device__ __forceinline__ void load8(const T* p, float* out) {
  uint4 u = __ldg(reinterpret_cast<const uint4*>(p));
  const T* h = reinterpret_cast<const T*>(&u);
#pragma unroll
  for (int i = 0; i < 8; ++i) out[i] = to_f32<T>(h[i]);
}

__device__ __forceinline__ void set_error(uint32_t* err, uint32_t bit) {
  if (err) atomicOr(err, bit);
}

// ------------------------------------------------------------ shared mem
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ------------------------------------------------- mbarrier + bulk copy
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count));
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(
                   smem_addr(bar)),
               "r"(bytes)
               : "memory");
}

// Bulk prefetch of global memory into L2 (no completion tracking).
__device__ __forceinline__ void prefetch_l2(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// One-dimensional bulk copy global -> shared, completion counted in bytes on
// the mbarrier. Both addresses 16-byte aligned, size a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes,
                                         uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}

// 16-byte asynchronous copy global -> shared by this thread (load/store
// pipe; no bulk-copy unit involved).
__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(dst)), "l"(src) : "memory");
}

// One arrival on `bar` once every cp.async this thread issued so far has
// landed (counts toward the phase: the barrier expects one per thread).
__device__ __forceinline__ void cp_async_arrive(uint64_t* bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_addr(bar)) : "memory");
}

// Waits until every cp.async this thread issued has landed.
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// TMA gather of four rows (x .. x + box - 1 of rows y0..y3) of a 2-D tensor
// map into shared memory, completion counted in bytes on `bar`.
__device__ __forceinline__ void tma_gather4(void* dst, const void* tmap, int x, int y0, int y1, int y2, int y3,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cta.global.tile::gather4.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4, "
      "%5, %6}], [%7];" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y0), "r"(y1), "r"(y2), "r"(y3), "r"(smem_addr(bar))
      : "memory");
}

// The waiting thread may be suspended (it issues nothing) until the phase
// completes or about 20 us pass.
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity), "r"(20000u)
      : "memory");
  return ok != 0;
}

// 2^x by the special-function unit (relative error about 2^-22; flushes
// subnormal results to zero, which only ever meets weights below 2^-126).
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Bounded wait: gives up after about `limit_cycles` SM clocks and returns
// false, so that a copy that never lands can not hang the GPU.
__device__ __forceinline__ bool mbar_test_phase(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Waits at most about limit_cycles for the phase. try_wait may suspend the
// thread until the phase completes, so a limit below kPollWaitBelow (a
// diagnostic setting) is kept by polling with the non-blocking test_wait.
constexpr long long kPollWaitBelow = 100000;
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity,
                                                  long long limit_cycles = 2000000000LL) {
  if (limit_cycles < kPollWaitBelow) {
    const long long t0 = clock64();
    while (!mbar_test_phase(bar, parity))
      if (clock64() - t0 > limit_cycles) return false;
    return true;
  }
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (clock64() - t0 > limit_cycles) return false;
  }
  return true;
}

// --------------------------------------------------------------- mma
// D(16x8 f32) += A(16x16 f16, row) * B(16x8 f16, col).
__device__ __forceinline__ void mma_f16(float* d, uint32_t a0, uint32_t a1, uint32_t a2,
                                        uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t h2_as_u32(__half2 h) {
  return *reinterpret_cast<uint32_t*>(&h);
}
__device__ __forceinline__ __half2 u32_as_h2(uint32_t u) {
  return *reinterpret_cast<__half2*>(&u);
}

// Split two fp32 values into fp16 hi + lo parts (x ~ hi + lo to ~2^-22).
__device__ __forceinline__ void split_hi_lo(float x0, float x1, uint32_t& hi, uint32_t& lo) {
  __half2 h = __floats2half2_rn(x0, x1);
  float2 hf = __half22float2(h);
  __half2 l = __floats2half2_rn(x0 - hf.x, x1 - hf.y);
  hi = h2_as_u32(h);
  lo = h2_as_u32(l);
}

// Pairs of fp32 values: one packed instruction for both (sm_100 and later).
__device__ __forceinline__ float2 f2(float x) { return make_float2(x, x); }
__device__ __forceinline__ float2 f2mul(float2 a, float2 b) { return __fmul2_rn(a, b); }
__device__ __forceinline__ float2 f2add(float2 a, float2 b) { return __fadd2_rn(a, b); }
__device__ __forceinline__ float2 f2fma(float2 a, float2 b, float2 c) { return __ffma2_rn(a, b, c); }

// split_hi_lo of a pair held as float2 (x - hi is exact, as above).
__device__ __forceinline__ void split_hi_lo2(float2 x, uint32_t& hi, uint32_t& lo) {
  const __half2 h = __float22half2_rn(x);
  const float2 r = __ffma2_rn(__half22float2(h), f2(-1.f), x);
  hi = h2_as_u32(h);
  lo = h2_as_u32(__float22half2_rn(r));
}

__device__ __forceinline__ uint32_t lop3_and_or(uint32_t x, uint32_t mask, uint32_t orv) {
  uint32_t r;
  // (x & mask) | orv
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(r) : "r"(x), "r"(mask), "r"(orv));
  return r;
}

// Codes to exact fp16 integers (the MLA latent words and the 1-bit planes).
// A 4-bit field at bits 0-3 (and 16-19) OR-ed into 0x6400 (fp16 1024) is
// 1024 + n; one at bits 4-7 is 1024 + 16n. The offsets below recentre them:
// 4-bit codes to n - 8. Every intermediate is an integer below 2048, so each
// step is exact and the mma sees ordinary normal fp16 operands. (Masked fields used
// directly as fp16 subnormals would save the recentring, but the tensor
// cores align a sum of such products as if the subnormal were 2^-14, which
// drops about 10 - p bits of a field at bit p from the sum.)
constexpr uint32_t kMagic = 0x64006400u;

// One K word -> 4 half2: (kc even: b01, b23), (kc odd: b01, b23).
__device__ __forceinline__ void dequant_k_word(uint32_t x, uint32_t* out) {
  const __half2 sub = __halves2half2(__ushort_as_half(0x6408), __ushort_as_half(0x6408));  // 1032
  const __half2 s16 = __halves2half2(__ushort_as_half(0x2C00), __ushort_as_half(0x2C00));  // 1/16
  const __half2 o16 = __halves2half2(__ushort_as_half(0xD480), __ushort_as_half(0xD480));  // -72
  const uint32_t y = x >> 8;
  out[0] = h2_as_u32(__hsub2(u32_as_h2(lop3_and_or(x, 0x000F000Fu, kMagic)), sub));
  out[1] = h2_as_u32(__hfma2(u32_as_h2(lop3_and_or(x, 0x00F000F0u, kMagic)), s16, o16));
  out[2] = h2_as_u32(__hsub2(u32_as_h2(lop3_and_or(y, 0x000F000Fu, kMagic)), sub));
  out[3] = h2_as_u32(__hfma2(u32_as_h2(lop3_and_or(y, 0x00F000F0u, kMagic)), s16, o16));
}

// fp16 bit patterns of small integers (|n| < 2048) and of powers of two,
// for compile-time operand constants.
__host__ __device__ constexpr unsigned short fp16_int(int n) {
  const unsigned short sgn = n < 0 ? 0x8000u : 0u;
  const int a = n < 0 ? -n : n;
  int e = 0;
  while ((2 << e) <= a) ++e;
  return a == 0 ? sgn : static_cast<unsigned short>(sgn | ((e + 15) << 10) | ((a - (1 << e)) << (10 - e)));
}
__host__ __device__ constexpr unsigned short fp16_pow2(int e) { return static_cast<unsigned short>((e + 15) << 10); }

__device__ __forceinline__ __half2 h2_bits(unsigned short b) {
  return __halves2half2(__ushort_as_half(b), __ushort_as_half(b));
}

// The W-bit fields at bits P and P + 16 of x (P + W <= 8) as the exact fp16
// pair (n - C): OR-ed into fp16 1024 a field is 1024 + 2^P n; scaling by
// 2^-P and subtracting 1024 / 2^P + C leaves n - C. Every intermediate is an
// integer below 2048 times a power of two, so each step is exact.
template <int W, int P, int C>
__device__ __forceinline__ uint32_t field_h2(uint32_t x) {
  constexpr uint32_t m = ((1u << W) - 1u) << P;
  const __half2 v = u32_as_h2(lop3_and_or(x, m | (m << 16), kMagic));
  if constexpr (P == 0)
    return h2_as_u32(__hsub2(v, h2_bits(fp16_int(1024 + C))));
  else
    return h2_as_u32(__hfma2(v, h2_bits(fp16_pow2(-P)), h2_bits(fp16_int(-((1024 >> P) + C)))));
}

// ---- code planes to tensor-core operands (page format in include/kvarn.h)
// Blackwell converts a pair of 6-bit e2m3 values (one per byte of a 16-bit
// half-word, bits 6-7 of each byte ignored) or of 4-bit e2m1 values (the two
// nibbles of a byte) to an fp16 pair in one instruction. With the sign and
// the upper exponent bit clear both formats are linear in their low bits: a
// 4-bit field n is the e2m3 value n / 8 (n < 8 subnormal m/8, n >= 8 the
// normal 1 + m/8) and a 2-bit field n the e2m1 value n / 2. Both are exact
// normal fp16 numbers, so a plane word becomes operands with one mask per
// four (4-bit) or eight (2-bit) registers and one conversion per register.
__device__ __forceinline__ uint32_t e2m3x2_lo(uint32_t x) {  // bytes 0, 1 -> fp16 pair
  uint32_t r;
  asm("{ .reg .b16 l, h; mov.b32 {l, h}, %1; cvt.rn.f16x2.e2m3x2 %0, l; }" : "=r"(r) : "r"(x));
  return r;
}
__device__ __forceinline__ uint32_t e2m3x2_hi(uint32_t x) {  // bytes 2, 3 -> fp16 pair
  uint32_t r;
  asm("{ .reg .b16 l, h; mov.b32 {l, h}, %1; cvt.rn.f16x2.e2m3x2 %0, h; }" : "=r"(r) : "r"(x));
  return r;
}
template <int BYTE>  // the two nibbles of byte BYTE -> fp16 pair (low nibble in the low half)
__device__ __forceinline__ uint32_t e2m1x2_byte(uint32_t x) {
  uint32_t r;
  if constexpr (BYTE == 0)
    asm("{ .reg .b8 a, b, c, d; mov.b32 {a, b, c, d}, %1; cvt.rn.f16x2.e2m1x2 %0, a; }" : "=r"(r) : "r"(x));
  else if constexpr (BYTE == 1)
    asm("{ .reg .b8 a, b, c, d; mov.b32 {a, b, c, d}, %1; cvt.rn.f16x2.e2m1x2 %0, b; }" : "=r"(r) : "r"(x));
  else if constexpr (BYTE == 2)
    asm("{ .reg .b8 a, b, c, d; mov.b32 {a, b, c, d}, %1; cvt.rn.f16x2.e2m1x2 %0, c; }" : "=r"(r) : "r"(x));
  else
    asm("{ .reg .b8 a, b, c, d; mov.b32 {a, b, c, d}, %1; cvt.rn.f16x2.e2m1x2 %0, d; }" : "=r"(r) : "r"(x));
  return r;
}

// Bit of element (h, e') (operand register h, its half e') of fragment f in
// a plane word of width w (page format in include/kvarn.h).
__host__ __device__ constexpr int plane_bit(int w, int f, int h, int ep) {
  return w == 4 ? 4 * f + 8 * ep + 16 * h : w == 2 ? 8 * f + 2 * h + 4 * ep : f + 8 * h + 16 * ep;
}

// Scale of a plane's operand values: a w-bit field n becomes plane_kappa(w) * n.
__host__ __device__ constexpr float plane_kappa(int w) { return w == 4 ? 0.125f : w == 2 ? 0.5f : 1.f; }
// Operand value of a b-bit code n: code_kappa(b) * (n - code_center(b)).
// 2-, 4- and 6-bit codes are used as they are. 3- and 5-bit codes are
// recentred on 2^(b-1) at no cost (their 1-bit plane's conversion takes the
// offset); 8-bit codes are recentred by one subtraction, which keeps their
// products near the size of the sums they feed (uncentred 8-bit codes lost
// accuracy in the tensor-core sums: max output error 1.5e-3 against 1.8e-4
// recentred; uncentred 6-bit codes measured 2.5e-4).
__host__ __device__ constexpr float code_kappa(int b) { return plane_kappa(plane_w0(b)); }
__host__ __device__ constexpr int code_center(int b) { return b == 3 || b == 5 || b == 8 ? 1 << (b - 1) : 0; }

// Operand pair (b0, b1) of fragment SLOT of a plane word of width W. Width 4:
// fragment SLOT is the low (0) or high (1) nibble of every byte, b0 the low
// half-word, b1 the high one, values n / 8. Width 2: fragment SLOT is byte
// SLOT, its bits 0-1 and 4-5 b0, bits 2-3 and 6-7 b1, values n / 2. Width 1:
// the fields at bits SLOT and SLOT + 16 form b0, those of the word >> 8 form
// b1, values n - C.
template <int W, int SLOT, int C = 0>
__device__ __forceinline__ void plane_pair(uint32_t x, uint32_t& b0, uint32_t& b1) {
  if constexpr (W == 4) {
    const uint32_t m = (SLOT ? (x >> 4) : x) & 0x0F0F0F0Fu;
    b0 = e2m3x2_lo(m);
    b1 = e2m3x2_hi(m);
  } else if constexpr (W == 2) {
    b0 = e2m1x2_byte<SLOT>(x & 0x33333333u);
    b1 = e2m1x2_byte<SLOT>((x >> 2) & 0x33333333u);
  } else {
    b0 = field_h2<W, W * SLOT, C>(x);
    b1 = field_h2<W, W * SLOT, C>(x >> 8);
  }
}

// Operand pair of a B-bit code (one or two planes) as exact fp16
// code_kappa(B) * (n - code_center(B)). x0 / x1: the words of plane 0 /
// plane 1 holding the fragment; S0 / S1 its slots in them. Two planes
// combine as kappa0 n0 + 2^W0 kappa0 n1, less the centre: a 1-bit plane
// takes its offset in its own conversion, an 8-bit code's centre is
// subtracted after the combination. Every value is a multiple of kappa0 of
// magnitude below 2^B kappa0 <= 32, exact in fp16.
template <int B, int S0, int S1>
__device__ __forceinline__ void code_pair(uint32_t x0, uint32_t x1, uint32_t& b0, uint32_t& b1) {
  constexpr int W0 = plane_w0(B), W1 = plane_w1(B);
  if constexpr (W1 == 0) {
    plane_pair<W0, S0>(x0, b0, b1);
  } else {
    uint32_t l0, l1, h0, h1;
    plane_pair<W0, S0>(x0, l0, l1);
    constexpr int LOG2_K0 = W0 == 4 ? -3 : -1;
    if constexpr (W1 == 1) {
      plane_pair<1, S1, (1 << (B - 1 - W0))>(x1, h0, h1);
      const __half2 sc = h2_bits(fp16_pow2(W0 + LOG2_K0));
      b0 = h2_as_u32(__hfma2(u32_as_h2(h0), sc, u32_as_h2(l0)));
      b1 = h2_as_u32(__hfma2(u32_as_h2(h1), sc, u32_as_h2(l1)));
    } else {
      plane_pair<W1, S1>(x1, h0, h1);
      const __half2 sc = h2_bits(fp16_pow2(W0 + LOG2_K0 - (W1 == 4 ? -3 : -1)));
      b0 = h2_as_u32(__hfma2(u32_as_h2(h0), sc, u32_as_h2(l0)));
      b1 = h2_as_u32(__hfma2(u32_as_h2(h1), sc, u32_as_h2(l1)));
      if constexpr (code_center(B) != 0) {
        const __half2 ctr = h2_bits(fp16_pow2(B - 1 + LOG2_K0));
        b0 = h2_as_u32(__hsub2(u32_as_h2(b0), ctr));
        b1 = h2_as_u32(__hsub2(u32_as_h2(b1), ctr));
      }
    }
  }
}

// Pairwise (tree) reduction of a register array in place: log2(N)
// dependent steps instead of N - 1. Returns a[0].
template <int N, typename T, typename Op>
__device__ __forceinline__ T tree_reduce(T (&a)[N], Op op) {
#pragma unroll
  for (int w = 1; w < N; w *= 2)
#pragma unroll
    for (int i = 0; i + w < N; i += 2 * w) a[i] = op(a[i], a[i + w]);
  return a[0];
}

// Compile-time loop: f(std::integral_constant<int, I>) for I in [B, E).
template <int B, int E, typename F>
__device__ __forceinline__ void static_for(F&& f) {
  if constexpr (B < E) {
    f(std::integral_constant<int, B>{});
    static_for<B + 1, E>(f);
  }
}

// NW consecutive 32-bit words from shared memory (NW = 1, 2 or 4, aligned).
template <int NW>
__device__ __forceinline__ void load_words(const unsigned char* p, uint32_t (&out)[NW]) {
  if constexpr (NW == 4) {
    const uint4 v = *reinterpret_cast<const uint4*>(p);
    out[0] = v.x; out[1] = v.y; out[2] = v.z; out[3] = v.w;
  } else if constexpr (NW == 2) {
    const uint2 v = *reinterpret_cast<const uint2*>(p);
    out[0] = v.x; out[1] = v.y;
  } else {
    out[0] = *reinterpret_cast<const uint32_t*>(p);
  }
}

// Two consecutive scale values (fp32 or fp16 in the page) as float2.
template <int SB>
__device__ __forceinline__ float2 load_scale2(const unsigned char* p) {
  if constexpr (SB == 4) return *reinterpret_cast<const float2*>(p);
  else return __half22float2(*reinterpret_cast<const __half2*>(p));
}

__device__ __forceinline__ float warp_max_xor(float v, int lo, int hi) {
  for (int o = lo; o < hi; o <<= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float warp_sum_xor(float v, int lo, int hi) {
  for (int o = lo; o < hi; o <<= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// ------------------------------------------------- programmatic launch
// A kernel that calls pdl_launch_dependents lets the next kernel on its
// stream, if that one is launched as a programmatic dependent, be scheduled
// while it still runs; the dependent calls pdl_wait_primary before it reads
// anything, which returns once the kernel before it has completed and its
// memory operations are visible. Both are no-ops for an ordinary launch.
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait_primary() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

}  // namespace kvarn

// Device helpers shared by the verify-step kernels (sm_103a).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "kernels.h"
#include "spec_verify.h"

namespace sv {

__device__ __forceinline__ void set_status(uint32_t *st, uint32_t bits) {
  if (st != nullptr) atomicOr(st, bits);
}

// ---------------------------------------------------------------- conversions
__device__ __forceinline__ float bf16_bits_to_f32(uint32_t b16) {
  return __uint_as_float(b16 << 16);
}

// Order-preserving integer key of a logit (larger value -> larger key).
// -0 is mapped to +0 so the two zeros form one tie class.  NaN never reaches
// here (its row is rejected first).
__device__ __forceinline__ uint32_t key_of_bf16(uint32_t b) {
  if (b == 0x8000u) b = 0;
  return (b & 0x8000u) ? (~b & 0xFFFFu) : (b | 0x8000u);
}
__device__ __forceinline__ uint32_t key_of_f32(uint32_t b) {
  if (b == 0x80000000u) b = 0;
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

// ---------------------------------------------------------------- Philox4x32-10
// Salmon, Moraes, Dror, Shaw, "Parallel Random Numbers: As Easy as 1, 2, 3"
// (SC'11), section "Philox": per round, counter words 0 and 2 are multiplied
// by two odd 32-bit constants; the high halves are mixed with words 1 and 3
// and the round key; the key advances by two Weyl constants between rounds.
struct U4 { uint32_t x, y, z, w; };

__device__ __forceinline__ U4 philox4x32_10(U4 c, uint32_t k0, uint32_t k1) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    if (r) { k0 += 0x9E3779B9u; k1 += 0xBB67AE85u; }
    const uint32_t lo0 = 0xD2511F53u * c.x, hi0 = __umulhi(0xD2511F53u, c.x);
    const uint32_t lo1 = 0xCD9E8D57u * c.z, hi1 = __umulhi(0xCD9E8D57u, c.z);
    c = U4{hi1 ^ c.y ^ k0, lo1, hi0 ^ c.w ^ k1, lo0};
  }
  return c;
}

// 24-bit uniform index k in [0, 2^24): u = k * 2^-24.
__device__ __forceinline__ uint32_t u24(uint32_t w) { return w >> 8; }

// ---------------------------------------------------------------- reductions
template <typename T>
__device__ __forceinline__ T warp_sum(T v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float warp_min(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fminf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ unsigned long long warp_sum_u64(unsigned long long v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Block-wide sum in a fixed tree order (deterministic).  `red` holds >= 32
// doubles of shared memory.  All threads get the result.
template <int NT>
__device__ __forceinline__ double block_sum_d(double v, double *red) {
  v = warp_sum(v);
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  __syncthreads();
  if (l == 0) red[w] = v;
  __syncthreads();
  double s = 0.0;
#pragma unroll
  for (int i = 0; i < NT / 32; ++i) s += red[i];
  return s;
}

template <int NT>
__device__ __forceinline__ float block_max_f(float v, float *red) {
  v = warp_max(v);
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  __syncthreads();
  if (l == 0) red[w] = v;
  __syncthreads();
  float s = -INFINITY;
#pragma unroll
  for (int i = 0; i < NT / 32; ++i) s = fmaxf(s, red[i]);
  return s;
}

// Exclusive prefix sum of one u64 per thread over the block, in thread order.
template <int NT>
__device__ __forceinline__ unsigned long long block_exclusive_scan_u64(
    unsigned long long v, unsigned long long *red, unsigned long long *total) {
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  unsigned long long inc = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long t = __shfl_up_sync(0xffffffffu, inc, o);
    if (l >= o) inc += t;
  }
  __syncthreads();
  if (l == 31) red[w] = inc;
  __syncthreads();
  unsigned long long base = 0, tot = 0;
#pragma unroll
  for (int i = 0; i < NT / 32; ++i) {
    if (i < w) base += red[i];
    tot += red[i];
  }
  *total = tot;
  return base + inc - v;
}

// ---------------------------------------------------------------- float-float sums
// Unevaluated sum hi + lo of two floats (about 48 significant bits), added with
// Knuth's two-sum.  Used for block reductions instead of fp64, which runs at a
// small fraction of the fp32 rate on this GPU.
struct FF {
  float hi, lo;
};

__device__ __forceinline__ FF ff_make(float x) { return FF{x, 0.0f}; }

__device__ __forceinline__ FF ff_add(FF a, FF b) {
  const float s = __fadd_rn(a.hi, b.hi);
  const float bv = __fsub_rn(s, a.hi);
  const float err = __fadd_rn(__fsub_rn(a.hi, __fsub_rn(s, bv)), __fsub_rn(b.hi, bv));
  const float lo = __fadd_rn(__fadd_rn(a.lo, b.lo), err);
  const float hi = __fadd_rn(s, lo);
  return FF{hi, __fsub_rn(lo, __fsub_rn(hi, s))};
}

__device__ __forceinline__ FF shfl_ff(FF v, int src) {
  return FF{__shfl_sync(0xffffffffu, v.hi, src), __shfl_sync(0xffffffffu, v.lo, src)};
}

__device__ __forceinline__ FF warp_sum_ff(FF v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    FF t;
    t.hi = __shfl_xor_sync(0xffffffffu, v.hi, o);
    t.lo = __shfl_xor_sync(0xffffffffu, v.lo, o);
    v = ff_add(v, t);
  }
  return v;
}

// a >= b for normalized float-float values.
__device__ __forceinline__ bool ff_ge(FF a, FF b) {
  return a.hi > b.hi || (a.hi == b.hi && a.lo >= b.lo);
}

__device__ __forceinline__ FF ff_from_double(double x) {
  const float hi = static_cast<float>(x);
  return FF{hi, static_cast<float>(x - static_cast<double>(hi))};
}

__device__ __forceinline__ double ff_to_double(FF a) {
  return static_cast<double>(a.hi) + static_cast<double>(a.lo);
}

// ---------------------------------------------------------------- error-free transforms
// Knuth's two-sum (any magnitudes), the fast two-sum (|a| >= |b|) and the
// fma-based exact product: the building blocks of float-float arithmetic.
__device__ __forceinline__ FF two_sum(float a, float b) {
  const float s = __fadd_rn(a, b);
  const float bv = __fsub_rn(s, a);
  return FF{s, __fadd_rn(__fsub_rn(a, __fsub_rn(s, bv)), __fsub_rn(b, bv))};
}
__device__ __forceinline__ FF quick_two_sum(float a, float b) {
  const float s = __fadd_rn(a, b);
  return FF{s, __fsub_rn(b, __fsub_rn(s, a))};
}
__device__ __forceinline__ FF two_prod(float a, float b) {
  const float p = __fmul_rn(a, b);
  return FF{p, __fmaf_rn(a, b, -p)};
}
__device__ __forceinline__ FF ff_mul(FF a, FF b) {
  const FF p = two_prod(a.hi, b.hi);
  return quick_two_sum(p.hi, __fmaf_rn(a.hi, b.lo, __fmaf_rn(a.lo, b.hi, p.lo)));
}
__device__ __forceinline__ FF ff_neg(FF a) { return FF{-a.hi, -a.lo}; }

// Table of 2^(j/64), j = -32..32, as float-float pairs (x = hi, y = lo): copied
// into shared memory by threads 0..64 of a block from the launch parameters
// (computed once on the host in double precision).
constexpr int kExp2Tab = 65;
__device__ __forceinline__ void exp2_table_fill(float2 *tab, const float2 *src) {
  const int t = threadIdx.x;
  if (t < kExp2Tab) tab[t] = src[t];
}

// 2^y for a float-float y <= 0, as a float-float with relative error near
// 2^-44: y = k + j/64 + s with integers k, j (|j| <= 32) and |s| <= 1/128 (both
// subtractions exact), 2^(j/64) from the table, 2^s = e^(s ln 2) by its Taylor
// series through the fifth power (remainder below 4e-17).  Results below
// 2^-126 are returned as 0.
__device__ __forceinline__ FF exp2_ff(FF y, const float2 *tab) {
  if (!(y.hi >= -126.0f)) return FF{0.0f, 0.0f};
  const float k = rintf(y.hi);
  const FF r = quick_two_sum(__fsub_rn(y.hi, k), y.lo);
  const float j = rintf(__fmul_rn(r.hi, 64.0f));
  const FF sx = quick_two_sum(__fsub_rn(r.hi, __fmul_rn(j, 0.015625f)), r.lo);
  constexpr float kLn2Hi = 0.6931471824645996f, kLn2Lo = -1.9046542121259336e-09f;
  FF u = two_prod(sx.hi, kLn2Hi);
  u = quick_two_sum(u.hi, __fmaf_rn(sx.hi, kLn2Lo, __fmaf_rn(sx.lo, kLn2Hi, u.lo)));
  const FF u2 = two_prod(u.hi, u.hi);
  const float u2lo = __fmaf_rn(2.0f * u.hi, u.lo, u2.lo);
  const float t3 = __fmul_rn(__fmul_rn(u2.hi, u.hi),
                             __fmaf_rn(u.hi, __fmaf_rn(u.hi, 1.0f / 120.0f, 1.0f / 24.0f),
                                       1.0f / 6.0f));
  const FF e1 = two_sum(1.0f, u.hi);
  const FF e2 = two_sum(e1.hi, __fmul_rn(0.5f, u2.hi));
  const float lo = __fadd_rn(__fadd_rn(__fadd_rn(e1.lo, e2.lo), __fadd_rn(u.lo, 0.5f * u2lo)), t3);
  FF e = quick_two_sum(e2.hi, lo);
  const float2 tj = tab[static_cast<int>(j) + 32];
  e = ff_mul(e, FF{tj.x, tj.y});
  const int ki = static_cast<int>(k);                       // -126 .. 0
  const float p2 = __int_as_float((ki + 127) << 23);         // 2^k exactly
  return FF{__fmul_rn(e.hi, p2), __fmul_rn(e.lo, p2)};
}

// ---------------------------------------------------------------- 64-bit fixed point
// Draw weights as exact integers in units of 2^-63: a float r in [0, 2) is
// exact down to 2^-40 and truncated below (the error of a sum of V weights is
// below V 2^-63, far below any draw's resolution); sums of weights that add
// up to at most 2 fit in 64 bits.
__device__ __forceinline__ unsigned long long fix63(float r) {
  const uint32_t b = __float_as_uint(r);
  const int e = static_cast<int>((b >> 23) & 0xFFu);
  if (e == 0) return 0ull;
  const unsigned long long m = (b & 0x7FFFFFu) | 0x800000u;  // r = m * 2^(e - 150)
  const int sh = e - 87;
  if (sh >= 0) return m << sh;
  return -sh < 24 ? (m >> (-sh)) : 0ull;
}

// floor(r * 2^44) for a float r in [0, 1] (integer operations only): the unit
// of the per-key masses of the histogram statistics, whose sums over at most
// 2^18 elements stay below 2^62.
__device__ __forceinline__ unsigned long long fix44(float r) {
  const uint32_t b = __float_as_uint(r);
  const int e = static_cast<int>((b >> 23) & 0xFFu);
  if (e == 0) return 0ull;
  const unsigned long long m = (b & 0x7FFFFFu) | 0x800000u;  // r = m * 2^(e - 150)
  const int sh = e - 106;
  if (sh >= 0) return m << sh;
  return -sh < 24 ? (m >> (-sh)) : 0ull;
}

__device__ __forceinline__ unsigned long long warp_inclusive_scan_u64(unsigned long long v) {
  const int l = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long t = __shfl_up_sync(0xffffffffu, v, o);
    if (l >= o) v += t;
  }
  return v;
}

// ---------------------------------------------------------------- 128-bit fixed point
// Draw weights as exact integers in units of 2^-116: a float r in [0, 2) is
// exact down to 2^-93 and truncated below; sums of up to 2^11 times the
// largest weight stay below 2^128.  Sums are order-independent, so the
// inverse-CDF walk finds the same crossing as the scans.
typedef unsigned __int128 u128;

__device__ __forceinline__ u128 fix116(float r) {
  const uint32_t b = __float_as_uint(r);
  const int e = static_cast<int>((b >> 23) & 0xFFu);
  if (e == 0) return 0;
  const u128 m = (b & 0x7FFFFFu) | 0x800000u;                // value = m * 2^(e - 150)
  const int sh = e - 34;
  if (sh >= 0) return m << sh;
  return -sh < 24 ? (m >> (-sh)) : static_cast<u128>(0);
}

// L2 load (bypassing L1) of a 16-byte aligned 128-bit value.
__device__ __forceinline__ u128 ldcg_u128(const u128 *p) {
  const ulonglong2 v = __ldcg(reinterpret_cast<const ulonglong2 *>(p));
  return (static_cast<u128>(v.y) << 64) | v.x;
}

// floor(ku * Z / 2^24) for a 24-bit ku.
__device__ __forceinline__ u128 scale_u24(unsigned long long ku, u128 Z) {
  const u128 a = static_cast<u128>(ku) * static_cast<unsigned long long>(Z >> 64);
  const u128 b = static_cast<u128>(ku) * static_cast<unsigned long long>(Z);
  return (a << 40) + (b >> 24);
}

__device__ __forceinline__ u128 shfl_u128(u128 v, int src) {
  const unsigned long long lo = __shfl_sync(0xffffffffu, static_cast<unsigned long long>(v), src);
  const unsigned long long hi = __shfl_sync(0xffffffffu, static_cast<unsigned long long>(v >> 64), src);
  return (static_cast<u128>(hi) << 64) | lo;
}
// A + beta * B for two fixed-point (2^-116 units) sums and a small beta
// (|beta| < 2^-13) given as round(beta * 2^56), in signed 128-bit integers:
// B is shifted right by 40 bits first (its low bits are below 2^-76 and beta
// scales them further), so the product stays below 2^120.
typedef __int128 i128;
__device__ __forceinline__ i128 comb(u128 a, u128 b, long long beta56) {
  return static_cast<i128>(a) + ((static_cast<i128>(b >> 40) * beta56) >> 16);
}
// The same for 2^-63 sums (b < 2^64, |beta56| < 2^42: the product fits).
__device__ __forceinline__ i128 comb63(unsigned long long a, unsigned long long b,
                                       long long beta56) {
  return static_cast<i128>(a) + ((static_cast<i128>(b) * beta56) >> 56);
}

__device__ __forceinline__ u128 shfl_up_u128(u128 v, int o) {
  const unsigned long long lo = __shfl_up_sync(0xffffffffu, static_cast<unsigned long long>(v), o);
  const unsigned long long hi = __shfl_up_sync(0xffffffffu, static_cast<unsigned long long>(v >> 64), o);
  return (static_cast<u128>(hi) << 64) | lo;
}
__device__ __forceinline__ u128 shfl_xor_u128(u128 v, int o) {
  const unsigned long long lo = __shfl_xor_sync(0xffffffffu, static_cast<unsigned long long>(v), o);
  const unsigned long long hi = __shfl_xor_sync(0xffffffffu, static_cast<unsigned long long>(v >> 64), o);
  return (static_cast<u128>(hi) << 64) | lo;
}

// Exclusive prefix sum of one u128 per thread over the block, in thread order.
__device__ __forceinline__ u128 warp_inclusive_scan_u128(u128 v) {
  const int l = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const u128 t = shfl_up_u128(v, o);
    if (l >= o) v += t;
  }
  return v;
}

template <int NT>
__device__ __forceinline__ u128 block_exclusive_scan_u128(u128 v, u128 *red, u128 *total) {
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  const u128 inc = warp_inclusive_scan_u128(v);
  __syncthreads();
  if (l == 31) red[w] = inc;
  __syncthreads();
  u128 base = 0, tot = 0;
#pragma unroll
  for (int i = 0; i < NT / 32; ++i) {
    if (i < w) base += red[i];
    tot += red[i];
  }
  *total = tot;
  return base + inc - v;
}

// Block-wide sum of 128-bit values (all threads get it; `red` >= NT/32 entries).
template <int NT>
__device__ __forceinline__ u128 block_sum_u128(u128 v, u128 *red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += shfl_xor_u128(v, o);
  __syncthreads();
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  u128 t = 0;
#pragma unroll
  for (int i = 0; i < NT / 32; ++i) t += red[i];
  return t;
}

// floor(r * 2^52) for a float r in [0, 2), computed with integer operations
// only (exact: the float's 24-bit significand shifted into place).
__device__ __forceinline__ unsigned long long fix52(float r) {
  const uint32_t b = __float_as_uint(r);
  const int e = static_cast<int>((b >> 23) & 0xFFu);
  if (e == 0) return 0ull;                                   // zero / subnormal (< 2^-126)
  const unsigned long long m = (b & 0x7FFFFFu) | 0x800000u;  // value = m * 2^(e - 150)
  const int sh = e - 98;                                     // * 2^52
  if (sh >= 0) return m << sh;
  return -sh < 32 ? (m >> (-sh)) : 0ull;
}

// ---------------------------------------------------------------- PTX wrappers
__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// 16-byte async copy global -> shared; src_bytes = 0 zero-fills.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src, int src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src),
               "r"(src_bytes));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N));
}

__device__ __forceinline__ void ldmatrix_x4(uint32_t addr, uint32_t &r0, uint32_t &r1,
                                            uint32_t &r2, uint32_t &r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldmatrix_x4_trans(uint32_t addr, uint32_t &r0, uint32_t &r1,
                                                  uint32_t &r2, uint32_t &r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

// D = A * B + D, m16n8k16, bf16 inputs, fp32 accumulators.
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], const uint32_t (&a)[4],
                                               uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Transpose of an 8x8 b16 matrix held one 32-bit pair per lane (row lane/4,
// columns 2*(lane%4) and +1).
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x) {
  uint32_t r;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;\n" : "=r"(r) : "r"(x));
  return r;
}

// 2^x with the SFU's approximate exp2 (relative error ~2^-22, subnormal results
// flushed to zero).
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;\n" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// D = A * B + D, m16n8k16, f16 inputs, fp32 accumulators.
__device__ __forceinline__ void mma_f16_16816(float (&d)[4], const uint32_t (&a)[4],
                                              uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;\n" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// Two E4M3 codes (the lower byte is the lower element) -> f16x2; exact, since
// every E4M3 value is an f16 value.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two_codes) {
  uint32_t r;
  const uint16_t x = static_cast<uint16_t>(two_codes);
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;\n" : "=r"(r) : "h"(x));
  return r;
}

// bf16x2 -> f16x2, round to nearest (exact for values inside the f16 range).
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t x) {
  return pack_f16x2(__uint_as_float(x << 16), __uint_as_float(x & 0xFFFF0000u));
}

__device__ __forceinline__ uint16_t f32_to_bf16_rn(float x) {
  uint16_t r;
  asm("cvt.rn.bf16.f32 %0, %1;\n" : "=h"(r) : "f"(x));
  return r;
}

// ---------------------------------------------------------------- expm1
// e^x - 1 with relative error ~1e-6 or better, cheaply: the Taylor series
// through x^8 for |x| < 0.35 (remainder below 6e-10 relative), else
// 2^(x log2 e) - 1 by the SFU exp2 (e^x is then at least 0.35 away from 1, so
// the exp2's 2^-22 relative error grows by at most 2.5x).
__device__ __forceinline__ float expm1_fast(float x) {
  if (fabsf(x) < 0.35f) {
    float p = 1.0f / 40320.0f;
    p = __fmaf_rn(p, x, 1.0f / 5040.0f);
    p = __fmaf_rn(p, x, 1.0f / 720.0f);
    p = __fmaf_rn(p, x, 1.0f / 120.0f);
    p = __fmaf_rn(p, x, 1.0f / 24.0f);
    p = __fmaf_rn(p, x, 1.0f / 6.0f);
    p = __fmaf_rn(p, x, 0.5f);
    p = __fmaf_rn(p, x, 1.0f);
    return __fmul_rn(p, x);
  }
  return __fsub_rn(fast_exp2(__fmul_rn(x, 1.4426950408889634f)), 1.0f);
}

// ---------------------------------------------------------------- residual weight
// max(0, q_hat - p_hat) at one token with relative (not absolute) accuracy, so
// that residuals of any total mass keep their normalized CDF.  In natural-log
// units, with the row maxima mq, mp, the rows' (kept-set) sums S of
// exp((l - max) / T) and
//   t = ((lp - lq) - (mp - mq)) / T,       L = ln(S_p / S_q),
// p_hat / q_hat = exp(t - L) and q_hat - p_hat = -q_hat expm1(t - L).  t - L is
// formed in float-float (the logit differences exactly) and rounded once, so
// a token whose two probabilities nearly agree still gets its small
// difference to fp32 relative accuracy.
struct ResidualFn {
  float mq, mp;          // row maxima (target, draft)
  FF dm;                 // mp - mq, exactly
  FF inv_t;              // 1 / T
  int unit_t;            // T == 1: t needs no scaling
  int exact_diff;        // fp32 logits: lp - lq taken exactly by two-sum
  float c_hi, c_lo;      // log2(e) / T (q_hat by the SFU exp2)
  FF L;                  // ln(S_p / S_q)
  float inv_sq;          // 1 / S_q: a common factor of every weight

  __device__ __forceinline__ float qhat(float lq) const {
    const float dl = __fsub_rn(lq, mq);
    return __fmul_rn(fast_exp2(__fmaf_rn(dl, c_hi, __fmul_rn(dl, c_lo))), inv_sq);
  }
  // t - Lx as a float, for finite lq and lp.
  __device__ __forceinline__ float arg(float lq, float lp, FF Lx) const {
    // bf16 logits: lp - lq is exact in fp32 unless their exponents differ by
    // more than 15 (then lq or lp is negligible next to the other)
    FF t = exact_diff ? two_sum(lp, -lq) : FF{__fsub_rn(lp, lq), 0.0f};
    const FF u = two_sum(t.hi, -dm.hi);
    t = FF{u.hi, __fadd_rn(u.lo, __fsub_rn(t.lo, dm.lo))};
    if (!unit_t) t = ff_mul(t, inv_t);
    const FF d = two_sum(t.hi, -Lx.hi);
    return __fadd_rn(d.hi, __fadd_rn(d.lo, __fsub_rn(t.lo, Lx.lo)));
  }
  __device__ __forceinline__ float operator()(float lq, float lp) const {
    if (lq == -INFINITY) return 0.0f;
    const float qh = qhat(lq);
    if (lp == -INFINITY) return qh;
    const float d = arg(lq, lp, L);
    return d < 0.0f ? __fmul_rn(qh, -expm1_fast(d)) : 0.0f;
  }
  // Parameters shared by both sampler paths (L and inv_sq set by the caller).
  __device__ __forceinline__ void init(float mq_, float mp_, float c_hi_, float c_lo_,
                                       FF inv_t_, int unit_t_, int exact_diff_) {
    mq = mq_;
    mp = mp_;
    dm = two_sum(mp_, -mq_);
    inv_t = inv_t_;
    unit_t = unit_t_;
    exact_diff = exact_diff_;
    c_hi = c_hi_;
    c_lo = c_lo_;
    L = FF{0.0f, 0.0f};
    inv_sq = 0.0f;
  }
};

// 1 / s of a positive float-float as a float-float (relative error near
// 2^-46): the rounded reciprocal and one correction step.
__device__ __forceinline__ FF ff_recip(FF s) {
  const float h = __frcp_rn(s.hi);
  float e = __fmaf_rn(-s.hi, h, 1.0f);
  e = __fmaf_rn(-s.lo, h, e);
  return quick_two_sum(h, __fmul_rn(e, h));
}

// ln(s) of a float-float s >= 1 as a float-float (absolute error near
// 2^-44): L0 = logf(s), then ln s = L0 + ln(1 + u) with u = s e^(-L0) - 1
// (|u| ~ 1e-6, e^(-L0) by exp2_ff), ln(1 + u) = u - u^2/2 (the u^3 term is
// below 2^-59).  No fp64: it runs at a small fraction of the fp32 rate here.
__device__ __forceinline__ FF ln_ff(FF s, const float2 *tab) {
  const float L0 = fmaxf(logf(s.hi), 0.0f);
  constexpr float kLog2eHi = 1.44269502162933349609375f, kLog2eLo = 1.925963033500011079e-08f;
  const FF p = two_prod(L0, kLog2eHi);
  const FF y = quick_two_sum(p.hi, __fmaf_rn(L0, kLog2eLo, p.lo));
  const FF e = exp2_ff(ff_neg(y), tab);
  const FF se = ff_mul(s, e);
  const FF u = quick_two_sum(__fsub_rn(se.hi, 1.0f), se.lo);      // se.hi - 1 is exact
  const FF lu = ff_add(u, ff_make(__fmul_rn(-0.5f, __fmul_rn(u.hi, u.hi))));
  return ff_add(FF{L0, 0.0f}, lu);
}

// ln(S_p / S_q) of two float-float sums >= 1 (row sums relative to the row
// maximum, whose own weight is 1), as a float-float.
__device__ __forceinline__ FF ln_ratio_ff(FF sp, FF sq, const float2 *tab) {
  return ff_add(ln_ff(sp, tab), ff_neg(ln_ff(sq, tab)));
}

}  // namespace sv

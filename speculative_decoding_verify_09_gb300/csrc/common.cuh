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

}  // namespace sv

// Modified rejection sampling for a padding-free batch (sm_103a).
//
// Method: "Accelerating Large Language Model Decoding with Speculative
// Sampling" (Chen et al.), section "Modified rejection sampling": accept draft
// x~ with probability min(1, q(x~)/p(x~)), left to right, stop at the first
// rejection and draw from (q - p)_+ ; if all K drafts pass, draw a bonus token
// from the last target row.  Same section: temperature / nucleus modify the
// probabilities before the scheme.  Batch without padding: EMS-SD abstract.
//
// Paths, chosen on the host (plan_sampler):
//  * Cluster path (bf16 or fp32, no nucleus, no top-k, T > 0, a row slice of
//    at most 512 vectors per CTA): one thread-block cluster of 8 CTAs per
//    sequence, every phase exchanged through distributed shared memory; a few
//    KB of shared memory per CTA, so in the fused step it runs beside the
//    attention's CTAs (see the cluster kernel).
//  * Window statistics (other bf16 rows: nucleus, top-k, greedy, per-sequence
//    parameters, long rows): one CTA per row counts the keys of a window below
//    the row maximum and takes every cut per distinct value (see the window
//    kernel); the last row of a sequence runs the accept tests.
//  * fp32 rows otherwise: chunked statistics (no nucleus: CTA (row, chunk),
//    the last chunk of a row merges) or one CTA per row with a nucleus search
//    over weight-exponent bins.
//  After the statistics, the draw kernel (per-sequence chunks of row n_i)
//  draws and, in the fused step, appends the accepted K/V rows.
//
// Precision: per-element weights 2^((l - lmax) log2(e)/T) in fp32 by the SFU's
// approximate exp2 (relative error ~2^-22); the accept test compares
// u * p_hat < q_hat in fp32; the residual max(0, q_hat - p_hat) is evaluated
// with relative accuracy (ResidualFn: the logit differences in float-float,
// ln(S_p / S_q) from float-float sums); the inverse-CDF draws accumulate exact
// fixed-point weights, so the chosen index does not depend on the summation
// order.  No fp64 on the device (a small fraction of the fp32 rate here).  The
// near-tie windows of the decisions (1e-5) are far wider than these errors.
#include <algorithm>
#include <cmath>

#include "common.cuh"
#include "kernels.h"

namespace sv {

namespace {

constexpr int kSampNT = 512;          // threads per sampler CTA
constexpr int kSampNW = kSampNT / 32;
constexpr int kMaxTiles = 64;         // vectors per thread per row (bounds V)
constexpr int kCandCap = 4096;        // nucleus candidates held in shared memory

template <typename T> struct LT;
template <> struct LT<float> {
  static constexpr int EPV = 4;
  static constexpr int KEY_BITS = 32;
  static constexpr uint32_t NEG_INF_BITS = 0xFF800000u;
  __device__ static float val(uint32_t b) { return __uint_as_float(b); }
  __device__ static uint32_t key(uint32_t b) { return key_of_f32(b); }
  __device__ static uint32_t bits(float x) { return __float_as_uint(x); }
};
template <> struct LT<uint16_t> {
  static constexpr int EPV = 8;
  static constexpr int KEY_BITS = 16;
  static constexpr uint32_t NEG_INF_BITS = 0xFF80u;
  __device__ static float val(uint32_t b) { return bf16_bits_to_f32(b); }
  __device__ static uint32_t key(uint32_t b) { return key_of_bf16(b); }
  __device__ static uint32_t bits(uint16_t x) { return x; }
};

// One 16-byte vector v (elements v*EPV ..) of a row as raw bits; elements past
// V read as -inf (weight 0, lowest key).  Unaligned rows use scalar loads.
template <typename T>
__device__ __forceinline__ uint4 load_vec(const T *row, int V, int v, bool aligned) {
  constexpr int EPV = LT<T>::EPV;
  const int e0 = v * EPV;
  if (aligned && e0 + EPV <= V) return __ldg(reinterpret_cast<const uint4 *>(row + e0));
  uint32_t b[EPV];
#pragma unroll
  for (int i = 0; i < EPV; ++i)
    b[i] = (e0 + i < V) ? LT<T>::bits(__ldg(row + e0 + i)) : LT<T>::NEG_INF_BITS;
  if constexpr (EPV == 4) {
    return make_uint4(b[0], b[1], b[2], b[3]);
  } else {
    return make_uint4(b[0] | (b[1] << 16), b[2] | (b[3] << 16), b[4] | (b[5] << 16),
                      b[6] | (b[7] << 16));
  }
}

template <typename T>
__device__ __forceinline__ void unpack(const uint4 raw, uint32_t (&b)[LT<T>::EPV]) {
  if constexpr (LT<T>::EPV == 4) {
    b[0] = raw.x; b[1] = raw.y; b[2] = raw.z; b[3] = raw.w;
  } else {
    const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      b[2 * i] = w[i] & 0xFFFFu;
      b[2 * i + 1] = w[i] >> 16;
    }
  }
}

// Bits of element e (0 <= e < EPV) of a loaded vector, without indexing a
// local array (a dynamic index would move the vector to local memory).
template <typename T>
__device__ __forceinline__ uint32_t elem_bits(const uint4 raw, int e) {
  if constexpr (LT<T>::EPV == 4) {
    return e < 2 ? (e == 0 ? raw.x : raw.y) : (e == 2 ? raw.z : raw.w);
  } else {
    const int q = e >> 1;
    const uint32_t w = q < 2 ? (q == 0 ? raw.x : raw.y) : (q == 2 ? raw.z : raw.w);
    return (e & 1) ? (w >> 16) : (w & 0xFFFFu);
  }
}

template <typename T>
__device__ __forceinline__ void load_bits(const T *row, int V, int v, bool aligned,
                                          uint32_t (&b)[LT<T>::EPV]) {
  unpack<T>(load_vec<T>(row, V, v, aligned), b);
}

constexpr int kRowSmemBytes = 64 * 1024;  // a row up to this size is cached in smem
constexpr int kStream = 4;                 // vectors per thread loaded together when streaming

// A logits row as seen by one CTA: vector v = k * kSampNT + tid for k = 0..
// A row of at most kRowSmemBytes is copied once from HBM into shared memory
// (cp.async, all copies in flight together) and every pass reads it there;
// a longer row is streamed from L2 on every pass in unrolled batches.
template <typename T>
struct RowPass {
  const T *row;
  const uint4 *srow;   // shared-memory copy (cached rows)
  int V, NV;
  bool aligned, cached;

  __device__ __forceinline__ void init(const T *r, int v_, uint4 *smem_row) {
    row = r;
    V = v_;
    NV = (V + LT<T>::EPV - 1) / LT<T>::EPV;
    aligned = (reinterpret_cast<uintptr_t>(r) & 15) == 0;
    cached = NV * 16 <= kRowSmemBytes;
    srow = smem_row;
    if (cached) {
      for (int v = threadIdx.x; v < NV; v += kSampNT) {
        if (aligned && (v + 1) * LT<T>::EPV <= V)
          cp_async16(smem_u32(smem_row + v), row + v * LT<T>::EPV, 16);
        else
          smem_row[v] = load_vec<T>(row, V, v, aligned);
      }
      cp_async_commit();
      cp_async_wait<0>();
      __syncthreads();
    }
  }

  // f(bits[EPV]) for every vector this thread owns, in increasing v.
  template <typename F>
  __device__ __forceinline__ void each(F &&f) const {
    each_v([&](int, const uint32_t (&b)[LT<T>::EPV]) { f(b); });
  }

  // f(v, bits[EPV]) for every vector v this thread owns, in increasing v.
  template <typename F>
  __device__ __forceinline__ void each_v(F &&f) const {
    constexpr int EPV = LT<T>::EPV;
    if (cached) {
      for (int v = threadIdx.x; v < NV; v += kSampNT) {
        uint32_t b[EPV];
        unpack<T>(srow[v], b);
        f(v, b);
      }
    } else {
      for (int base = 0; base < NV; base += kStream * kSampNT) {
        uint4 tmp[kStream];
#pragma unroll
        for (int k = 0; k < kStream; ++k) {
          const int v = base + k * kSampNT + threadIdx.x;
          if (v < NV) tmp[k] = load_vec<T>(row, V, v, aligned);
        }
#pragma unroll
        for (int k = 0; k < kStream; ++k) {
          if (base + k * kSampNT + static_cast<int>(threadIdx.x) < NV) {
            uint32_t b[EPV];
            unpack<T>(tmp[k], b);
            f(base + k * kSampNT + static_cast<int>(threadIdx.x), b);
          }
        }
      }
    }
  }
};

// Block-wide float-float sums of N values per thread in one pass: every
// thread adds the per-warp partials in the same order, so all get the same
// result (one barrier; `red` must not be reused before the next barrier).
template <int N>
__device__ __forceinline__ void block_sum_ff(FF (&v)[N], FF *red) {
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
#pragma unroll
  for (int k = 0; k < N; ++k) v[k] = warp_sum_ff(v[k]);
  if (l == 0) {
#pragma unroll
    for (int k = 0; k < N; ++k) red[k * kSampNW + w] = v[k];
  }
  __syncthreads();
#pragma unroll
  for (int k = 0; k < N; ++k) {
    FF t = red[k * kSampNW];
#pragma unroll
    for (int i = 1; i < kSampNW; ++i) t = ff_add(t, red[k * kSampNW + i]);
    v[k] = t;
  }
}

// exp((l - lmax) / T) in fp32, with c = log2(e) / T split as c_hi + c_lo, by
// the SFU's exp2 (relative error ~2^-22).  Explicit round-to-nearest
// intrinsics: every pass recomputes identical bits.
struct WeightFn {
  float lmax, c_hi, c_lo;
  __device__ __forceinline__ float operator()(float l) const {
    if (l == -INFINITY) return 0.0f;
    const float dl = __fsub_rn(l, lmax);
    return fast_exp2(__fmaf_rn(dl, c_hi, __fmul_rn(dl, c_lo)));
  }
};

struct SampParams {
  sv_sample_args a;
  SamplerWs ws;
  SamplerPlan plan;
  int do_append;
  AppendView app;
  float c_hi, c_lo;   // log2(e)/T as two floats
  float it_hi, it_lo; // 1/T as two floats
  int pdl_secondary;  // launched early behind another grid (see PdlTail)
  uint32_t stream;    // Philox counter word 3: 0 verify, 1 draft-token draws
  float2 exp2tab[kExp2Tab];   // 2^(j/64), j = -32..32, float-float (exp2_ff)
};

// A launch that may start before the previous grid on its stream has finished
// (programmatic dependent launch) must not finish before it: every exit path
// of such a kernel waits for the previous grid first.
struct PdlTail {
  int on;
  __device__ __forceinline__ ~PdlTail() {
    if (on) asm volatile("griddepcontrol.wait;\n" ::: "memory");
  }
};

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n"
               "barrier.cluster.wait.acquire.aligned;\n" ::: "memory");
}

// Generic address of `p` in the shared memory of cluster CTA `rank`.
template <typename X>
__device__ __forceinline__ X *dsmem(X *p, uint32_t rank) {
  uint64_t r;
  asm volatile("mapa.u64 %0, %1, %2;" : "=l"(r) : "l"(reinterpret_cast<uint64_t>(p)), "r"(rank));
  return reinterpret_cast<X *>(r);
}

struct SampSmem {
  float2 exp2tab[kExp2Tab];   // 2^(j/64) as float-float (accurate kept-set sums)
  float tconst[4];            // log2(e)/T and 1/T of the row, float pairs
  FF red[2][8 * kSampNW];     // double-buffered float-float partials
  float redf[32];
  unsigned long long red64[32];
  int bcast[8];
  unsigned long long sel[4];              // broadcast of a select step
  union {
    struct {                              // nucleus cut: candidates
      uint32_t cand_key[kCandCap];
      float cand_w[kCandCap];
    };
    unsigned long long hist[kSampNW][256];  // top-k select: per-warp histograms
  };
};

constexpr size_t kSmemRowOff = (sizeof(SampSmem) + 127) / 128 * 128;

// Block-row offset of sequence i.  A null cu_q means one row per sequence
// (K_i = 0), the layout of a draft-token draw.
__device__ __forceinline__ int cuq(const sv_sample_args &a, int i) {
  return a.cu_q ? a.cu_q[i] : i;
}

// Validity of sequence i's row bookkeeping against the host bounds.
__device__ __forceinline__ bool seq_rows_ok(const sv_sample_args &a, int i) {
  const int r0 = cuq(a, i), r1 = cuq(a, i + 1);
  const int Ri = r1 - r0;
  return r0 >= i && Ri >= 1 && Ri <= a.max_q_rows && r1 <= a.num_rows &&
         (r1 - (i + 1)) <= a.num_rows - a.batch;
}

// Largest i with key_of(i) <= x over a monotone array (binary search).
__device__ __forceinline__ int seq_of_target_row(const int32_t *cu_q, int B, int r) {
  int lo = 0, hi = B - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (cu_q[mid] <= r) lo = mid; else hi = mid - 1;
  }
  return lo;
}
__device__ __forceinline__ int seq_of_draft_row(const int32_t *cu_q, int B, int pr) {
  int lo = 0, hi = B - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (cu_q[mid] - mid <= pr) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// --------------------------------------------------------------------------
// Nucleus cut: the largest key tau such that the weight of {key >= tau} is at
// least top_p * S (ties kept together).  Coarse pass over weight-exponent bins
// finds the bin holding the cut; the exact bitwise search then runs over that
// bin's elements in shared memory, with the heavier bins' mass added (or, if
// the bin has too many elements, over the whole row).
// --------------------------------------------------------------------------
template <typename T>
__device__ void nucleus_cut(const RowPass<T> &rp, const WeightFn &wf0, uint32_t kmin, double S,
                            float top_p, SampSmem &sm, uint32_t &tau_out, double &ssum_out) {
  constexpr int EPV = LT<T>::EPV;
  const int tid = threadIdx.x;
  const double target = static_cast<double>(top_p) * S;
  // weights of the elements kept by top-k (keys below kmin weigh 0)
  struct Masked {
    WeightFn f;
    uint32_t kmin;
    __device__ __forceinline__ float operator()(uint32_t bits) const {
      return LT<T>::key(bits) < kmin ? 0.0f : f(LT<T>::val(bits));
    }
  } wb{wf0, kmin};

  // coarse bins: bin b = min((127 - biased_exp(w)) / 4, 7)
  float acc[8];
#pragma unroll
  for (int b = 0; b < 8; ++b) acc[b] = 0.0f;
  rp.each([&](const uint32_t (&bits)[EPV]) {
#pragma unroll
    for (int e = 0; e < EPV; ++e) {
      const float x = wb(bits[e]);
      const int ex = 127 - static_cast<int>((__float_as_uint(x) >> 23) & 0xFFu);
      const int b = min(max(ex, 0) >> 2, 7);
#pragma unroll
      for (int k = 0; k < 8; ++k) acc[k] += (b == k) ? x : 0.0f;
    }
  });
  FF bins[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) bins[k] = ff_make(acc[k]);
  block_sum_ff<8>(bins, sm.red[0]);
  // Candidates: bins klo..kb around the cut, where klo is the first bin whose
  // cumulative mass reaches top_p * S * (1 - 1e-5) and kb the first reaching
  // (1 + 1e-5) (the float bin sums are far more accurate than that), so the
  // heavier bins' mass `heavy` is surely below the target and bins up to kb
  // surely reach it.  A heavier bin holds larger weights, hence larger logits
  // and keys, than every candidate, so for a probe key inside the candidates'
  // range the mass at or above it is heavy plus the candidates' at or above
  // it; for probes above that range heavy alone stays below the target, and
  // for probes below it heavy plus every candidate reaches it: the exact
  // search takes the same decisions as over the whole row.
  const FF tgt_safe = ff_from_double(target * (1.0 + 1e-5));
  const FF tgt_low = ff_from_double(target * (1.0 - 1e-5));
  FF cum = ff_make(0.0f), heavy = ff_make(0.0f);
  int kb = 7, klo = 7;
#pragma unroll
  for (int k = 0; k < 7; ++k) {
    const FF next = ff_add(cum, bins[k]);
    if (klo == 7 && ff_ge(next, tgt_low)) {
      klo = k;
      heavy = cum;
    }
    if (kb == 7 && ff_ge(next, tgt_safe)) kb = k;
    cum = next;
  }
  if (klo == 7) heavy = cum;          // the cut lies in the tail bin
  auto is_cand = [&](float x) {
    const int ex = 127 - static_cast<int>((__float_as_uint(x) >> 23) & 0xFFu);
    const int b = min(max(ex, 0) >> 2, 7);
    return b >= klo && b <= kb;
  };
  int mine = 0;
  rp.each([&](const uint32_t (&bits)[EPV]) {
#pragma unroll
    for (int e = 0; e < EPV; ++e) mine += is_cand(wb(bits[e])) ? 1 : 0;
  });
  unsigned long long total = 0;
  const unsigned long long off =
      block_exclusive_scan_u64<kSampNT>(static_cast<unsigned long long>(mine), sm.red64, &total);
  const bool in_smem = total <= static_cast<unsigned long long>(kCandCap);
  if (in_smem) {
    int o = static_cast<int>(off);
    rp.each([&](const uint32_t (&bits)[EPV]) {
#pragma unroll
      for (int e = 0; e < EPV; ++e) {
        const float x = wb(bits[e]);
        if (is_cand(x)) {
          sm.cand_key[o] = LT<T>::key(bits[e]);
          sm.cand_w[o] = x;
          ++o;
        }
      }
    });
  }
  __syncthreads();
  const int C = static_cast<int>(total);
  // this thread's part of the weight of {key >= cand}
  auto partial = [&](uint32_t cand) {
    float sum = 0.0f;
    if (in_smem) {
      for (int c = tid; c < C; c += kSampNT)
        if (sm.cand_key[c] >= cand) sum += sm.cand_w[c];
    } else {
      rp.each([&](const uint32_t (&bits)[EPV]) {
#pragma unroll
        for (int e = 0; e < EPV; ++e)
          if (LT<T>::key(bits[e]) >= cand) sum += wb(bits[e]);
      });
    }
    return sum;
  };
  // bitwise search, one barrier per bit (double-buffered partial sums)
  const FF tgt = ff_from_double(target);
  uint32_t tau = 0;
  int buf = 1;
  for (int bit = LT<T>::KEY_BITS - 1; bit >= 0; --bit) {
    const uint32_t cand = tau | (1u << bit);
    FF W[1] = {ff_make(partial(cand))};
    block_sum_ff<1>(W, sm.red[buf]);
    if (in_smem) W[0] = ff_add(W[0], heavy);
    if (ff_ge(W[0], tgt)) tau = cand;
    buf ^= 1;
  }
  FF ss[1] = {ff_make(partial(tau))};
  block_sum_ff<1>(ss, sm.red[buf]);
  if (in_smem) ss[0] = ff_add(ss[0], heavy);
  ssum_out = ff_to_double(ss[0]);
  tau_out = tau;
}

// --------------------------------------------------------------------------
// Top-k key: the largest order-preserving key tau with at least k elements at
// or above it (the k-th largest, ties kept), by a radix select over key bytes
// from the top: per pass a 256-bin count of the elements matching the bytes
// fixed so far (one private histogram per warp, added per bin afterwards),
// then the largest bin whose upper count still reaches k.
// --------------------------------------------------------------------------
template <typename T>
__device__ uint32_t topk_key(const RowPass<T> &rp, int k, SampSmem &sm) {
  constexpr int EPV = LT<T>::EPV;
  constexpr int KB = LT<T>::KEY_BITS;
  const int tid = threadIdx.x, w = tid >> 5;
  const unsigned long long target = static_cast<unsigned long long>(k);
  unsigned long long *myh = sm.hist[w];
  uint32_t prefix = 0;               // key bits fixed so far
  unsigned long long above = 0;      // count of elements above the prefix range
  for (int fixed = 0; fixed < KB; fixed += 8) {
    const int shift = KB - fixed - 8;
    for (int b = tid; b < kSampNW * 256; b += kSampNT) (&sm.hist[0][0])[b] = 0ull;
    __syncthreads();
    rp.each([&](const uint32_t (&bits)[EPV]) {
#pragma unroll
      for (int e = 0; e < EPV; ++e) {
        const uint32_t key = LT<T>::key(bits[e]);
        if (fixed > 0 && (key >> (shift + 8)) != prefix) continue;
        atomicAdd(&myh[(key >> shift) & 255u], 1ull);
      }
    });
    __syncthreads();
    for (int b = tid; b < 256; b += kSampNT) {          // add the warps' histograms
      unsigned long long t = 0;
#pragma unroll
      for (int x = 0; x < kSampNW; ++x) t += sm.hist[x][b];
      sm.hist[0][b] = t;
    }
    __syncthreads();
    if (tid < 32) {                  // warp 0: the largest bin whose upper count reaches k
      unsigned long long h[8], own = 0;
#pragma unroll
      for (int q = 0; q < 8; ++q) { h[q] = sm.hist[0][8 * tid + q]; own += h[q]; }
      unsigned long long suf = own;  // inclusive suffix over lanes >= tid
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const unsigned long long y = __shfl_down_sync(0xffffffffu, suf, o);
        if (tid + o < 32) suf += y;
      }
      unsigned long long run = above + suf - own;
      int best = -1;
      unsigned long long best_above = 0;
#pragma unroll
      for (int q = 7; q >= 0; --q) {
        if (best < 0 && run + h[q] >= target) {
          best = 8 * tid + q;
          best_above = run;
        }
        run += h[q];
      }
      const unsigned hit = __ballot_sync(0xffffffffu, best >= 0);
      const int src = hit ? 31 - __clz(hit) : 0;        // the highest lane holds the largest bin
      best = __shfl_sync(0xffffffffu, best, src);
      best_above = __shfl_sync(0xffffffffu, best_above, src);
      if (tid == 0) {
        if (best < 0) { best = 0; best_above = above; }
        sm.sel[0] = (static_cast<unsigned long long>(prefix) << 8) | static_cast<unsigned>(best);
        sm.sel[1] = best_above;
      }
    }
    __syncthreads();
    prefix = static_cast<uint32_t>(sm.sel[0]);
    above = sm.sel[1];
    __syncthreads();
  }
  return prefix;
}

// --------------------------------------------------------------------------
// Probabilities.  q_hat(l) = [key(l) >= tau] * w(l) / S with w(l) = exp((l -
// lmax)/T) in fp32 and 1/S held as a float-float pair (no per-thread fp64).
// --------------------------------------------------------------------------
struct RowProb {
  WeightFn wf;
  uint32_t tau;
  float inv_hi, inv_lo;
  int amax;            // >= 0: greedy row, one-hot at this index
};

__device__ __forceinline__ RowProb rowprob_of(const RowStats *st) {
  RowProb r;
  r.wf = WeightFn{__ldcg(&st->lmax), __ldcg(&st->c_hi), __ldcg(&st->c_lo)};
  r.tau = __ldcg(&st->tau_key);
  r.inv_hi = __ldcg(&st->inv_hi);
  r.inv_lo = __ldcg(&st->inv_lo);
  r.amax = __ldcg(&st->amax);
  return r;
}

// q_hat of vocabulary index x whose logit has the bits `bits`.
template <typename T>
__device__ __forceinline__ float row_prob(const RowProb &rp, uint32_t bits, int x) {
  if (rp.amax >= 0) return x == rp.amax ? 1.0f : 0.0f;
  if (LT<T>::key(bits) < rp.tau) return 0.0f;
  const float w = rp.wf(LT<T>::val(bits));
  return __fmaf_rn(w, rp.inv_hi, __fmul_rn(w, rp.inv_lo));
}

// Draw weight of vocabulary index x: mode 0 the residual max(0, q_hat -
// p_hat) (with relative accuracy, see ResidualFn; exact 0 / 1 differences for
// greedy one-hot rows), mode 1 q_hat.
struct DrawWeight {
  RowProb pq, pp;
  ResidualFn rf;
  int mode;
  bool onehot;
  template <typename T>
  __device__ __forceinline__ float w(uint32_t bq, uint32_t bp, int x) const {
    if (mode != 0) return row_prob<T>(pq, bq, x);
    if (onehot) return fmaxf(__fsub_rn(row_prob<T>(pq, bq, x), row_prob<T>(pp, bp, x)), 0.0f);
    const float lq = LT<T>::key(bq) < pq.tau ? -INFINITY : LT<T>::val(bq);
    const float lp = LT<T>::key(bp) < pp.tau ? -INFINITY : LT<T>::val(bp);
    return rf(lq, lp);
  }
  template <typename T>
  __device__ __forceinline__ u128 fix(uint32_t bq, uint32_t bp, int x) const {
    return fix116(w<T>(bq, bp, x));
  }
};

// Finish a row's statistics (one thread): ssum and its float-float inverse,
// the row's log2(e)/T constant and, for a greedy row, its argmax.
__device__ __forceinline__ void write_stats(RowStats *st, float lmax, uint32_t tau, bool valid,
                                            double ssum, float c_hi, float c_lo, int amax,
                                            FF acc, float it_hi, float it_lo) {
  RowStats o;
  o.lmax = lmax;
  o.tau_key = tau;
  o.valid = valid ? 1u : 0u;
  const double inv = valid && ssum > 0.0 ? 1.0 / ssum : 0.0;
  o.inv_hi = static_cast<float>(inv);
  o.inv_lo = static_cast<float>(inv - static_cast<double>(o.inv_hi));
  o.amax = valid ? amax : -1;
  o.c_hi = c_hi;
  o.c_lo = c_lo;
  o.acc_hi = acc.hi;
  o.acc_lo = acc.lo;
  o.it_hi = it_hi;
  o.it_lo = it_lo;
  *st = o;
}

// --------------------------------------------------------------------------
// Accept tests of sequence i (warp 0 of the CTA that completed its rows):
// lane j tests draft j+1 against target row j and draft row j with the
// acceptance uniform of token index L_i + j + 1.  Writes num_accepted, the
// accepted drafts and -1 elsewhere (the drawn token comes in the draw phase).
// --------------------------------------------------------------------------
template <typename T>
__device__ void accept_sequence(const SampParams &P, int i) {
  const sv_sample_args &a = P.a;
  const int lane = threadIdx.x & 31;
  const int V = a.vocab, R = static_cast<int>(a.num_rows);
  const int r0 = cuq(a, i), K = cuq(a, i + 1) - r0 - 1, p0 = r0 - i;
  const int L = a.kv_len[i];
  const RowStats *st = P.ws.stats;
  // pair j (target row j, draft row j; the bonus row alone at j = K) is valid
  int ok = 1;
  if (lane <= K) ok = __ldcg(&st[r0 + lane].valid) != 0;
  if (lane < K) ok = ok && (__ldcg(&st[R + p0 + lane].valid) != 0);
  const unsigned badm = __ballot_sync(0xffffffffu, lane <= K && !ok);
  if (L < 0) {
    if (lane <= K) a.out_tokens[r0 + lane] = -1;
    if (lane == 0) {
      a.num_accepted[i] = -1;
      set_status(a.dev_status, SV_DEV_BAD_LENGTH);
    }
    return;
  }
  const long long sid = a.seq_ids ? a.seq_ids[i] : static_cast<long long>(i);
  const uint32_t k0 = static_cast<uint32_t>(a.seed), k1 = static_cast<uint32_t>(a.seed >> 32);
  const uint32_t sid_lo = static_cast<uint32_t>(static_cast<unsigned long long>(sid));
  const uint32_t sid_hi = static_cast<uint32_t>(static_cast<unsigned long long>(sid) >> 32);
  bool rej = false, bad = false;
  int d = 0;
  if (lane < K && ok) {
    d = a.draft_tokens[p0 + lane];
    if (d < 0 || d >= V) {
      rej = bad = true;
    } else {
      const T *tgt = static_cast<const T *>(a.target_logits);
      const T *drf = static_cast<const T *>(a.draft_logits);
      const RowProb pq = rowprob_of(&st[r0 + lane]);
      const RowProb pp = rowprob_of(&st[R + p0 + lane]);
      const float qh = row_prob<T>(pq, LT<T>::bits(tgt[static_cast<int64_t>(r0 + lane) * V + d]), d);
      const float ph = row_prob<T>(pp, LT<T>::bits(drf[static_cast<int64_t>(p0 + lane) * V + d]), d);
      const U4 w = philox4x32_10(U4{static_cast<uint32_t>(L + lane + 1), sid_lo, sid_hi, P.stream}, k0, k1);
      const float u = static_cast<float>(u24(w.x)) * 0x1p-24f;          // exact
      rej = !(__fmul_rn(u, ph) < qh);
    }
  }
  const unsigned rm = __ballot_sync(0xffffffffu, rej);
  const unsigned bm = __ballot_sync(0xffffffffu, bad);
  // the loop stops at the first rejection or the first invalid pair; only
  // rows it reaches are used, so an invalid pair fails the sequence only if
  // no rejection comes before it
  const int first_rej = rm ? (__ffs(rm) - 1) : K;
  const int first_bad = badm ? (__ffs(badm) - 1) : K + 1;
  const int n = first_bad <= first_rej ? -1 : first_rej;
  if (lane <= K) a.out_tokens[r0 + lane] = (n >= 0 && lane < n) ? d : -1;
  if (lane == 0) {
    a.num_accepted[i] = n;
    if (n < 0) set_status(a.dev_status, SV_DEV_NONFINITE);
    else if (n < K && ((bm >> n) & 1u)) set_status(a.dev_status, SV_DEV_BAD_TOKEN);
  }
}

// The CTA that finished the last row of sequence i runs its accept tests.
template <typename T>
__device__ __forceinline__ void arrive_sequence(const SampParams &P, int i, int *flag) {
  if (threadIdx.x == 0) {
    __threadfence();
    const int nrows = 2 * (cuq(P.a, i + 1) - cuq(P.a, i)) - 1;
    const unsigned old = atomicInc(&P.ws.seq_cnt1[i], static_cast<unsigned>(nrows - 1));
    *flag = old == static_cast<unsigned>(nrows - 1) ? 1 : 0;
  }
  __syncthreads();
  if (*flag && threadIdx.x < 32) {
    __threadfence();
    accept_sequence<T>(P, i);
  }
}

__device__ __forceinline__ int row_seq(const sv_sample_args &a, int r, const void *&base,
                                       int64_t &row_off) {
  const int R = static_cast<int>(a.num_rows);
  if (r < R) {
    row_off = static_cast<int64_t>(r) * a.vocab;
    base = a.target_logits;
    return a.cu_q ? seq_of_target_row(a.cu_q, a.batch, r) : r;
  }
  row_off = static_cast<int64_t>(r - R) * a.vocab;
  base = a.draft_logits;
  return seq_of_draft_row(a.cu_q, a.batch, r - R);
}

// --------------------------------------------------------------------------
// Phase 1a (no nucleus): CTA (row, chunk) computes the chunk's max and the sum
// of exp((l - m_chunk)/T); the last chunk of a row merges them, the last row
// of a sequence runs the accept tests.
// --------------------------------------------------------------------------
constexpr int kStatNT = 256;
constexpr int kStatVec = 4;          // vectors per thread per chunk

template <typename T>
__global__ void __launch_bounds__(kStatNT) stats_chunk_kernel(const SampParams P) {
  const PdlTail tail{P.pdl_secondary};
  constexpr int EPV = LT<T>::EPV;
  constexpr int NW = kStatNT / 32;
  __shared__ float redf[NW];
  __shared__ FF redff[NW], redacc[NW];
  __shared__ float2 tab[kExp2Tab];
  __shared__ int flag[2];
  exp2_table_fill(tab, P.exp2tab);
  const sv_sample_args &a = P.a;
  const int NCH = P.plan.stat_chunks;
  const int r = blockIdx.x / NCH, c = blockIdx.x - r * NCH;
  const int tid = threadIdx.x, w = tid >> 5, l = tid & 31;
  const void *base;
  int64_t off;
  const int i = row_seq(a, r, base, off);
  if (!seq_rows_ok(a, i)) {
    if (tid == 0) set_status(a.dev_status, SV_DEV_BAD_LENGTH);
    return;
  }
  const T *row = static_cast<const T *>(base) + off;
  const int V = a.vocab, NV = (V + EPV - 1) / EPV;
  const int per = (NV + NCH - 1) / NCH;
  const int v0 = c * per, v1 = min(NV, v0 + per);
  const bool aligned = (reinterpret_cast<uintptr_t>(row) & 15) == 0;
  uint4 vec[kStatVec];
#pragma unroll
  for (int k = 0; k < kStatVec; ++k) {
    const int v = v0 + k * kStatNT + tid;
    if (v < v1) vec[k] = load_vec<T>(row, V, v, aligned);
  }
  float mx = -INFINITY;
  int bad = 0;
#pragma unroll
  for (int k = 0; k < kStatVec; ++k) {
    if (v0 + k * kStatNT + tid < v1) {
      uint32_t b[EPV];
      unpack<T>(vec[k], b);
#pragma unroll
      for (int e = 0; e < EPV; ++e) {
        const float x = LT<T>::val(b[e]);
        bad |= (x != x) || (x == INFINITY);
        mx = fmaxf(mx, x);
      }
    }
  }
  // chunks longer than kStatVec * kStatNT vectors stream the rest
  for (int v = v0 + kStatVec * kStatNT + tid; v < v1; v += kStatNT) {
    uint32_t b[EPV];
    load_bits<T>(row, V, v, aligned, b);
#pragma unroll
    for (int e = 0; e < EPV; ++e) {
      const float x = LT<T>::val(b[e]);
      bad |= (x != x) || (x == INFINITY);
      mx = fmaxf(mx, x);
    }
  }
  bad = __syncthreads_or(bad);
  mx = warp_max(mx);
  if (l == 0) redf[w] = mx;
  __syncthreads();
  mx = redf[0];
#pragma unroll
  for (int k = 1; k < NW; ++k) mx = fmaxf(mx, redf[k]);
  // chunk sum of exp((l - mx)/T), Kahan per thread, float-float across threads
  const WeightFn wf{mx, P.c_hi, P.c_lo};
  const FF cc{P.c_hi, P.c_lo};
  float sum = 0.0f, comp = 0.0f;
  FF acc = ff_make(0.0f);
  auto kahan = [&](const uint32_t (&b)[EPV]) {
#pragma unroll
    for (int e = 0; e < EPV; ++e) {
      const float l = LT<T>::val(b[e]);
      const float y = __fsub_rn(wf(l), comp);
      const float t = __fadd_rn(sum, y);
      comp = __fsub_rn(__fsub_rn(t, sum), y);
      sum = t;
      if (l != -INFINITY) acc = ff_add(acc, exp2_ff(ff_mul(two_sum(l, -mx), cc), tab));
    }
  };
  if (mx > -INFINITY) {
#pragma unroll
    for (int k = 0; k < kStatVec; ++k) {
      if (v0 + k * kStatNT + tid < v1) {
        uint32_t b[EPV];
        unpack<T>(vec[k], b);
        kahan(b);
      }
    }
    for (int v = v0 + kStatVec * kStatNT + tid; v < v1; v += kStatNT) {
      uint32_t b[EPV];
      load_bits<T>(row, V, v, aligned, b);
      kahan(b);
    }
  }
  FF f = warp_sum_ff(FF{sum, -comp});
  acc = warp_sum_ff(acc);
  if (l == 0) {
    redff[w] = f;
    redacc[w] = acc;
  }
  __syncthreads();
  if (tid == 0) {
    FF t = redff[0], ta = redacc[0];
    for (int k = 1; k < NW; ++k) {
      t = ff_add(t, redff[k]);
      ta = ff_add(ta, redacc[k]);
    }
    ChunkPart cp;
    cp.m = mx;
    cp.s_hi = t.hi;
    cp.s_lo = t.lo;
    cp.bad = bad ? 1u : 0u;
    cp.a_hi = ta.hi;
    cp.a_lo = ta.lo;
    P.ws.parts[static_cast<int64_t>(r) * NCH + c] = cp;
    __threadfence();
    const unsigned old = atomicInc(&P.ws.row_cnt[r], static_cast<unsigned>(NCH - 1));
    flag[0] = old == static_cast<unsigned>(NCH - 1) ? 1 : 0;
    if (flag[0]) {          // last chunk of the row: merge (max, sum) online
      __threadfence();
      float M = -INFINITY;
      uint32_t anybad = 0;
      const ChunkPart *parts = P.ws.parts + static_cast<int64_t>(r) * NCH;
      for (int k = 0; k < NCH; ++k) {
        M = fmaxf(M, __ldcg(&parts[k].m));
        anybad |= __ldcg(&parts[k].bad);
      }
      FF S = ff_make(0.0f), A = ff_make(0.0f);
      if (M > -INFINITY) {
        const WeightFn sc{M, P.c_hi, P.c_lo};
        for (int k = 0; k < NCH; ++k) {
          const float qm = __ldcg(&parts[k].m);
          if (qm == -INFINITY) continue;
          const float f = sc(qm);                        // exp((m_k - M)/T)
          S = ff_add(S, ff_add(FF{__fmul_rn(__ldcg(&parts[k].s_hi), f), 0.0f},
                               FF{__fmul_rn(__ldcg(&parts[k].s_lo), f), 0.0f}));
          const FF fa = exp2_ff(ff_mul(two_sum(qm, -M), cc), tab);
          A = ff_add(A, ff_mul(FF{__ldcg(&parts[k].a_hi), __ldcg(&parts[k].a_lo)}, fa));
        }
      }
      const bool valid = !anybad && M > -INFINITY;
      write_stats(&P.ws.stats[r], M, 0u, valid, ff_to_double(S), P.c_hi, P.c_lo, -1, A, P.it_hi,
                  P.it_lo);
    }
  }
  __syncthreads();
  if (flag[0]) arrive_sequence<T>(P, i, &flag[1]);
}

// --------------------------------------------------------------------------
// Phase 1b (nucleus, top-k, greedy, per-sequence parameters): one CTA per row.
// The row is read once from HBM into shared memory (or streamed from L2 when
// longer than 64 KB), then max, top-k key, sum and the nucleus cut run on chip.
// --------------------------------------------------------------------------
template <typename T>
__global__ void __launch_bounds__(kSampNT) stats_row_kernel(const SampParams P) {
  const PdlTail tail{P.pdl_secondary};
  extern __shared__ __align__(16) unsigned char smem_raw[];
  SampSmem &sm = *reinterpret_cast<SampSmem *>(smem_raw);
  const sv_sample_args &a = P.a;
  const int r = blockIdx.x;
  const int tid = threadIdx.x;
  const void *base;
  int64_t off;
  const int i = row_seq(a, r, base, off);
  if (!seq_rows_ok(a, i)) {
    if (tid == 0) set_status(a.dev_status, SV_DEV_BAD_LENGTH);
    return;
  }
  const T *row = static_cast<const T *>(base) + off;
  constexpr int EPV = LT<T>::EPV;
  exp2_table_fill(sm.exp2tab, P.exp2tab);
  RowPass<T> rp;
  rp.init(row, a.vocab, reinterpret_cast<uint4 *>(smem_raw + kSmemRowOff));  // the one HBM read
  float mx = -INFINITY;
  int bad = 0;
  rp.each([&](const uint32_t (&bits)[EPV]) {
#pragma unroll
    for (int e = 0; e < EPV; ++e) {
      const float x = LT<T>::val(bits[e]);
      bad |= (x != x) || (x == INFINITY);
      mx = fmaxf(mx, x);
    }
  });
  bad = __syncthreads_or(bad);
  mx = block_max_f<kSampNT>(mx, sm.redf);
  // this sequence's processing parameters (arrays override the scalars)
  const float Tr = a.temperatures ? a.temperatures[i] : a.temperature;
  const float tpr = a.top_ps ? a.top_ps[i] : a.top_p;
  const int tkr = a.top_ks ? a.top_ks[i] : a.top_k;
  const bool param_ok = Tr >= 0.0f && tpr > 0.0f && tkr >= 0;     // NaN fails the compares
  if (!param_ok && tid == 0) set_status(a.dev_status, SV_DEV_BAD_PARAM);
  const bool valid = param_ok && !bad && mx > -INFINITY;
  uint32_t tau = 0;
  double ssum = 0.0;
  FF acc = ff_make(0.0f);
  float c_hi = 0.0f, c_lo = 0.0f, it_hi = 0.0f, it_lo = 0.0f;
  int amax = -1;
  if (valid && Tr == 0.0f) {
    // greedy: one-hot at the lowest index holding the maximum
    float first = -static_cast<float>(a.vocab);
    rp.each_v([&](int v, const uint32_t (&bits)[EPV]) {
#pragma unroll
      for (int e = 0; e < EPV; ++e)
        if (LT<T>::val(bits[e]) == mx) first = fmaxf(first, -static_cast<float>(v * EPV + e));
    });
    __syncthreads();
    amax = static_cast<int>(-block_max_f<kSampNT>(first, sm.redf));
    ssum = 1.0;
  } else if (valid) {
    if (tid == 0) {                   // fp64 once per CTA
      const double c = 1.4426950408889634 / static_cast<double>(Tr);
      const double it = 1.0 / static_cast<double>(Tr);
      sm.tconst[0] = static_cast<float>(c);
      sm.tconst[1] = static_cast<float>(c - static_cast<double>(sm.tconst[0]));
      sm.tconst[2] = static_cast<float>(it);
      sm.tconst[3] = static_cast<float>(it - static_cast<double>(sm.tconst[2]));
    }
    __syncthreads();
    c_hi = sm.tconst[0];
    c_lo = sm.tconst[1];
    it_hi = sm.tconst[2];
    it_lo = sm.tconst[3];
    const WeightFn wf{mx, c_hi, c_lo};
    uint32_t kmin = 0;
    if (tkr > 0 && tkr < a.vocab) kmin = topk_key<T>(rp, tkr, sm);
    float s = 0.0f, comp = 0.0f;
    rp.each([&](const uint32_t (&bits)[EPV]) {
#pragma unroll
      for (int e = 0; e < EPV; ++e) {
        const float wv = LT<T>::key(bits[e]) < kmin ? 0.0f : wf(LT<T>::val(bits[e]));
        const float y = __fsub_rn(wv, comp);
        const float t = __fadd_rn(s, y);
        comp = __fsub_rn(__fsub_rn(t, s), y);
        s = t;
      }
    });
    FF S[1] = {FF{s, -comp}};
    block_sum_ff<1>(S, sm.red[1]);
    if (tpr < 1.0f) {
      nucleus_cut<T>(rp, wf, kmin, ff_to_double(S[0]), tpr, sm, tau, ssum);
    } else {
      tau = kmin;
      ssum = ff_to_double(S[0]);
    }
    // the kept set's sum again from float-float weights (residual draws)
    const FF cc{c_hi, c_lo};
    FF acc1 = ff_make(0.0f);
    rp.each([&](const uint32_t (&bits)[EPV]) {
#pragma unroll
      for (int e = 0; e < EPV; ++e) {
        const float l = LT<T>::val(bits[e]);
        if (LT<T>::key(bits[e]) >= tau && l != -INFINITY)
          acc1 = ff_add(acc1, exp2_ff(ff_mul(two_sum(l, -mx), cc), sm.exp2tab));
      }
    });
    FF A1[1] = {acc1};
    __syncthreads();
    block_sum_ff<1>(A1, sm.red[0]);
    acc = A1[0];
  }
  if (tid == 0) write_stats(&P.ws.stats[r], mx, tau, valid, ssum, c_hi, c_lo, amax, acc, it_hi, it_lo);
  arrive_sequence<T>(P, i, &sm.bcast[3]);
}

// --------------------------------------------------------------------------
// Phase 1c (bf16 rows off the cluster path): one CTA per row, statistics from
// a histogram of the keys in a window just below the row's maximum.  Equal
// bf16 logits have equal weights, so within the window every cut and sum
// follows exactly from the count of each key: work per distinct value, not
// per element.
//   Pass 1 streams the row for its largest and smallest key (NaN / +inf lie
// above 0xFF7F, NaN below 0x7F).  Pass 2 (from L2) counts the keys of the
// window [kb - 2047, kb], kb the largest key, and sums exp((l - max)/T) of
// the elements below it (their float sum completes the row's sum S).  Then,
// on the window's 64 chunks of 32 keys: per-chunk counts and 2^-44 masses,
// their prefixes, the top-k key, the nucleus cut, and the kept set's sum
// from float-float weights.  Should a cut lie below the window (a flat row,
// a large top-k), the next window starts at the largest key below this one
// and the row is counted again; keys above a window are already in the
// prefixes.  Shared memory: about 10 KB, so the CTAs run beside the
// attention's in the fused step.
// --------------------------------------------------------------------------
constexpr int kWinNT = 256;
constexpr int kWinNW = kWinNT / 32;
constexpr int kWinKeys = 2048;                         // keys per window
constexpr int kWinCh = kWinKeys / 32;                  // chunks of 32 keys
constexpr uint32_t kKeyNegInf = 0x007Fu;               // -inf; keys below it: NaN

struct WinSmem {                                       // (the row stream's ring follows)
  unsigned long long cmass[kWinCh], cpm[kWinCh];       // per chunk: 2^-44 mass, its prefix
  uint32_t win[kWinKeys];                              // count of key kb - d at d
  uint32_t ccnt[kWinCh], cpc[kWinCh];                  // per chunk: count, its prefix
  float2 exp2tab[kExp2Tab];
  FF redff[2][kWinNW];
  uint32_t redu[2][kWinNW];
  unsigned long long tot[2];                           // the window's count and mass
  float tconst[4];
  uint32_t cut_key[2];                                 // top-k key, nucleus cut
  unsigned long long cut_m[2];                         // mass at and above each
  int flag[2];
};

// The bf16 value of an order-preserving key, as a float.
__device__ __forceinline__ float key_value(uint32_t k) {
  const uint32_t b = (k & 0x8000u) ? (k & 0x7FFFu) : (~k & 0xFFFFu);
  return __uint_as_float(b << 16);
}

// Order-preserving keys of the two bf16 values of a word (packed halves).
__device__ __forceinline__ uint32_t keys2_of(uint32_t wd) {
  const uint32_t sg = (wd >> 15) & 0x00010001u;
  return wd ^ (0x80008000u | (sg * 0x7FFFu));
}

// f(v, vector) for every 16-byte vector of the row this thread owns (v =
// k * kWinNT + tid, in increasing order).  An aligned row streams through a
// ring of STAGES 16-byte slots per thread in shared memory (slot s of thread
// t at ring[s * kWinNT + t]), filled by cp.async STAGES vectors ahead: deep
// prefetch without registers; each thread reads only its own slots, so no
// barrier; a slot is refilled after its vector has been used.  An unaligned
// row, and a row's ragged last vector, use plain loads.  Elements past V read
// as -inf.
template <int STAGES, typename F>
__device__ __forceinline__ void win_stream(const uint16_t *row, int V, int NV, bool aligned,
                                           uint4 *ring, F &&f) {
  const int tid = threadIdx.x;
  if (!aligned) {
#pragma unroll 1
    for (int v = tid; v < NV; v += kWinNT) f(v, load_vec<uint16_t>(row, V, v, false));
    return;
  }
  auto issue = [&](int v, int slot) {
    if (v < NV) {
      uint4 *dst = ring + slot * kWinNT + tid;
      if (v * 8 + 8 <= V) cp_async16(smem_u32(dst), row + v * 8, 16);
      else *dst = load_vec<uint16_t>(row, V, v, true);
    }
    cp_async_commit();                           // one group per step (maybe empty)
  };
#pragma unroll
  for (int k = 0; k < STAGES; ++k) issue(k * kWinNT + tid, k);
  int slot = 0;
#pragma unroll 1
  for (int v = tid; v < NV; v += kWinNT) {
    cp_async_wait<STAGES - 1>();                 // this thread's oldest group has landed
    const uint4 cur = ring[slot * kWinNT + tid];
    f(v, cur);
    issue(v + STAGES * kWinNT, slot);
    slot = slot + 1 == STAGES ? 0 : slot + 1;
  }
  cp_async_wait<0>();
}

// Per-half maximum of two bf16 pairs; a NaN half wins (NaN propagates).
__device__ __forceinline__ uint32_t bmax2_nan(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.NaN.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// Keys of the two bf16 values of a word with -0 taken as +0 (as key_of_bf16).
__device__ __forceinline__ uint32_t keys2_merged(uint32_t wd) {
  return keys2_of(wd & ~__vcmpeq2(wd, 0x80008000u));
}

// Block-wide float-float sum of one value per thread (fixed order; all get it).
__device__ __forceinline__ FF win_sum_ff(FF v, FF *red) {
  v = warp_sum_ff(v);
  __syncthreads();
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  FF t = red[0];
#pragma unroll
  for (int k = 1; k < kWinNW; ++k) t = ff_add(t, red[k]);
  return t;
}

// A 2^-44 fixed-point sum as a float-float (both parts exact conversions).
__device__ __forceinline__ FF ff_from_fix44(unsigned long long x) {
  const float hi = __ull2float_rn(x);
  const long long rem = static_cast<long long>(x - __float2ull_rn(hi));
  return FF{__fmul_rn(hi, 0x1p-44f), __fmul_rn(__ll2float_rn(rem), 0x1p-44f)};
}

// floor(s * p) for a 2^-44 sum s < 2^62 and a float p in (0, 1), exactly.
__device__ __forceinline__ unsigned long long mul_fix_p(unsigned long long s, float p) {
  const uint32_t b = __float_as_uint(p);
  const int e = static_cast<int>((b >> 23) & 0xFFu);
  const unsigned long long m = e ? ((b & 0x7FFFFFu) | 0x800000u) : (b & 0x7FFFFFu);
  const int sh = e ? 150 - e : 149;                     // p = m * 2^-sh
  const u128 prod = static_cast<u128>(s) * m;
  return sh < 128 ? static_cast<unsigned long long>(prod >> sh) : 0ull;
}

// Row statistics from the row's finished sums (one thread).
__device__ __forceinline__ void write_stats_ff(RowStats *st, float lmax, uint32_t tau, bool valid,
                                               FF ssum, float c_hi, float c_lo, int amax, FF acc,
                                               float it_hi, float it_lo) {
  RowStats o;
  o.lmax = lmax;
  o.tau_key = tau;
  o.valid = valid ? 1u : 0u;
  const FF inv = valid ? ff_recip(ssum) : FF{0.0f, 0.0f};
  o.inv_hi = inv.hi;
  o.inv_lo = inv.lo;
  o.amax = valid ? amax : -1;
  o.c_hi = c_hi;
  o.c_lo = c_lo;
  o.acc_hi = acc.hi;
  o.acc_lo = acc.lo;
  o.it_hi = it_hi;
  o.it_lo = it_lo;
  *st = o;
}

// log2(e)/T and 1/T as float-float pairs (no fp64): quotient, exact
// remainder by fma, corrected quotient.
__device__ __forceinline__ void temp_consts(float T, float *out) {
  constexpr float kLog2eHi = 1.44269502162933349609375f, kLog2eLo = 1.925963033500011079e-08f;
  const float q = __fdiv_rn(kLog2eHi, T);
  const float rq = __fadd_rn(__fmaf_rn(-q, T, kLog2eHi), kLog2eLo);
  const FF c = quick_two_sum(q, __fdiv_rn(rq, T));
  const float t = __frcp_rn(T);
  const FF it = quick_two_sum(t, __fdiv_rn(__fmaf_rn(-t, T, 1.0f), T));
  out[0] = c.hi;
  out[1] = c.lo;
  out[2] = it.hi;
  out[3] = it.lo;
}

// A 2^-44 fixed-point value of a non-negative float-float below 2^18.
__device__ __forceinline__ unsigned long long fix44_ff(FF x) {
  return __float2ull_rn(__fmul_rn(x.hi, 0x1p44f)) +
         static_cast<unsigned long long>(__float2ll_rn(__fmul_rn(x.lo, 0x1p44f)));
}

constexpr size_t kWinSmemOff = (sizeof(WinSmem) + 127) / 128 * 128;   // the ring's offset

template <int STAGES>
__global__ void __launch_bounds__(kWinNT, 2) stats_win_kernel(const SampParams P) {
  const PdlTail tail{P.pdl_secondary};
  extern __shared__ __align__(16) unsigned char smem_raw[];
  WinSmem &sm = *reinterpret_cast<WinSmem *>(smem_raw);
  uint4 *ring = reinterpret_cast<uint4 *>(smem_raw + kWinSmemOff);
  const sv_sample_args &a = P.a;
  const int r = blockIdx.x;
  const int tid = threadIdx.x, w = tid >> 5, l = tid & 31;
  const void *base;
  int64_t off;
  const int i = row_seq(a, r, base, off);
  if (!seq_rows_ok(a, i)) {
    if (tid == 0) set_status(a.dev_status, SV_DEV_BAD_LENGTH);
    return;
  }
  const uint16_t *row = static_cast<const uint16_t *>(base) + off;
  const int V = a.vocab, NV = (V + 7) / 8;
  const bool aligned = (reinterpret_cast<uintptr_t>(row) & 15) == 0;
  exp2_table_fill(sm.exp2tab, P.exp2tab);
  const float Tr = a.temperatures ? a.temperatures[i] : a.temperature;
  const float tpr = a.top_ps ? a.top_ps[i] : a.top_p;
  const int tkr = a.top_ks ? a.top_ks[i] : a.top_k;
  const bool param_ok = Tr >= 0.0f && tpr > 0.0f && tkr >= 0;     // NaN fails the compares
  if (tid == 0) {
    if (!param_ok) set_status(a.dev_status, SV_DEV_BAD_PARAM);
    if (a.temperatures && param_ok && Tr > 0.0f) temp_consts(Tr, sm.tconst);
  }
  // ---- pass 1: the largest value, NaN propagating (elements past V read as
  // -inf: no maximum unless every logit is -inf)
  // Greedy rows also keep each thread's first index of its running maximum
  // (a thread's vectors come in increasing order, so a later equal value
  // never replaces it; values are compared, so -0 and +0 are equal).
  uint32_t mx2 = 0xFF80FF80u;
  const bool greedy = Tr == 0.0f;
  float gbest = -INFINITY;
  int gidx = INT_MAX;
  win_stream<STAGES>(row, V, NV, aligned, ring, [&](int v, const uint4 &x) {
    const uint32_t v2 = bmax2_nan(bmax2_nan(x.x, x.y), bmax2_nan(x.z, x.w));
    mx2 = bmax2_nan(mx2, v2);
    if (greedy) {
      const float vm = fmaxf(__uint_as_float(v2 << 16), __uint_as_float(v2 & 0xFFFF0000u));
      if (vm > gbest) {
        uint32_t b[8];
        unpack<uint16_t>(x, b);
        int e0 = 7;
#pragma unroll
        for (int e = 7; e >= 0; --e)
          if (LT<uint16_t>::val(b[e]) == vm) e0 = e;
        gbest = vm;
        gidx = v * 8 + e0;
      }
    }
  });
  const uint32_t mb = bmax2_nan(mx2, mx2 >> 16) & 0xFFFFu;
  // a NaN maximum takes the largest key, so the reduction keeps it
  uint32_t tmax = (mb & 0x7FFFu) > 0x7F80u ? 0xFFFFu : key_of_bf16(mb);
  tmax = __reduce_max_sync(0xffffffffu, tmax);
  if (l == 0) sm.redu[0][w] = tmax;
  __syncthreads();
  uint32_t maxkey = 0u;
#pragma unroll
  for (int k = 0; k < kWinNW; ++k) maxkey = max(maxkey, sm.redu[0][k]);
  const bool bad = maxkey >= 0xFF80u;              // +inf or NaN
  bool valid = param_ok && !bad && maxkey > kKeyNegInf;          // some finite logit
  const float M = valid ? key_value(maxkey) : -INFINITY;
  RowStats *out = &P.ws.stats[r];
  if (!valid) {
    if (tid == 0)
      write_stats_ff(out, M, 0u, false, FF{0.0f, 0.0f}, 0.0f, 0.0f, -1, FF{0.0f, 0.0f}, 0.0f, 0.0f);
  } else if (Tr == 0.0f) {
    // ---- greedy: one-hot at the lowest index holding the maximum: the
    // smallest first index among the threads whose running maximum is it
    int first = gbest == M ? gidx : INT_MAX;
    first = __reduce_min_sync(0xffffffffu, first);
    __syncthreads();
    if (l == 0) sm.redu[0][w] = static_cast<uint32_t>(first);
    __syncthreads();
    if (tid == 0) {
      int f = INT_MAX;
      for (int k = 0; k < kWinNW; ++k) f = min(f, static_cast<int>(sm.redu[0][k]));
      write_stats_ff(out, M, 0u, true, FF{1.0f, 0.0f}, 0.0f, 0.0f, f, FF{1.0f, 0.0f}, 0.0f, 0.0f);
    }
  } else {
    const bool own_t = a.temperatures != nullptr;
    const float c_hi = own_t ? sm.tconst[0] : P.c_hi, c_lo = own_t ? sm.tconst[1] : P.c_lo;
    const float it_hi = own_t ? sm.tconst[2] : P.it_hi, it_lo = own_t ? sm.tconst[3] : P.it_lo;
    const WeightFn wf{M, c_hi, c_lo};
    const FF cc{c_hi, c_lo};
    const bool topk = tkr > 0 && tkr < V, nucleus = tpr < 1.0f;
    const bool keep_all = !topk && !nucleus;
    const unsigned long long K = topk ? static_cast<unsigned long long>(tkr) : 0ull;
    auto wfix = [&](uint32_t k) -> unsigned long long {          // 2^-44 weight of a key
      return k > kKeyNegInf ? fix44(wf(key_value(k))) : 0ull;
    };
    auto wff = [&](uint32_t k) -> FF {                           // float-float weight
      return exp2_ff(ff_mul(two_sum(key_value(k), -M), cc), sm.exp2tab);
    };
    uint32_t kb = maxkey;                      // the window: keys [klo, kb]
    unsigned long long pre_c = 0, pre_m = 0;   // count / mass of the keys above the window
    unsigned long long sk = 0, S_fix = 0, ssum = 0;
    FF acc_pre = ff_make(0.0f), acc_tail = ff_make(0.0f), acc = ff_make(0.0f);
    bool have_k = !topk, have_p = !nucleus, done = false;
    uint32_t kmin = 0u, tau = 0u;
    for (int it = 0; it < 64 && !done; ++it) {   // 32 windows cover every key
      // The first pass takes keys raw (-0 one below +0, merged into it after
      // the pass); its window ends one key higher when its last slot would
      // hold +0, so the two zeros are never split.  Later passes use merged keys.
      const uint32_t wlim =
          it == 0 && kb - 0x8000u == static_cast<uint32_t>(kWinKeys - 1) ? kWinKeys - 1 : kWinKeys;
      const uint32_t klo = kb >= wlim - 1 ? kb - (wlim - 1) : 0u;   // the window: keys [klo, kb]
      for (int d = tid; d < kWinKeys; d += kWinNT) sm.win[d] = 0u;
      __syncthreads();
      // ---- pass 2: count the window's keys; the first pass also sums every
      // element's fp32 weight (the row's sum S, Kahan-compensated per vector)
      float s = 0.0f, sc = 0.0f;
      const float mc_hi = c_hi, mc_lo = c_lo;
      auto count_vec = [&](const uint4 &x, int nel, bool sum) {
        const uint32_t wd[4] = {x.x, x.y, x.z, x.w};
        float vs = 0.0f;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const uint32_t kk = keys2_merged(wd[q]);
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const bool live = 2 * q + h < nel;
            const uint32_t d = kb - (h ? (kk >> 16) : (kk & 0xFFFFu));   // keys above kb wrap
            if (live && d < wlim) atomicAdd(&sm.win[d], 1u);
            if (sum) {
              const float lv = __uint_as_float(h ? (wd[q] & 0xFFFF0000u) : (wd[q] << 16));
              const float dl = fmaxf(__fsub_rn(lv, M), -1.0e30f);       // -inf: weight 0, never NaN
              const float wv = fast_exp2(__fmaf_rn(dl, mc_hi, __fmul_rn(dl, mc_lo)));
              vs = __fadd_rn(vs, live ? wv : 0.0f);
            }
          }
        }
        if (sum) {
          const float y = __fsub_rn(vs, sc);
          const float t = __fadd_rn(s, y);
          sc = __fsub_rn(__fsub_rn(t, s), y);
          s = t;
        }
      };
      if (it == 0) {
        // (no key exceeds kb in the first pass)
        const float2 nm2 = make_float2(-M, -M), ch2 = make_float2(mc_hi, mc_hi), cl2 = make_float2(mc_lo, mc_lo);
        win_stream<STAGES>(row, V, NV, aligned, ring, [&](int v, const uint4 &x) {
          if (v * 8 + 8 > V) {                 // the ragged last vector
            count_vec(x, V - v * 8, true);
            return;
          }
          const uint32_t wd[4] = {x.x, x.y, x.z, x.w};
          float2 vs2 = make_float2(0.0f, 0.0f);
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const uint32_t kk = keys2_of(wd[q]);
            const uint32_t d0 = kb - (kk & 0xFFFFu), d1 = kb - (kk >> 16);
            if (d0 < wlim) atomicAdd(&sm.win[d0], 1u);
            if (d1 < wlim) atomicAdd(&sm.win[d1], 1u);
            const float2 lv = make_float2(__uint_as_float(wd[q] << 16), __uint_as_float(wd[q] & 0xFFFF0000u));
            // a masked (-inf) logit: the difference is clamped to a huge
            // negative finite value, so that -inf * c_hi + (-inf) * c_lo (c_lo
            // may be negative) cannot give NaN; its weight is 0
            float2 dl = __fadd2_rn(lv, nm2);
            dl = make_float2(fmaxf(dl.x, -1.0e30f), fmaxf(dl.y, -1.0e30f));
            const float2 ag = __ffma2_rn(dl, ch2, __fmul2_rn(dl, cl2));
            vs2 = __fadd2_rn(vs2, make_float2(fast_exp2(ag.x), fast_exp2(ag.y)));
          }
          const float y = __fsub_rn(__fadd_rn(vs2.x, vs2.y), sc);
          const float t = __fadd_rn(s, y);
          sc = __fsub_rn(__fsub_rn(t, s), y);
          s = t;
        });
        __syncthreads();
        if (tid == 0 && kb >= 0x8000u) {       // -0 (key 0x7FFF) into +0
          const uint32_t dz = kb - 0x8000u;
          if (dz + 1u < wlim) {
            sm.win[dz] += sm.win[dz + 1u];
            sm.win[dz + 1u] = 0u;
          }
        }
      } else {
        win_stream<STAGES>(row, V, NV, aligned, ring, [&](int v, const uint4 &x) { count_vec(x, V - v * 8, false); });
      }
      FF at = ff_make(0.0f);                   // keep-all rows: float-float tail weights
      if (it == 0 && keep_all) {
        win_stream<STAGES>(row, V, NV, aligned, ring, [&](int v, const uint4 &x) {
          const int nel = min(8, V - v * 8);
#pragma unroll 1
          for (int e = 0; e < nel; ++e) {
            const uint32_t k = key_of_bf16(elem_bits<uint16_t>(x, e));
            if (k < klo && k > kKeyNegInf) at = ff_add(at, wff(k));
          }
        });
      }
      FF rowsum = ff_make(0.0f);
      if (it == 0) {
        rowsum = win_sum_ff(FF{s, -sc}, sm.redff[0]);
        if (keep_all) acc_tail = win_sum_ff(at, sm.redff[1]);
      }
      __syncthreads();
      // ---- per chunk: count and mass (lane l: key kb - (32 ch + l))
      for (int ch = w; ch < kWinCh; ch += kWinNW) {
        const int d = 32 * ch + l;
        const uint32_t c = sm.win[d];
        const unsigned long long m = c ? static_cast<unsigned long long>(c) * wfix(kb - d) : 0ull;
        const uint32_t cs = __reduce_add_sync(0xffffffffu, c);
        const unsigned long long ms = warp_sum_u64(m);
        if (l == 0) {
          sm.ccnt[ch] = cs;
          sm.cmass[ch] = ms;
        }
      }
      __syncthreads();
      if (w == 0) {                            // prefixes over the chunks, in key order
        const unsigned long long c0 = sm.ccnt[2 * l], c1 = sm.ccnt[2 * l + 1];
        const unsigned long long m0 = sm.cmass[2 * l], m1 = sm.cmass[2 * l + 1];
        const unsigned long long ic = warp_inclusive_scan_u64(c0 + c1);
        const unsigned long long im = warp_inclusive_scan_u64(m0 + m1);
        sm.cpc[2 * l] = static_cast<uint32_t>(ic - c0 - c1);
        sm.cpc[2 * l + 1] = static_cast<uint32_t>(ic - c1);
        sm.cpm[2 * l] = im - m0 - m1;
        sm.cpm[2 * l + 1] = im - m1;
        if (l == 31) {
          sm.tot[0] = ic;
          sm.tot[1] = im;
        }
      }
      __syncthreads();
      const unsigned long long wc = sm.tot[0], wm = sm.tot[1];
      if (it == 0) {
        S_fix = fix44_ff(rowsum);              // the sum over every element
        if (!topk) sk = S_fix;
      }
      // Warp 0: the chunk whose prefix range holds `tg` (counts or masses),
      // then its lanes' inclusive scan: the key where the running value first
      // reaches tg, and the mass at and above it, into slot q.
      auto crossing = [&](bool by_count, unsigned long long tg, int q) {
        const unsigned long long pre = by_count ? pre_c : pre_m;
        auto lo = [&](int ch) { return pre + (by_count ? sm.cpc[ch] : sm.cpm[ch]); };
        auto val = [&](int ch) { return by_count ? static_cast<unsigned long long>(sm.ccnt[ch]) : sm.cmass[ch]; };
        const bool o0 = lo(2 * l) < tg && tg <= lo(2 * l) + val(2 * l);
        const bool o1 = lo(2 * l + 1) < tg && tg <= lo(2 * l + 1) + val(2 * l + 1);
        const unsigned bal = __ballot_sync(0xffffffffu, o0 || o1);
        const int src = bal ? __ffs(bal) - 1 : 0;
        const int ch = 2 * src + (__shfl_sync(0xffffffffu, o0 ? 1 : 0, src) ? 0 : 1);
        const int d = 32 * ch + l;
        const uint32_t c = sm.win[d];
        const unsigned long long m = c ? static_cast<unsigned long long>(c) * wfix(kb - d) : 0ull;
        const unsigned long long icn = warp_inclusive_scan_u64(c), imn = warp_inclusive_scan_u64(m);
        const unsigned hit = __ballot_sync(0xffffffffu, lo(ch) + (by_count ? icn : imn) >= tg);
        if (hit && l == __ffs(hit) - 1) {
          sm.cut_key[q] = kb - static_cast<uint32_t>(d);
          sm.cut_m[q] = pre_m + sm.cpm[ch] + imn;
        }
      };
      // ---- top-k: the largest key with at least k elements at or above it
      bool restart = false;
      if (!have_k && pre_c + wc >= K) {
        if (w == 0) crossing(true, K, 0);
        __syncthreads();
        kmin = sm.cut_key[0];
        sk = sm.cut_m[0];
        have_k = true;
        // a nucleus target (top_p times the top-k mass) met above this window:
        // count the windows again from the top
        restart = nucleus && max(mul_fix_p(sk, tpr), 1ull) <= pre_m;
      }
      if (restart) {
        kb = maxkey;
        pre_c = 0;
        pre_m = 0;
        acc_pre = ff_make(0.0f);
        __syncthreads();
        continue;
      }
      // ---- nucleus: the largest key whose mass at or above it reaches top_p * S
      if (have_k && !have_p) {
        const unsigned long long tg = max(mul_fix_p(sk, tpr), 1ull);
        if (pre_m + wm >= tg) {
          if (w == 0) crossing(false, tg, 1);
          __syncthreads();
          tau = sm.cut_key[1];
          ssum = sm.cut_m[1];
          have_p = true;
        }
      }
      // ---- the float-float sum of this window's keys at or above the cut
      // (all of them when the cuts lie further down)
      done = have_k && have_p;
      const uint32_t cut = done ? (nucleus ? tau : kmin) : klo;
      FF aw = ff_make(0.0f);
      for (int ch = w; ch < kWinCh; ch += kWinNW) {
        if (kb < cut + 32u * static_cast<uint32_t>(ch)) break;    // chunks fall in key order
        if (sm.ccnt[ch] == 0u) continue;
        const int d = 32 * ch + l;
        const uint32_t c = sm.win[d];
        if (c != 0u && kb - static_cast<uint32_t>(d) >= cut && kb - static_cast<uint32_t>(d) > kKeyNegInf)
          aw = ff_add(aw, ff_mul(FF{static_cast<float>(c), 0.0f}, wff(kb - d)));
      }
      aw = win_sum_ff(aw, sm.redff[0]);
      acc_pre = ff_add(acc_pre, aw);
      if (done) {
        tau = cut;
        if (!nucleus) ssum = topk ? sk : S_fix;
        acc = ff_add(acc_pre, acc_tail);       // acc_tail: keep-all rows only
      } else {
        pre_c += wc;
        pre_m += wm;
        // the next window starts at the largest key below this one
        uint32_t nxt = 0u;                     // 1 + that key (0: none)
        win_stream<STAGES>(row, V, NV, aligned, ring, [&](int v, const uint4 &x) {
          const int nel = V - v * 8;
          const uint32_t wd[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const uint32_t kk = keys2_merged(wd[q]);
            const uint32_t k0 = kk & 0xFFFFu, k1 = kk >> 16;
            if (2 * q < nel && k0 < klo) nxt = max(nxt, k0 + 1u);
            if (2 * q + 1 < nel && k1 < klo) nxt = max(nxt, k1 + 1u);
          }
        });
        nxt = __reduce_max_sync(0xffffffffu, nxt);
        __syncthreads();
        if (l == 0) sm.redu[0][w] = nxt;
        __syncthreads();
        uint32_t n1 = 0u;
#pragma unroll
        for (int k = 0; k < kWinNW; ++k) n1 = max(n1, sm.redu[0][k]);
        if (n1 == 0u) {
          // no key left below: a nucleus target above the exact total mass
          // (top_p within the sum's rounding of 1) keeps every key
          if (have_k && !have_p && !topk) {
            tau = 0u;
            ssum = pre_m;
            acc = acc_pre;
            done = true;
          }
          break;
        }
        kb = n1 - 1u;
      }
      __syncthreads();
    }
    if (!done) valid = false;
    if (tid == 0)
      write_stats_ff(out, M, tau, valid, ff_from_fix44(ssum), c_hi, c_lo, -1, acc, it_hi, it_lo);
  }
  arrive_sequence<uint16_t>(P, i, &sm.flag[0]);
  asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
}

// --------------------------------------------------------------------------
// Phase 2: draw and append.  CTA (sequence i, chunk c): fixed-point sum of the
// draw weights of its chunk of row n_i (residual of target/draft row n_i, or
// the bonus target row); the last chunk to finish scans the chunk sums, finds
// the chunk holding the crossing and walks it.  Every chunk CTA also copies its
// slice of block rows 0..n_i to the KV pool (fused step).
// --------------------------------------------------------------------------
constexpr int kDrawNT = 256;
constexpr int kDrawVec = 2;          // contiguous vectors per thread (one run)

struct DrawSmem {
  float2 exp2tab[kExp2Tab];
  u128 red[kDrawNT / 32];
  u128 bc128[2];
  FF L;
  float inv_sq;
  int bc[4];
};

// Sum of the chunk's fixed-point draw weights (block-wide, all threads get it).
template <typename T>
__device__ u128 chunk_sum(const T *trow, const T *drow, int V, int v0, int v1,
                          const DrawWeight &dw, DrawSmem &sm) {
  constexpr int EPV = LT<T>::EPV;
  const bool two = dw.mode == 0;
  const bool al_t = (reinterpret_cast<uintptr_t>(trow) & 15) == 0;
  const bool al_d = two && (reinterpret_cast<uintptr_t>(drow) & 15) == 0;
  u128 s = 0;
  for (int vb = v0; vb < v1; vb += kDrawVec * kDrawNT) {
    uint4 q[kDrawVec], d[kDrawVec];
#pragma unroll
    for (int k = 0; k < kDrawVec; ++k) {
      const int v = vb + k * kDrawNT + threadIdx.x;
      if (v < v1) {
        q[k] = load_vec<T>(trow, V, v, al_t);
        if (two) d[k] = load_vec<T>(drow, V, v, al_d);
      }
    }
#pragma unroll
    for (int k = 0; k < kDrawVec; ++k) {
      const int v = vb + k * kDrawNT + threadIdx.x;
      if (v < v1) {
        uint32_t bq[EPV], bd[EPV];
        unpack<T>(q[k], bq);
        if (two) unpack<T>(d[k], bd);
#pragma unroll
        for (int e = 0; e < EPV; ++e) s += dw.fix<T>(bq[e], two ? bd[e] : 0u, v * EPV + e);
      }
    }
  }
  return block_sum_u128<kDrawNT>(s, sm.red);
}

// Fixed-point sum of the draw weights of one run: vectors [va, va + kDrawVec)
// clipped to v1 (one thread).
template <typename T>
__device__ __forceinline__ u128 run_sum(const T *trow, const T *drow, int V, int va, int v1,
                                        const DrawWeight &dw) {
  constexpr int EPV = LT<T>::EPV;
  const bool two = dw.mode == 0;
  const bool al_t = (reinterpret_cast<uintptr_t>(trow) & 15) == 0;
  const bool al_d = two && (reinterpret_cast<uintptr_t>(drow) & 15) == 0;
  uint4 q[kDrawVec], d[kDrawVec];
#pragma unroll
  for (int k = 0; k < kDrawVec; ++k) {
    if (va + k < v1) {
      q[k] = load_vec<T>(trow, V, va + k, al_t);
      if (two) d[k] = load_vec<T>(drow, V, va + k, al_d);
    }
  }
  u128 s = 0;
#pragma unroll
  for (int k = 0; k < kDrawVec; ++k) {
    if (va + k < v1) {
      uint32_t bq[EPV], bd[EPV];
      unpack<T>(q[k], bq);
      if (two) unpack<T>(d[k], bd);
#pragma unroll
      for (int e = 0; e < EPV; ++e) s += dw.fix<T>(bq[e], two ? bd[e] : 0u, (va + k) * EPV + e);
    }
  }
  return s;
}

// The warp of the thread whose run [vf, vf + kDrawVec) holds the target walks
// that run together: lane e recomputes element e of the run (the same weight
// bits as the run sums), an inclusive scan over the lanes gives the running
// sums from `lof` (the run's start), the first lane past `tgt` holds the
// token.  Call with the whole warp; returns the token index on every lane.
template <typename T>
__device__ __forceinline__ int run_walk(const T *trow, const T *drow, int V, int vf, int v1,
                                        const DrawWeight &dw, u128 lof, u128 tgt) {
  constexpr int EPV = LT<T>::EPV;
  constexpr int RUN = kDrawVec * EPV;
  static_assert(RUN <= 32, "a run has at most 32 elements");
  const bool two = dw.mode == 0;
  const bool al_t = (reinterpret_cast<uintptr_t>(trow) & 15) == 0;
  const bool al_d = two && (reinterpret_cast<uintptr_t>(drow) & 15) == 0;
  const int lane = threadIdx.x & 31;
  const bool in = lane < RUN && vf + lane / EPV < v1;
  u128 wgt = 0;
  if (in) {
    const int v = vf + lane / EPV, e = lane % EPV;
    const uint32_t eq = elem_bits<T>(load_vec<T>(trow, V, v, al_t), e);
    const uint32_t ed = two ? elem_bits<T>(load_vec<T>(drow, V, v, al_d), e) : 0u;
    wgt = dw.fix<T>(eq, ed, v * EPV + e);
  }
  const u128 cum = warp_inclusive_scan_u128(wgt);
  const unsigned hit = __ballot_sync(0xffffffffu, in && lof + cum > tgt);
  const unsigned inm = __ballot_sync(0xffffffffu, in);
  return vf * EPV + (hit ? __ffs(hit) - 1 : 31 - __clz(inm));
}

// Index of the first element of vectors [v0, v1) whose running weight sum,
// starting at 0, exceeds `tgt` (requires the chunk total > tgt).  Thread t
// owns kDrawVec contiguous vectors, so thread order is vocabulary order.
template <typename T>
__device__ int chunk_walk(const T *trow, const T *drow, int V, int v0, int v1,
                          const DrawWeight &dw, u128 tgt, DrawSmem &sm, u128 *scan_red) {
  constexpr int EPV = LT<T>::EPV;
  const bool two = dw.mode == 0;
  const bool al_t = (reinterpret_cast<uintptr_t>(trow) & 15) == 0;
  const bool al_d = two && (reinterpret_cast<uintptr_t>(drow) & 15) == 0;
  const int tid = threadIdx.x;
  int result = -1;
  if (tid == 0) sm.bc[0] = -1;
  u128 base = 0;
  for (int vb = v0; vb < v1; vb += kDrawVec * kDrawNT) {
    const int va = vb + tid * kDrawVec;
    uint32_t bq[kDrawVec][EPV], bd[kDrawVec][EPV];
    u128 s = 0;
#pragma unroll
    for (int k = 0; k < kDrawVec; ++k) {
      if (va + k < v1) {
        unpack<T>(load_vec<T>(trow, V, va + k, al_t), bq[k]);
        if (two) unpack<T>(load_vec<T>(drow, V, va + k, al_d), bd[k]);
#pragma unroll
        for (int e = 0; e < EPV; ++e) s += dw.fix<T>(bq[k][e], two ? bd[k][e] : 0u, (va + k) * EPV + e);
      }
    }
    u128 total;
    const u128 ex = block_exclusive_scan_u128<kDrawNT>(s, scan_red, &total);
    const u128 lo = base + ex;
    const unsigned fm = __ballot_sync(0xffffffffu, s > 0 && lo <= tgt && tgt < lo + s);
    if (fm) {
      const int src = __ffs(fm) - 1;
      const int x = run_walk<T>(trow, drow, V, __shfl_sync(0xffffffffu, va, src), v1, dw,
                                shfl_u128(lo, src), tgt);
      if ((tid & 31) == 0) sm.bc[0] = x;
    }
    __syncthreads();
    result = sm.bc[0];
    if (result >= 0) break;
    base += total;
  }
  return result;
}

template <typename T>
__global__ void __launch_bounds__(kDrawNT, 4) draw_kernel(const SampParams P) {
  __shared__ DrawSmem sm;
  __shared__ u128 scan_red[kDrawNT / 32];
  // launched early behind the histogram statistics: nothing is read before
  // that grid has finished (a no-op after a plain launch)
  asm volatile("griddepcontrol.wait;\n" ::: "memory");
  exp2_table_fill(sm.exp2tab, P.exp2tab);
  const sv_sample_args &a = P.a;
  const int NCH = P.plan.draw_chunks;
  const int i = blockIdx.x / NCH, c = blockIdx.x - i * NCH;
  const int tid = threadIdx.x;
  if (!seq_rows_ok(a, i)) return;                 // flagged in phase 1
  const int V = a.vocab, R = static_cast<int>(a.num_rows);
  const int r0 = cuq(a, i), K = cuq(a, i + 1) - r0 - 1, p0 = r0 - i;
  const int L = a.kv_len[i];
  const int n = a.num_accepted[i];
  if (n < 0 || n > K) {                           // failed sequence: nothing to draw
    if (P.do_append && c == 0 && tid == 0) P.app.new_kv_len[i] = L;
    return;
  }
  // ---- append this chunk's slice of block rows 0..n (fused step)
  if (P.do_append) {
    const AppendView &A = P.app;
    const int64_t start = A.kv_start[i];
    const bool cap_ok = L + n + 1 <= A.kv_cap[i];
    const bool pool_ok = start >= 0 && start + L + n + 1 <= A.pool_rows;
    if (cap_ok && pool_ok) {
      const int64_t nvec = static_cast<int64_t>(n + 1) * A.row_bytes / 16;
      const int64_t a0 = nvec * c / NCH, a1 = nvec * (c + 1) / NCH;
      const uint4 *__restrict__ sk = reinterpret_cast<const uint4 *>(
          static_cast<const char *>(A.k_new) + static_cast<int64_t>(r0) * A.row_bytes);
      const uint4 *__restrict__ svv = reinterpret_cast<const uint4 *>(
          static_cast<const char *>(A.v_new) + static_cast<int64_t>(r0) * A.row_bytes);
      uint4 *__restrict__ dk = reinterpret_cast<uint4 *>(static_cast<char *>(A.k_cache) +
                                                         (start + L) * A.row_bytes);
      uint4 *__restrict__ dv = reinterpret_cast<uint4 *>(static_cast<char *>(A.v_cache) +
                                                         (start + L) * A.row_bytes);
      constexpr int U = 4;
      for (int64_t b = a0; b < a1; b += U * kDrawNT) {
        uint4 x[U], y[U];
#pragma unroll
        for (int k = 0; k < U; ++k) {
          const int64_t v = b + k * kDrawNT + tid;
          if (v < a1) { x[k] = __ldcg(sk + v); y[k] = __ldcg(svv + v); }
        }
#pragma unroll
        for (int k = 0; k < U; ++k) {
          const int64_t v = b + k * kDrawNT + tid;
          if (v < a1) { dk[v] = x[k]; dv[v] = y[k]; }
        }
      }
    }
    if (c == 0 && tid == 0) {
      if (!cap_ok) set_status(a.dev_status, SV_DEV_CAPACITY);
      else if (!pool_ok) set_status(a.dev_status, SV_DEV_BAD_LENGTH);
      A.new_kv_len[i] = cap_ok && pool_ok ? L + n + 1 : L;
    }
  }
  // ---- chunk sum of the draw weights
  constexpr int EPV = LT<T>::EPV;
  const int mode = n < K ? 0 : 1;
  const T *trow = static_cast<const T *>(a.target_logits) + static_cast<int64_t>(r0 + n) * V;
  const T *drow = mode == 0 ? static_cast<const T *>(a.draft_logits) + static_cast<int64_t>(p0 + n) * V
                            : trow;
  const RowStats *sq = &P.ws.stats[r0 + n];
  const RowStats *sp = &P.ws.stats[R + p0 + n];
  DrawWeight dw;
  dw.pq = rowprob_of(sq);
  dw.pp = mode == 0 ? rowprob_of(sp) : dw.pq;
  dw.mode = mode;
  dw.onehot = dw.pq.amax >= 0 || dw.pp.amax >= 0;
  if (dw.pq.amax >= 0 && (mode == 1 || dw.pp.amax >= 0)) {
    // greedy rows (one-hot q_hat and p_hat): the bonus draw, and the residual
    // of a rejection, are one-hot at the target row's maximum; when both rows
    // peak at the same index the residual is empty and the draw takes q_hat
    if (c == 0 && tid == 0) {
      if (mode == 0 && dw.pp.amax == dw.pq.amax) set_status(a.dev_status, SV_DEV_EMPTY_RESIDUAL);
      a.out_tokens[r0 + n] = dw.pq.amax;
    }
    return;
  }
  dw.rf.init(__ldcg(&sq->lmax), mode == 0 ? __ldcg(&sp->lmax) : 0.0f, __ldcg(&sq->c_hi),
             __ldcg(&sq->c_lo), FF{__ldcg(&sq->it_hi), __ldcg(&sq->it_lo)},
             __ldcg(&sq->it_hi) == 1.0f && __ldcg(&sq->it_lo) == 0.0f, sizeof(T) == 4);
  if (mode == 0 && !dw.onehot) {
    __syncthreads();                  // the exp2 table
    if (tid == 0) {                   // float-float, once per CTA
      const FF aq{__ldcg(&sq->acc_hi), __ldcg(&sq->acc_lo)};
      const FF ap{__ldcg(&sp->acc_hi), __ldcg(&sp->acc_lo)};
      sm.L = ln_ratio_ff(ap, aq, sm.exp2tab);
      sm.inv_sq = __frcp_rn(aq.hi);   // a common factor of all weights: any rounding
    }
    __syncthreads();
    dw.rf.L = sm.L;
    dw.rf.inv_sq = sm.inv_sq;
  }
  DrawWeight dq = dw;                 // q_hat of row n (empty-residual fallback)
  dq.mode = 1;
  const int NV = (V + EPV - 1) / EPV;
  const int per = (NV + NCH - 1) / NCH;
  const int v0 = min(NV, c * per), v1 = min(NV, v0 + per);
  // thread t's run: vectors [v0 + t kDrawVec, +kDrawVec) (a chunk has at most
  // kDrawVec * kDrawNT vectors); the run sums are kept for the last CTA
  const u128 st = run_sum<T>(trow, drow, V, v0 + tid * kDrawVec, v1, dw);
  P.ws.draw_thr[(static_cast<int64_t>(i) * NCH + c) * kDrawNT + tid] = st;
  __threadfence();
  const u128 cs = block_sum_u128<kDrawNT>(st, sm.red);
  if (tid == 0) {
    P.ws.draw_parts[static_cast<int64_t>(i) * NCH + c] = cs;
    __threadfence();
    const unsigned old = atomicInc(&P.ws.seq_cnt2[i], static_cast<unsigned>(NCH - 1));
    sm.bc[1] = old == static_cast<unsigned>(NCH - 1) ? 1 : 0;
  }
  __syncthreads();
  if (!sm.bc[1]) return;
  // ---- last chunk: find the crossing chunk, walk it
  __threadfence();
  const long long sid = a.seq_ids ? a.seq_ids[i] : static_cast<long long>(i);
  const U4 wv = philox4x32_10(U4{static_cast<uint32_t>(L + n + 1),
                                 static_cast<uint32_t>(static_cast<unsigned long long>(sid)),
                                 static_cast<uint32_t>(static_cast<unsigned long long>(sid) >> 32), P.stream},
                              static_cast<uint32_t>(a.seed), static_cast<uint32_t>(a.seed >> 32));
  const unsigned long long ku = u24(wv.y);
  int use_mode = mode;
  for (int attempt = 0; attempt < 2; ++attempt) {
    u128 Z = 0, tgt = 0, cum = 0;
    int cstar = NCH - 1;
    if (attempt == 0) {
      // warp 0: the chunk sums in order (four per lane, draw_chunks <= 128),
      // the total, the target floor(k Z / 2^24) and the chunk holding it
      static_assert(kDrawNT >= 32, "one warp at least");
      if (tid < 32) {
        const u128 *parts = P.ws.draw_parts + static_cast<int64_t>(i) * NCH;
        u128 z[4];
#pragma unroll
        for (int q = 0; q < 4; ++q)
          z[q] = 4 * tid + q < NCH ? ldcg_u128(parts + 4 * tid + q) : static_cast<u128>(0);
        const u128 own = z[0] + z[1] + z[2] + z[3];
        const u128 inc = warp_inclusive_scan_u128(own);
        const u128 Zw = shfl_u128(inc, 31);
        const u128 tg = scale_u24(ku, Zw);
        const u128 ex = inc - own;
        if (tid == 0) {
          sm.bc128[0] = Zw;
          sm.bc128[1] = 0;
          sm.bc[2] = NCH - 1;
        }
        __syncwarp();
        if (Zw > 0 && ex <= tg && tg < inc) {     // one lane
          u128 b = ex;
          int q = 0;
          while (q < 3 && tg >= b + z[q]) b += z[q++];
          sm.bc[2] = 4 * tid + q;
          sm.bc128[1] = b;
        }
      }
      __syncthreads();
      Z = sm.bc128[0];
      cum = sm.bc128[1];
      cstar = sm.bc[2];
      tgt = scale_u24(ku, Z);
    } else {                       // fallback: q_hat of row n, chunk sums computed here
      for (int k = 0; k < NCH; ++k) {
        const int a0 = min(NV, k * per), a1 = min(NV, a0 + per);
        Z += chunk_sum<T>(trow, trow, V, a0, a1, dq, sm);
      }
      tgt = scale_u24(ku, Z);
      for (int k = 0; k < NCH; ++k) {
        const int a0 = min(NV, k * per), a1 = min(NV, a0 + per);
        const u128 zk = chunk_sum<T>(trow, trow, V, a0, a1, dq, sm);
        if (tgt < cum + zk) { cstar = k; break; }
        cum += zk;
      }
    }
    if (Z == 0) {
      if (attempt == 0 && mode == 0) {
        if (tid == 0) set_status(a.dev_status, SV_DEV_EMPTY_RESIDUAL);
        use_mode = 1;
        __syncthreads();           // sm.bc128 is rewritten by the fallback
        continue;
      }
      if (tid == 0) a.out_tokens[r0 + n] = -1;   // empty q_hat: cannot happen for a valid row
      return;
    }
    const int a0 = min(NV, cstar * per), a1 = min(NV, a0 + per);
    int x;
    if (use_mode == mode) {
      // the stored run sums of chunk cstar, scanned in vocabulary order; the
      // warp of the run holding the target walks it
      const u128 tr = tgt - cum;
      const u128 sr = ldcg_u128(P.ws.draw_thr + (static_cast<int64_t>(i) * NCH + cstar) * kDrawNT + tid);
      if (tid == 0) sm.bc[0] = -1;
      u128 total;
      const u128 ex = block_exclusive_scan_u128<kDrawNT>(sr, scan_red, &total);
      const unsigned fm = __ballot_sync(0xffffffffu, sr > 0 && ex <= tr && tr < ex + sr);
      if (fm) {
        const int src = __ffs(fm) - 1;
        const int xf = run_walk<T>(trow, drow, V, a0 + ((tid & ~31) + src) * kDrawVec, a1, dw,
                                   shfl_u128(ex, src), tr);
        if ((tid & 31) == 0) sm.bc[0] = xf;
      }
      __syncthreads();
      x = sm.bc[0];
    } else {
      x = chunk_walk<T>(trow, trow, V, a0, a1, dq, tgt - cum, sm, scan_red);
    }
    if (tid == 0) a.out_tokens[r0 + n] = x;
    return;
  }
}

// --------------------------------------------------------------------------
// Cluster path (no nucleus): one thread-block cluster of kClusterN CTAs per
// sequence; CTA k owns vocabulary slice k of every row of the sequence.  The
// phases meet at two cluster barriers (one more per extra round of the draw)
// and exchange data through distributed shared memory: no global atomics, no
// fences, no second launch.
//   A  CTA k loads slice k of every row into registers (rows in groups of
//      kRowGroup, all loads of a group in flight together); per row the warp
//      max, then each thread's 2^((l - max) log2(e)/T) summed across the warp,
//      merged across the CTA as (max, sum) pairs.  Barrier (1).
//   B  every CTA merges each row's kClusterN slice statistics (remote reads),
//      evaluates the draft tokens' probabilities and runs the accept tests,
//      so all CTAs hold n without another barrier; CTA 0 writes the outputs.
//   C  append slice k of the accepted block rows; exact fixed-point sums of
//      row n (the residual, and q_hat for the empty-residual fallback) per
//      thread run, re-read from L2, scanned inside the CTA; each CTA pushes
//      its slice totals into every CTA's table.  Barrier (2).
// Shared memory holds only the statistics (a few KB), so a cluster's CTAs fit
// beside the attention's CTAs on any SM in the fused step.
//   D  every CTA reads the kClusterN slice totals from its own table and
//      locates the target in vocabulary order; inside the owner CTA the
//      thread whose run holds it walks that run.  No CTA touches another's
//      shared memory after barrier (2), so none waits for the others to
//      leave.
// Weights use the SFU's approximate exp2 (relative error ~2^-22) and fp32
// (max, sum) merges: relative error of a probability stays below ~2e-6, far
// inside the 1e-5 near-tie windows of the decisions.
// --------------------------------------------------------------------------
constexpr int kClusterN = 8;
constexpr int kClNT = 256;
constexpr int kClNW = kClNT / 32;
constexpr int kMaxRows = 2 * kMaxQRows - 1;          // 2K+1 rows per sequence
constexpr int kRowGroup = 4;                         // rows reduced together
constexpr int kClVPT = 2;                            // vectors per thread per row slice

struct ClusterSmem {
  float pm[kMaxRows], ps[kMaxRows];                  // slice (max, sum) per row
  uint32_t pbad[kMaxRows];
  float st_m[kMaxRows], st_inv[kMaxRows];            // merged per row (every CTA)
  uint32_t st_bad[kMaxRows];
  float pdraft[kMaxRows];                            // probability of the row's draft token
  uint32_t dbits[kMaxRows];                          // logit bits at the draft token
  int dtok[kMaxRows];
  union {                                            // never live together:
    struct {                                         // phase A: per-warp row statistics
      float redm[kMaxRows][kClNW], reds[kMaxRows][kClNW];
      uint32_t redb[kMaxRows][kClNW];
    } a;
    ulonglong2 tab[kClusterN][2];                    // phase D: every CTA's slice totals A, B
  } scr;                                             // and its two float-float sums, pushed by it
  unsigned long long scan64[kClNW];
  unsigned long long dec_pa, dec_pb;                 // prefix of the owner slice
  FF dec_L;                                          // exact ln(S_p / S_q) (recut pass)
  i128 dec_tg;                                       // the target, in units of A + beta B
  long long dec_beta;                                // beta * 2^56
  FF redff[2][kClNW];
  FF Lr;                                             // ln(S_p / S_q) of rows n
  int walker;                                        // thread whose run holds the target
  uint32_t draw_u24[kMaxQRows];                      // draw uniform if n = index
  int dec_use, dec_owner;
  int n;
};

// 2^(d * log2(e)/T) for d = l - max <= 0 (0 for d = -inf).
struct Ex2c {
  float c_hi, c_lo;
  __device__ __forceinline__ float operator()(float d) const {
    return d == -INFINITY ? 0.0f : fast_exp2(__fmaf_rn(d, c_hi, __fmul_rn(d, c_lo)));
  }
};

// expm1_fast(x) without a branch: both of its forms, then the one it would
// take (the same operations, so the same bits).  Unrolled over a vector, the
// elements' chains interleave instead of running one after another.
__device__ __forceinline__ float expm1_sel(float x) {
  float p = 1.0f / 40320.0f;
  p = __fmaf_rn(p, x, 1.0f / 5040.0f);
  p = __fmaf_rn(p, x, 1.0f / 720.0f);
  p = __fmaf_rn(p, x, 1.0f / 120.0f);
  p = __fmaf_rn(p, x, 1.0f / 24.0f);
  p = __fmaf_rn(p, x, 1.0f / 6.0f);
  p = __fmaf_rn(p, x, 0.5f);
  p = __fmaf_rn(p, x, 1.0f);
  const float taylor = __fmul_rn(p, x);
  const float viaexp = __fsub_rn(fast_exp2(__fmul_rn(x, 1.4426950408889634f)), 1.0f);
  return fabsf(x) < 0.35f ? taylor : viaexp;
}

// fix63(r) for r in [0, 2) by one conversion: r * 2^63 is exact (a power of
// two) and below 2^64, and truncation toward zero is the floor that fix63's
// shifts take; subnormal r and -0 give 0 in both.  The draw weights lie in
// [0, 1] (probabilities and their parts), so the fast loops use this form and
// the walker's recomputation (fix63) sees the same integers.
__device__ __forceinline__ unsigned long long fix63_cvt(float r) {
  return __float2ull_rz(__fmul_rn(r, 0x1p63f));
}

// Whether any element of a row vector is -inf (a masked token, or past V).
template <typename T>
__device__ __forceinline__ bool vec_has_neg_inf(const uint4 x) {
  const uint32_t w[4] = {x.x, x.y, x.z, x.w};
  bool any = false;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    if constexpr (LT<T>::EPV == 8)
      any = any || (w[k] & 0xFFFFu) == 0xFF80u || (w[k] >> 16) == 0xFF80u;
    else
      any = any || w[k] == 0xFF800000u;
  }
  return any;
}

// A float-float as one 64-bit word (hi in the low half) and back.
__device__ __forceinline__ unsigned long long ff_bits(FF v) {
  return (static_cast<unsigned long long>(__float_as_uint(v.lo)) << 32) | __float_as_uint(v.hi);
}
__device__ __forceinline__ FF ff_of_bits(unsigned long long b) {
  return FF{__uint_as_float(static_cast<uint32_t>(b)), __uint_as_float(static_cast<uint32_t>(b >> 32))};
}

// (m, s) <- merge of two (max, sum of weights relative to max) pairs.
__device__ __forceinline__ void ms_merge(float &m, float &s, float m2, float s2, const Ex2c &e) {
  const float mn = fmaxf(m, m2);
  float r = 0.0f;
  if (m > -INFINITY) r = __fmul_rn(s, e(m - mn));
  if (m2 > -INFINITY) r = __fmaf_rn(s2, e(m2 - mn), r);
  m = mn;
  s = r;
}

template <typename T, int NVT>
__global__ void __launch_bounds__(kClNT, 4) sampler_cluster_kernel(const SampParams P) {
  const PdlTail tail{P.pdl_secondary};
  __shared__ ClusterSmem sm;
  constexpr int EPV = LT<T>::EPV;
  constexpr int C = kClusterN;
  const sv_sample_args &a = P.a;
  const Ex2c ex2c{P.c_hi, P.c_lo};
  const uint32_t k = cluster_ctarank();
  const int i = blockIdx.x / C;
  const int tid = threadIdx.x, w = tid >> 5, l = tid & 31;
  if (!seq_rows_ok(a, i)) {            // uniform over the cluster: all CTAs leave
    if (k == 0 && tid == 0) set_status(a.dev_status, SV_DEV_BAD_LENGTH);
    return;
  }
  const int V = a.vocab;
  const int r0 = cuq(a, i), K = cuq(a, i + 1) - r0 - 1, p0 = r0 - i;
  const int nrows = 2 * K + 1;
  const int L = a.kv_len[i];
  const T *tgt = static_cast<const T *>(a.target_logits);
  const T *drf = static_cast<const T *>(a.draft_logits);
  auto row_ptr = [&](int q) -> const T * {
    return q <= K ? tgt + static_cast<int64_t>(r0 + q) * V
                  : drf + static_cast<int64_t>(p0 + q - K - 1) * V;
  };
  const int NV = (V + EPV - 1) / EPV;
  const int per = (NV + C - 1) / C;                  // vectors per CTA slice
  const int v0 = min(NV, static_cast<int>(k) * per), v1 = min(NV, v0 + per);
  const int nv = v1 - v0;

  // ---- the logit at each row's draft token (every CTA needs the probabilities)
  if (tid < nrows) {
    int tok = -1;
    uint32_t bits = 0;
    if (tid != K) {
      const int j = tid < K ? tid : tid - K - 1;
      tok = a.draft_tokens[p0 + j];
      if (tok >= 0 && tok < V) bits = LT<T>::bits(row_ptr(tid)[tok]);
    }
    sm.dtok[tid] = tok;
    sm.dbits[tid] = bits;
  }
  // ---- phase A: slice k of every row into registers, (max, sum) per row
  // Vector j of this thread in row q (elements past V and past the slice read
  // as -inf).
  auto row_vec = [&](int q, int j) -> uint4 {
    const int v = tid + j * kClNT;
    const uint32_t ni = LT<T>::NEG_INF_BITS * (EPV == 8 ? 0x10001u : 1u);
    if (v >= nv) return make_uint4(ni, ni, ni, ni);
    const T *rp = row_ptr(q);
    return load_vec<T>(rp, V, v0 + v, (reinterpret_cast<uintptr_t>(rp) & 15) == 0);
  };
  for (int g0 = 0; g0 < nrows; g0 += kRowGroup) {
    uint4 raw[kRowGroup][NVT];
#pragma unroll
    for (int u = 0; u < kRowGroup; ++u)
#pragma unroll
      for (int j = 0; j < NVT; ++j)
        if (g0 + u < nrows) raw[u][j] = row_vec(g0 + u, j);
    float mx[kRowGroup], sx[kRowGroup];
    uint32_t bad[kRowGroup];
#pragma unroll
    for (int u = 0; u < kRowGroup; ++u) {
      mx[u] = -INFINITY;
      bad[u] = 0;
      if (g0 + u < nrows) {
#pragma unroll
        for (int j = 0; j < NVT; ++j) {
          uint32_t b[EPV];
          unpack<T>(raw[u][j], b);
#pragma unroll
          for (int e = 0; e < EPV; ++e) {
            const float x = LT<T>::val(b[e]);
            bad[u] |= (x != x) || (x == INFINITY);
            mx[u] = fmaxf(mx[u], x);
          }
        }
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
#pragma unroll
      for (int u = 0; u < kRowGroup; ++u) {
        mx[u] = fmaxf(mx[u], __shfl_xor_sync(0xffffffffu, mx[u], o));
        bad[u] |= __shfl_xor_sync(0xffffffffu, bad[u], o);
      }
#pragma unroll
    for (int u = 0; u < kRowGroup; ++u) {
      sx[u] = 0.0f;
      if (g0 + u < nrows && mx[u] > -INFINITY) {
#pragma unroll
        for (int j = 0; j < NVT; ++j) {
          uint32_t b[EPV];
          unpack<T>(raw[u][j], b);
          float t[EPV];
#pragma unroll
          for (int e = 0; e < EPV; ++e) t[e] = ex2c(LT<T>::val(b[e]) - mx[u]);
#pragma unroll
          for (int st = EPV / 2; st > 0; st >>= 1)
#pragma unroll
            for (int e = 0; e < st; ++e) t[e] = __fadd_rn(t[e], t[e + st]);
          sx[u] = __fadd_rn(sx[u], t[0]);
        }
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
#pragma unroll
      for (int u = 0; u < kRowGroup; ++u) sx[u] = __fadd_rn(sx[u], __shfl_xor_sync(0xffffffffu, sx[u], o));
    if (l == 0) {
#pragma unroll
      for (int u = 0; u < kRowGroup; ++u)
        if (g0 + u < nrows) {
          sm.scr.a.redm[g0 + u][w] = mx[u];
          sm.scr.a.reds[g0 + u][w] = sx[u];
          sm.scr.a.redb[g0 + u][w] = bad[u];
        }
    }
  }
  __syncthreads();
  if (tid < nrows) {
    float m = sm.scr.a.redm[tid][0], s = sm.scr.a.reds[tid][0];
    uint32_t bd = sm.scr.a.redb[tid][0];
#pragma unroll
    for (int x = 1; x < kClNW; ++x) {
      ms_merge(m, s, sm.scr.a.redm[tid][x], sm.scr.a.reds[tid][x], ex2c);
      bd |= sm.scr.a.redb[tid][x];
    }
    sm.pm[tid] = m;
    sm.ps[tid] = s;
    sm.pbad[tid] = bd;
  }
  cluster_sync_all();                              // (1) slice statistics of all rows

  // ---- phase B (every CTA): merge row mq from slice mc, C lanes per row
  {
    const int mq = tid / C, mc = tid % C;
    static_assert(kClNT / C * 2 >= kMaxRows, "rows merged in two passes of C-lane groups");
    for (int pass = 0; pass < 2; ++pass) {
      const int q = mq + pass * (kClNT / C);
      const bool live = q < nrows;
      float m = -INFINITY, s = 0.0f;
      uint32_t bd = 0;
      if (live) {
        m = *dsmem(&sm.pm[q], mc);
        s = *dsmem(&sm.ps[q], mc);
        bd = *dsmem(&sm.pbad[q], mc);
      }
#pragma unroll
      for (int o = C / 2; o > 0; o >>= 1) {
        const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
        const float s2 = __shfl_xor_sync(0xffffffffu, s, o);
        bd |= __shfl_xor_sync(0xffffffffu, bd, o);
        ms_merge(m, s, m2, s2, ex2c);
      }
      if (live && mc == 0) {
        const bool ok = !bd && m > -INFINITY && s > 0.0f;
        const float inv = ok ? __frcp_rn(s) : 0.0f;
        sm.st_m[q] = m;
        sm.st_inv[q] = inv;
        sm.st_bad[q] = ok ? 0u : 1u;
        float pd = 0.0f;
        const int tok = sm.dtok[q];
        if (q != K && ok && tok >= 0 && tok < V)
          pd = __fmul_rn(ex2c(LT<T>::val(sm.dbits[q]) - m), inv);
        sm.pdraft[q] = pd;
      }
    }
  }
  __syncthreads();
  // accept tests, lane j for draft j+1 (same decisions in every CTA)
  if (w == 0) {
    // pair l (target row l, draft row l; the bonus row alone at l = K) valid
    const bool pair_ok = l <= K && sm.st_bad[l] == 0 && (l == K || sm.st_bad[K + 1 + l] == 0);
    const unsigned badm = __ballot_sync(0xffffffffu, l <= K && !pair_ok);
    const bool okall = L >= 0;
    const long long sid = a.seq_ids ? a.seq_ids[i] : static_cast<long long>(i);
    bool rej = false, bad = false;
    int d = 0;
    if (okall && l < K && pair_ok) {
      d = sm.dtok[l];
      if (d < 0 || d >= V) {
        rej = bad = true;
      } else {
        const U4 wq = philox4x32_10(U4{static_cast<uint32_t>(L + l + 1),
                                       static_cast<uint32_t>(static_cast<unsigned long long>(sid)),
                                       static_cast<uint32_t>(static_cast<unsigned long long>(sid) >> 32), P.stream},
                                    static_cast<uint32_t>(a.seed), static_cast<uint32_t>(a.seed >> 32));
        const float u = static_cast<float>(u24(wq.x)) * 0x1p-24f;     // exact
        rej = !(__fmul_rn(u, sm.pdraft[K + 1 + l]) < sm.pdraft[l]);
      }
    }
    const unsigned rm = __ballot_sync(0xffffffffu, rej);
    const unsigned bm = __ballot_sync(0xffffffffu, bad);
    // the loop stops at the first rejection or the first invalid pair (only
    // rows it reaches are used)
    const int first_rej = rm ? (__ffs(rm) - 1) : K;
    const int first_bad = badm ? (__ffs(badm) - 1) : K + 1;
    const int n = !okall || first_bad <= first_rej ? -1 : first_rej;
    if (l == 0) sm.n = n;
    if (k == 0) {
      if (l <= K) a.out_tokens[r0 + l] = (n >= 0 && l < n) ? d : -1;
      if (l == 0) {
        a.num_accepted[i] = n;
        if (!okall) set_status(a.dev_status, SV_DEV_BAD_LENGTH);
        else if (n < 0) set_status(a.dev_status, SV_DEV_NONFINITE);
        else if (n < K && ((bm >> n) & 1u)) set_status(a.dev_status, SV_DEV_BAD_TOKEN);
      }
    }
  }
  if (w == 1 && l <= K) {            // draw uniforms for every possible n (position L + n + 1)
    const long long sid = a.seq_ids ? a.seq_ids[i] : static_cast<long long>(i);
    const U4 wv = philox4x32_10(U4{static_cast<uint32_t>(L + l + 1),
                                   static_cast<uint32_t>(static_cast<unsigned long long>(sid)),
                                   static_cast<uint32_t>(static_cast<unsigned long long>(sid) >> 32), P.stream},
                                static_cast<uint32_t>(a.seed), static_cast<uint32_t>(a.seed >> 32));
    sm.draw_u24[l] = u24(wv.y);
  }
  __syncthreads();
  const int n = sm.n;

  // ---- phase C: append slice k of block rows 0..n, run sums of row n
  if (P.do_append) {
    const AppendView &A = P.app;
    if (n < 0) {
      if (k == 0 && tid == 0) A.new_kv_len[i] = L;
    } else {
      const int64_t start = A.kv_start[i];
      const bool cap_ok = L + n + 1 <= A.kv_cap[i];
      const bool pool_ok = start >= 0 && start + L + n + 1 <= A.pool_rows;
      if (cap_ok && pool_ok) {
        const int64_t nvec = static_cast<int64_t>(n + 1) * A.row_bytes / 16;
        const int64_t a0 = nvec * k / C, a1 = nvec * (k + 1) / C;
        const uint4 *sk = reinterpret_cast<const uint4 *>(static_cast<const char *>(A.k_new) +
                                                          static_cast<int64_t>(r0) * A.row_bytes);
        const uint4 *svv = reinterpret_cast<const uint4 *>(static_cast<const char *>(A.v_new) +
                                                           static_cast<int64_t>(r0) * A.row_bytes);
        uint4 *dk = reinterpret_cast<uint4 *>(static_cast<char *>(A.k_cache) + (start + L) * A.row_bytes);
        uint4 *dv = reinterpret_cast<uint4 *>(static_cast<char *>(A.v_cache) + (start + L) * A.row_bytes);
        for (int64_t v = a0 + tid; v < a1; v += kClNT) {
          const uint4 x = __ldcg(sk + v), y = __ldcg(svv + v);
          dk[v] = x;
          dv[v] = y;
        }
      }
      if (k == 0 && tid == 0) {
        if (!cap_ok) set_status(a.dev_status, SV_DEV_CAPACITY);
        else if (!pool_ok) set_status(a.dev_status, SV_DEV_BAD_LENGTH);
        A.new_kv_len[i] = cap_ok && pool_ok ? L + n + 1 : L;
      }
    }
  }
  if (n < 0) {
    cluster_sync_all();                            // no CTA leaves while others read it
    return;
  }
  const int mode = n < K ? 0 : 1;
  const int qt = n, qd = K + 1 + n;                 // target row n, draft row n
  const float mq_ = sm.st_m[qt];
  const int vpt = (per + kClNT - 1) / kClNT;        // vectors per run
  const int ra = min(nv, tid * vpt), rb = min(nv, ra + vpt);
  const T *rq = row_ptr(qt), *rd = row_ptr(qd);
  const bool alq = (reinterpret_cast<uintptr_t>(rq) & 15) == 0;
  const bool ald = (reinterpret_cast<uintptr_t>(rd) & 15) == 0;
  ResidualFn rf;
  rf.init(mq_, mode == 0 ? sm.st_m[qd] : 0.0f, P.c_hi, P.c_lo, FF{P.it_hi, P.it_lo},
          P.it_hi == 1.0f && P.it_lo == 0.0f, sizeof(T) == 4);
  rf.inv_sq = sm.st_inv[qt];
  const float ip = mode == 0 ? sm.st_inv[qd] : 0.0f;
  // ---- C (one pass): the draw weights of row n as two exact fixed-point sums
  // A and B, combined as A + beta * B once beta is known.
  //  * bonus draw, or the empty-residual fallback (use 1): A = q_hat, beta = 0;
  //  * after a rejection (use 0): with L0 = ln(S_p / S_q) from the fp32 sums,
  //    A = q_hat max(0, -expm1(t - L0)) and B = q_hat exp(t - L0) [t < L0]
  //    (q_hat and 0 where p_hat = 0 or q_hat = 0, see ResidualFn), and
  //      G = sum_x q_hat_x expm1(t_x - L0) + sum_{x: q_hat_x = 0} p_hat_x
  //        = (S_p / S_q) exp(-L0) - 1,
  //    a small number (L0 is close) known to a small fraction of the residual
  //    mass itself (summed in float-float).  The exact L satisfies
  //    exp(L - L0) = 1 + G, so where t < L0 the residual at L is
  //    q_hat (1 - exp(t - L0) / (1 + G)) = A + beta * B, beta = G / (1 + G);
  //    only tokens with t between L0 and L (a band of width |L - L0| ~ 1e-6)
  //    are off, by at most q_hat |L - L0|.
  // A and B are 2^-63 fixed-point sums; A + beta * B is evaluated in 128-bit
  // integers from the prefix sums at every decision point, the same function
  // of the same integers everywhere, so the slice, thread and token searches
  // agree.
  const float L0 = mode == 0 ? logf(__fdividef(rf.inv_sq, ip)) : 0.0f;
  rf.L = FF{L0, 0.0f};
  const float mp_ = rf.mp;
  // use 0: the one-pass sums above (and the distances dneg / dpos of the
  // nearest t - L0 below / at-or-above 0, which tell whether the exact L cuts
  // the tokens where L0 did); use 2: the residual at the exact L directly
  // (beta = 0), when it does not; use 1: q_hat.
  float dneg = INFINITY, dpos = INFINITY;
  auto weights = [&](int use, uint32_t bq, uint32_t bd, unsigned long long &wa,
                     unsigned long long &wb, float &gterm) {
    const float lq = LT<T>::val(bq);
    wa = 0;
    wb = 0;
    gterm = 0.0f;
    if (use == 1) {                                // (a masked token weighs 0)
      wa = lq == -INFINITY ? 0ull : fix63(rf.qhat(lq));
      return;
    }
    const float lp = LT<T>::val(bd);
    if (use == 2) {
      wa = fix63(rf(lq, lp));
      return;
    }
    if (lq == -INFINITY) {
      if (lp != -INFINITY) gterm = __fmul_rn(ex2c(lp - mp_), ip);
      return;
    }
    const float qh = rf.qhat(lq);
    if (lp == -INFINITY) {
      wa = fix63(qh);
      gterm = -qh;
      return;
    }
    const float d = rf.arg(lq, lp, rf.L);
    const float em = expm1_fast(d);
    gterm = __fmul_rn(qh, em);
    if (d < 0.0f) {
      wa = fix63(-gterm);
      wb = fix63(__fmaf_rn(qh, em, qh));
      dneg = fminf(dneg, -d);
    } else {
      dpos = fminf(dpos, d);
    }
  };
  FF rf_L_exact = FF{0.0f, 0.0f};
  int use = mode;
  for (int round = 0; round < 3; ++round) {
    unsigned long long sa = 0, sb = 0;
    float gs = 0.0f, gc = 0.0f;                    // Kahan sum of G's terms
    for (int v = ra; v < rb; ++v) {
      const uint4 xq = load_vec<T>(rq, V, v0 + v, alq);
      const uint4 xd = use != 1 ? load_vec<T>(rd, V, v0 + v, ald) : xq;
      const bool masked = vec_has_neg_inf<T>(xq) || (use == 0 && vec_has_neg_inf<T>(xd));
      if (use == 0 && !masked) {
        // every logit finite: weights() of use 0 without branches
#pragma unroll
        for (int e = 0; e < EPV; ++e) {
          const float lq = LT<T>::val(elem_bits<T>(xq, e)), lp = LT<T>::val(elem_bits<T>(xd, e));
          const float qh = rf.qhat(lq);
          const float d = rf.arg(lq, lp, rf.L);
          const float em = expm1_sel(d);
          const float gt = __fmul_rn(qh, em);
          const bool neg = d < 0.0f;
          sa += fix63_cvt(neg ? -gt : 0.0f);
          sb += fix63_cvt(neg ? __fmaf_rn(qh, em, qh) : 0.0f);
          dneg = neg ? fminf(dneg, -d) : dneg;
          dpos = neg ? dpos : fminf(dpos, d);
          const float y = __fsub_rn(gt, gc);
          const float t2 = __fadd_rn(gs, y);
          gc = __fsub_rn(__fsub_rn(t2, gs), y);
          gs = t2;
        }
      } else if (use == 1 && !masked) {
        // the bonus draw (or the empty-residual fallback): q_hat alone
#pragma unroll
        for (int e = 0; e < EPV; ++e) sa += fix63_cvt(rf.qhat(LT<T>::val(elem_bits<T>(xq, e))));
      } else {
#pragma unroll 1
        for (int e = 0; e < EPV; ++e) {
          unsigned long long wa, wb;
          float gt;
          weights(use, elem_bits<T>(xq, e), elem_bits<T>(xd, e), wa, wb, gt);
          sa += wa;
          sb += wb;
          const float y = __fsub_rn(gt, gc);
          const float t2 = __fadd_rn(gs, y);
          gc = __fsub_rn(__fsub_rn(t2, gs), y);
          gs = t2;
        }
      }
    }
    unsigned long long ta, tb = 0;
    const unsigned long long exa = block_exclusive_scan_u64<kClNT>(sa, sm.scan64, &ta);
    __syncthreads();
    const unsigned long long exb =
        use == 0 ? block_exclusive_scan_u64<kClNT>(sb, sm.scan64, &tb) : 0ull;
    if (use == 0) {
      const FF g = warp_sum_ff(FF{gs, -gc});
      dneg = warp_min(dneg);
      dpos = warp_min(dpos);
      if (l == 0) {
        sm.redff[0][w] = g;
        sm.redff[1][w] = FF{dneg, dpos};
      }
      __syncthreads();
    }
    if (tid == 0) {
      FF x = ff_make(0.0f), dd = FF{INFINITY, INFINITY};
      if (use == 0) {
        x = sm.redff[0][0];
        dd = sm.redff[1][0];
#pragma unroll
        for (int q = 1; q < kClNW; ++q) {
          x = ff_add(x, sm.redff[0][q]);
          dd = FF{fminf(dd.hi, sm.redff[1][q].hi), fminf(dd.lo, sm.redff[1][q].lo)};
        }
      }
      // slot k of every CTA's table: this slice's totals and sums, so that
      // after the barrier each CTA's owner search reads only its own memory
      const ulonglong2 t0 = make_ulonglong2(ta, use == 0 ? tb : 0ull);
      const ulonglong2 t1 = make_ulonglong2(ff_bits(x), ff_bits(dd));
#pragma unroll 1
      for (int q = 0; q < C; ++q) {
        ulonglong2 *dst = dsmem(&sm.scr.tab[k][0], static_cast<uint32_t>(q));
        dst[0] = t0;
        dst[1] = t1;
      }
    }
    cluster_sync_all();                            // (2) slice totals and G visible
    // ---- D: every CTA finds the slice holding the target (warp 0)
    if (w == 0) {
      const ulonglong2 t0 = l < C ? sm.scr.tab[l][0] : make_ulonglong2(0ull, 0ull);
      const ulonglong2 t1 = l < C ? sm.scr.tab[l][1] : make_ulonglong2(0ull, 0ull);
      const unsigned long long a0 = t0.x, b0 = t0.y;
      FF gl = l < C ? ff_of_bits(t1.x) : ff_make(0.0f);
      const FF dl = l < C ? ff_of_bits(t1.y) : FF{INFINITY, INFINITY};
      FF G = shfl_ff(gl, 0);
#pragma unroll 1
      for (int q = 1; q < C; ++q) G = ff_add(G, shfl_ff(gl, q));   // the same order everywhere
      // exp(-L) = exp(-L0) / (1 + G): the residual at L is exactly A + beta B
      // with beta = 1 - exp(L0 - L) = G / (1 + G) = G - G^2 + ..., unless L
      // and L0 cut the tokens differently (some t between them), or beta is
      // not small: then an exact pass at L.  No fp64 on this path (it runs
      // at a small fraction of the fp32 rate on this GPU).
      const float Gs = __fadd_rn(G.hi, G.lo);
      const float dL = use == 0 ? log1pf(Gs) : 0.0f;                         // L - L0
      const float nneg = warp_min(dl.hi), npos = warp_min(dl.lo);
      const float margin = __fadd_rn(__fmul_rn(2.0f, fabsf(dL)), 1e-7f);
      const bool big = use == 0 && !(fabsf(G.hi) < 0x1p-14f);
      const bool recut = big || (use == 0 && (dL >= 0.0f ? npos <= margin : nneg <= margin));
      // beta * 2^56 as an integer: G.hi 2^56 is exact; the rest (G.lo - G^2
      // + G^3, below 2^-28 here) rounds to an integer
      const long long beta = use == 0 && !big
          ? __float2ll_rn(__fmul_rn(G.hi, 0x1p56f)) +
            __float2ll_rn(__fmul_rn(__fadd_rn(G.lo, __fmul_rn(__fmul_rn(G.hi, G.hi),
                                                             __fsub_rn(G.hi, 1.0f))),
                                    0x1p56f))
          : 0ll;
      if (recut && l == 0) {
        rf_L_exact = two_sum(L0, dL);
      }
      const unsigned long long ca = warp_inclusive_scan_u64(a0);   // inclusive prefixes over slices
      const unsigned long long cb = warp_inclusive_scan_u64(b0);
      const i128 Z = comb63(__shfl_sync(0xffffffffu, ca, 31), __shfl_sync(0xffffffffu, cb, 31), beta);
      const i128 tg = Z > 0 ? static_cast<i128>(scale_u24(sm.draw_u24[n], static_cast<u128>(Z)))
                            : static_cast<i128>(0);
      const unsigned hit = __ballot_sync(0xffffffffu, l < C && comb63(ca, cb, beta) > tg);
      const int owner = hit ? __ffs(hit) - 1 : C - 1;
      const unsigned long long pa = __shfl_sync(0xffffffffu, ca - a0, owner);
      const unsigned long long pb = __shfl_sync(0xffffffffu, cb - b0, owner);
      if (l == 0) {
        sm.dec_use = recut ? -2 : Z > 0 ? use : -1;
        sm.dec_L = rf_L_exact;
        sm.dec_owner = owner == static_cast<int>(k);
        sm.dec_pa = pa;
        sm.dec_pb = pb;
        sm.dec_beta = beta;
        sm.dec_tg = tg;
        sm.walker = kClNT;
      }
    }
    __syncthreads();
    if (sm.dec_use == -2) {                        // exact pass at L (the same in every CTA)
      rf.L = sm.dec_L;
      use = 2;
      cluster_sync_all();                          // every CTA has read its table (pushed again next round)
      continue;
    }
    if (sm.dec_use < 0) {                          // Z <= 0 (the same in every CTA)
      if (use != 1) {                              // rejected, empty residual: draw from q_hat
        if (k == 0 && tid == 0) set_status(a.dev_status, SV_DEV_EMPTY_RESIDUAL);
        use = 1;
        cluster_sync_all();                        // every CTA has read its table (pushed again next round)
        continue;
      }
      if (k == 0 && tid == 0) a.out_tokens[r0 + n] = -1;   // empty q_hat: not for a valid row
      break;
    }
    // The last round: every access to another CTA's shared memory (phase B's
    // reads, the pushed totals) ended before barrier (2), so the CTAs leave
    // without another cluster barrier and the owner walks alone.
    if (sm.dec_owner) {                            // uniform within the CTA
      const long long beta = sm.dec_beta;
      const i128 tg = sm.dec_tg;
      const unsigned long long pa = sm.dec_pa, pb = sm.dec_pb;
      // the first thread whose run ends past the target
      if (comb63(pa + exa + sa, pb + exb + sb, beta) > tg) atomicMin(&sm.walker, tid);
      __syncthreads();
      const int wt = min(sm.walker, kClNT - 1);
      if (w == (wt >> 5)) {
        // The walker's warp walks its run together: lane e recomputes element
        // e of the run (the same weight bits as the run sums), inclusive
        // scans over the lanes give the running sums, the first lane past the
        // target holds the token.
        static_assert(kClVPT * 8 <= 32, "a run has at most 32 elements");
        const int wra = min(nv, wt * vpt), wrb = min(nv, wra + vpt);
        const int nel = (wrb - wra) * EPV;
        const unsigned long long wxa = __shfl_sync(0xffffffffu, exa, wt & 31);
        const unsigned long long wxb = __shfl_sync(0xffffffffu, exb, wt & 31);
        unsigned long long fa = 0, fb = 0;
        if (l < nel) {
          const int v = wra + l / EPV, e = l % EPV;
          const uint4 xq = load_vec<T>(rq, V, v0 + v, alq);
          const uint4 xd = use != 1 ? load_vec<T>(rd, V, v0 + v, ald) : xq;
          float gt;
          weights(use, elem_bits<T>(xq, e), elem_bits<T>(xd, e), fa, fb, gt);
        }
        fa = warp_inclusive_scan_u64(fa);
        fb = warp_inclusive_scan_u64(fb);
        const unsigned hit =
            __ballot_sync(0xffffffffu, l < nel && comb63(pa + wxa + fa, pb + wxb + fb, beta) > tg);
        const int last = max(nel - 1, 0);
        if (l == 0) a.out_tokens[r0 + n] = (v0 + wra) * EPV + (hit ? __ffs(hit) - 1 : last);
      }
    }
    break;
  }
}

}  // namespace

SamplerPlan plan_sampler(const sv_sample_args &a) {
  SamplerPlan p;
  const int epv = a.dtype == SV_BF16 ? 8 : 4;
  const int nv = (a.vocab + epv - 1) / epv;
  // greedy, top-k and per-sequence parameters take the row path (stat_chunks 1)
  const bool extended = a.temperature == 0.0f || a.top_k > 0 || a.temperatures || a.top_ps ||
                        a.top_ks;
  p.stat_chunks = a.top_p < 1.0f || extended ? 1 : std::max(1, std::min(32, (nv + 1023) / 1024));
  // one run of kDrawVec vectors per thread: chunks of at most kDrawVec * kDrawNT vectors
  p.draw_chunks = std::max(1, std::min(128, (nv + kDrawVec * kDrawNT - 1) / (kDrawVec * kDrawNT)));
  p.draw_threads = kDrawNT;
  // one cluster per sequence when there is no nucleus and the rows' slices fit
  const int per = (nv + kClusterN - 1) / kClusterN;
  p.cluster_nvt = per > kClNT ? 2 : 1;
  p.cluster = a.top_p >= 1.0f && !extended && per <= kClVPT * kClNT;
  // bf16 rows off the cluster path: the window-histogram statistics kernel
  p.win_stats = a.dtype == SV_BF16 ? 1 : 0;
  if (p.win_stats) p.stat_chunks = 1;
  return p;
}

int sampler_max_vocab(int dtype) {
  return kMaxTiles * kSampNT * (dtype == SV_BF16 ? 8 : 4);
}

int sampler_cluster_smem(const SamplerPlan &p) {
  return p.cluster ? static_cast<int>(sizeof(ClusterSmem)) : 0;
}

template <typename T>
static cudaError_t launch_cluster(const SampParams &P, cudaStream_t s) {
  auto kern = P.plan.cluster_nvt == 2 ? sampler_cluster_kernel<T, 2> : sampler_cluster_kernel<T, 1>;
  const int smem = 0;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                                       cudaSharedmemCarveoutMaxShared);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(P.a.batch * kClusterN);
  cfg.blockDim = dim3(kClNT);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kClusterN;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = P.pdl_secondary ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, kern, P);
}

// Launch of the first kernel of a path, early (programmatic) when the sampler
// runs behind another grid.
template <typename K>
static cudaError_t launch_first(K kern, int grid, int block, size_t smem, const SampParams &P,
                                cudaStream_t s) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(block);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = P.pdl_secondary ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, P);
}

template <typename T>
static cudaError_t launch_t(const SampParams &P, cudaStream_t s) {
  const int rows = static_cast<int>(2 * P.a.num_rows - P.a.batch);
  cudaError_t e;
  if (P.plan.cluster) {
    e = launch_cluster<T>(P, s);
    if (e == cudaSuccess) return e;
    (void)cudaGetLastError();          // no room for a cluster: two-kernel path
  }
  const bool win = P.plan.win_stats != 0;
  if (win) {
    // ring depth 16: a 32k row is read whole at once (16 vectors per thread)
    constexpr int kStages = 16;
    auto kern = stats_win_kernel<kStages>;
    const int stages = kStages;
    const int smem = static_cast<int>(kWinSmemOff) + stages * kWinNT * 16;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    e = launch_first(kern, rows, kWinNT, static_cast<size_t>(smem), P, s);
  } else if (P.plan.stat_chunks > 1) {
    e = launch_first(stats_chunk_kernel<T>, rows * P.plan.stat_chunks, kStatNT, 0, P, s);
  } else {
    const size_t smem = kSmemRowOff + kRowSmemBytes;
    e = cudaFuncSetAttribute(stats_row_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    e = launch_first(stats_row_kernel<T>, rows, kSampNT, smem, P, s);
  }
  if (e != cudaSuccess) return e;
  // behind the window statistics kernel the draw starts early (it waits for
  // the statistics grid before reading anything)
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(P.a.batch * P.plan.draw_chunks);
  cfg.blockDim = dim3(kDrawNT);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = win ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, draw_kernel<T>, P);
}

// 2^(j/64) for j = -32..32 as float-float pairs, from double precision
// (built once, thread-safe static initialization).
struct Exp2Table {
  float2 v[kExp2Tab];
  Exp2Table() {
    for (int t = 0; t < kExp2Tab; ++t) {
      const double x = std::exp2(static_cast<double>(t - 32) / 64.0);
      const float hi = static_cast<float>(x);
      v[t] = make_float2(hi, static_cast<float>(x - static_cast<double>(hi)));
    }
  }
};
static const float2 *exp2_table_host() {
  static const Exp2Table tab;
  return tab.v;
}

cudaError_t launch_sampler(const SamplerLaunch &L, cudaStream_t s) {
  SampParams P;
  const float2 *tab = exp2_table_host();
  for (int t = 0; t < kExp2Tab; ++t) P.exp2tab[t] = tab[t];
  P.a = L.a;
  P.ws = L.ws;
  P.plan = L.plan;
  P.do_append = L.do_append ? 1 : 0;
  P.app = L.app;
  const double c = 1.4426950408889634 / static_cast<double>(L.a.temperature);
  P.c_hi = static_cast<float>(c);
  P.c_lo = static_cast<float>(c - static_cast<double>(P.c_hi));
  const double it = 1.0 / static_cast<double>(L.a.temperature);
  P.it_hi = static_cast<float>(it);
  P.it_lo = static_cast<float>(it - static_cast<double>(P.it_hi));
  P.pdl_secondary = L.pdl_secondary ? 1 : 0;
  P.stream = L.philox_stream;
  if (2 * L.a.num_rows - L.a.batch <= 0) return cudaSuccess;
  return L.a.dtype == SV_BF16 ? launch_t<uint16_t>(P, s) : launch_t<float>(P, s);
}

}  // namespace sv

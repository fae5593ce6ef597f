// Modified rejection sampling for a padding-free batch (sm_103a).
//
// Method: "Accelerating Large Language Model Decoding with Speculative
// Sampling" (Chen et al.), section "Modified rejection sampling": accept draft
// x~ with probability min(1, q(x~)/p(x~)), left to right, stop at the first
// rejection and draw from (q - p)_+ ; if all K drafts pass, draw a bonus token
// from the last target row.  Same section: temperature / nucleus modify the
// probabilities before the scheme.  Batch without padding: EMS-SD abstract.
//
// Kernel layout: one CTA per logits row (target rows 0..R-1, then draft rows).
// Each CTA streams its row once from HBM (max), then re-reads it from L2 for
// the weight sum and, with top_p < 1, for the nucleus cut.  The last CTA of a
// sequence to finish (atomic arrival count, no waiting) takes that sequence's
// decisions, draws its token and, in the fused step, appends its accepted K/V
// rows.
//
// Precision: per-element weights exp((l - lmax)/T) are fp32 (exp2f with the
// constant log2(e)/T held as two floats); sums use Kahan fp32 per thread and
// fp64 across threads; the accept test is evaluated in fp64; the inverse-CDF
// draw accumulates exact 64-bit fixed-point values (2^-52 units), so the
// chosen index does not depend on the summation order.
#include "common.cuh"
#include "kernels.h"

namespace sv {

namespace {

constexpr int kSampNT = 512;          // threads per sampler CTA
constexpr int kSampNW = kSampNT / 32;
constexpr int kMaxTiles = 64;         // vectors per thread per row (bounds V)
constexpr int kCandCap = 4096;        // nucleus candidates held in shared memory
constexpr float kFix = 4503599627370496.0f;  // 2^52

template <typename T> struct LT;
template <> struct LT<float> {
  static constexpr int EPV = 4;
  static constexpr int KEY_BITS = 32;
  static constexpr uint32_t NEG_INF_BITS = 0xFF800000u;
  __device__ static float val(uint32_t b) { return __uint_as_float(b); }
  __device__ static uint32_t key(uint32_t b) { return key_of_f32(b); }
};
template <> struct LT<uint16_t> {
  static constexpr int EPV = 8;
  static constexpr int KEY_BITS = 16;
  static constexpr uint32_t NEG_INF_BITS = 0xFF80u;
  __device__ static float val(uint32_t b) { return bf16_bits_to_f32(b); }
  __device__ static uint32_t key(uint32_t b) { return key_of_bf16(b); }
};

// Raw bits of the EPV elements of vector v (elements v*EPV ..); past-the-end
// elements read as -inf (weight 0, lowest key).
template <typename T>
__device__ __forceinline__ void load_bits(const T *row, int V, int v, bool aligned,
                                          uint32_t (&b)[LT<T>::EPV]) {
  constexpr int EPV = LT<T>::EPV;
  const int e0 = v * EPV;
  if (aligned && e0 + EPV <= V) {
    const uint4 raw = __ldg(reinterpret_cast<const uint4 *>(row + e0));
    if constexpr (EPV == 4) {
      b[0] = raw.x; b[1] = raw.y; b[2] = raw.z; b[3] = raw.w;
    } else {
      const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        b[2 * i] = w[i] & 0xFFFFu;
        b[2 * i + 1] = w[i] >> 16;
      }
    }
  } else {
#pragma unroll
    for (int i = 0; i < EPV; ++i)
      b[i] = (e0 + i < V) ? static_cast<uint32_t>(__ldg(row + e0 + i)) : LT<T>::NEG_INF_BITS;
  }
}

// exp((l - lmax) / T) in fp32, with c = log2(e) / T split as c_hi + c_lo.
// Explicit round-to-nearest intrinsics: every pass recomputes identical bits.
struct WeightFn {
  float lmax, c_hi, c_lo;
  __device__ __forceinline__ float operator()(float l) const {
    if (l == -INFINITY) return 0.0f;
    const float dl = __fsub_rn(l, lmax);
    return exp2f(__fmaf_rn(dl, c_hi, __fmul_rn(dl, c_lo)));
  }
};

struct SampParams {
  sv_sample_args a;
  RowStats *stats;
  uint32_t *counters;
  int do_append;
  AppendView app;
  float c_hi, c_lo;   // log2(e)/T as two floats
  double inv_T;
  int pdl_primary;
};

struct SampSmem {
  double red[32];
  float redf[32];
  unsigned long long red64[32];
  unsigned long long wsum[kMaxTiles][kSampNW];
  unsigned long long tile_tot[kMaxTiles];
  unsigned long long bcast64[4];
  int bcast[8];
  uint32_t cand_key[kCandCap];
  float cand_w[kCandCap];
};

// Validity of sequence i's row bookkeeping against the host bounds.
__device__ __forceinline__ bool seq_rows_ok(const sv_sample_args &a, int i) {
  const int r0 = a.cu_q[i], r1 = a.cu_q[i + 1];
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
// picks a candidate set that surely contains the cut; the exact bitwise search
// then runs over those candidates in shared memory (or, if there are too
// many, over the whole row).
// --------------------------------------------------------------------------
template <typename T>
__device__ void nucleus_cut(const T *row, int V, bool aligned, const WeightFn &wf, double S,
                            float top_p, SampSmem &sm, uint32_t &tau_out, double &ssum_out) {
  constexpr int EPV = LT<T>::EPV;
  const int NV = (V + EPV - 1) / EPV;
  const int tid = threadIdx.x;
  const double target = static_cast<double>(top_p) * S;

  // coarse bins: bin b = min((127 - biased_exp(w)) / 4, 7)
  float acc[8];
#pragma unroll
  for (int b = 0; b < 8; ++b) acc[b] = 0.0f;
  for (int v = tid; v < NV; v += kSampNT) {
    uint32_t bits[EPV];
    load_bits<T>(row, V, v, aligned, bits);
#pragma unroll
    for (int e = 0; e < EPV; ++e) {
      const float w = wf(LT<T>::val(bits[e]));
      const int ex = 127 - static_cast<int>((__float_as_uint(w) >> 23) & 0xFFu);
      const int b = min(max(ex, 0) >> 2, 7);
#pragma unroll
      for (int k = 0; k < 8; ++k) acc[k] += (b == k) ? w : 0.0f;
    }
  }
  double cum = 0.0;
  int kb = 7;
  for (int k = 0; k < 8; ++k) {
    cum += block_sum_d<kSampNT>(static_cast<double>(acc[k]), sm.red);
    if (kb == 7 && k < 7 && cum >= target * (1.0 + 1e-5)) kb = k;
  }
  // candidates: bin <= kb (all elements when kb == 7)
  auto is_cand = [&](float w) {
    if (kb == 7) return true;
    const int ex = 127 - static_cast<int>((__float_as_uint(w) >> 23) & 0xFFu);
    return (max(ex, 0) >> 2) <= kb;
  };
  int mine = 0;
  for (int v = tid; v < NV; v += kSampNT) {
    uint32_t bits[EPV];
    load_bits<T>(row, V, v, aligned, bits);
#pragma unroll
    for (int e = 0; e < EPV; ++e) mine += is_cand(wf(LT<T>::val(bits[e]))) ? 1 : 0;
  }
  unsigned long long total = 0;
  const unsigned long long off =
      block_exclusive_scan_u64<kSampNT>(static_cast<unsigned long long>(mine), sm.red64, &total);
  const bool in_smem = total <= static_cast<unsigned long long>(kCandCap);
  if (in_smem) {
    int o = static_cast<int>(off);
    for (int v = tid; v < NV; v += kSampNT) {
      uint32_t bits[EPV];
      load_bits<T>(row, V, v, aligned, bits);
#pragma unroll
      for (int e = 0; e < EPV; ++e) {
        const float w = wf(LT<T>::val(bits[e]));
        if (is_cand(w)) {
          sm.cand_key[o] = LT<T>::key(bits[e]);
          sm.cand_w[o] = w;
          ++o;
        }
      }
    }
  }
  __syncthreads();
  const int C = static_cast<int>(total);
  // partial weight of {key >= cand} held by this thread
  auto partial = [&](uint32_t cand) {
    float s = 0.0f;
    if (in_smem) {
      for (int c = tid; c < C; c += kSampNT)
        if (sm.cand_key[c] >= cand) s += sm.cand_w[c];
    } else {
      for (int v = tid; v < NV; v += kSampNT) {
        uint32_t bits[EPV];
        load_bits<T>(row, V, v, aligned, bits);
#pragma unroll
        for (int e = 0; e < EPV; ++e)
          if (LT<T>::key(bits[e]) >= cand) s += wf(LT<T>::val(bits[e]));
      }
    }
    return s;
  };
  uint32_t tau = 0;
  for (int bit = LT<T>::KEY_BITS - 1; bit >= 0; --bit) {
    const uint32_t cand = tau | (1u << bit);
    const double W = block_sum_d<kSampNT>(static_cast<double>(partial(cand)), sm.red);
    if (W >= target) tau = cand;
  }
  ssum_out = block_sum_d<kSampNT>(static_cast<double>(partial(tau)), sm.red);
  tau_out = tau;
}

// --------------------------------------------------------------------------
// Inverse-CDF draw over one vocabulary row (block-wide).  mode 0: residual
// max(0, q_hat - p_hat) of (trow, drow); mode 1: q_hat of trow.  Returns the
// first index x with C(x) * 2^24 > k * Z (C, Z in 2^-52 fixed point), or -1
// when Z == 0.
// --------------------------------------------------------------------------
struct RowProb {      // q_hat(l) = [key(l) >= tau] * w(l) / S, w(l) = exp((l-lmax)/T)
  WeightFn wf;
  uint32_t tau;
  float inv_hi, inv_lo;  // 1/S as two floats
};

template <typename T>
__device__ __forceinline__ float row_prob(const RowProb &rp, uint32_t bits) {
  if (LT<T>::key(bits) < rp.tau) return 0.0f;
  const float w = rp.wf(LT<T>::val(bits));
  return __fmaf_rn(w, rp.inv_hi, __fmul_rn(w, rp.inv_lo));
}

template <typename T>
__device__ __forceinline__ unsigned long long vec_fix_sum(const T *trow, const T *drow, int V,
                                                          bool al_t, bool al_d, int v,
                                                          const RowProb &pq, const RowProb &pp,
                                                          int mode) {
  constexpr int EPV = LT<T>::EPV;
  uint32_t bq[EPV], bp[EPV];
  load_bits<T>(trow, V, v, al_t, bq);
  if (mode == 0) load_bits<T>(drow, V, v, al_d, bp);
  unsigned long long s = 0;
#pragma unroll
  for (int e = 0; e < EPV; ++e) {
    float r = row_prob<T>(pq, bq[e]);
    if (mode == 0) r = fmaxf(__fsub_rn(r, row_prob<T>(pp, bp[e])), 0.0f);
    s += __float2ull_rz(__fmul_rn(r, kFix));
  }
  return s;
}

template <typename T>
__device__ int block_draw(const T *trow, const T *drow, int V, const RowProb &pq,
                          const RowProb &pp, int mode, uint32_t k24, SampSmem &sm) {
  constexpr int EPV = LT<T>::EPV;
  const int NV = (V + EPV - 1) / EPV;
  const int NK = (NV + kSampNT - 1) / kSampNT;
  const int tid = threadIdx.x, w = tid >> 5, l = tid & 31;
  const bool al_t = (reinterpret_cast<uintptr_t>(trow) & 15) == 0;
  const bool al_d = mode == 0 && (reinterpret_cast<uintptr_t>(drow) & 15) == 0;
  for (int k = 0; k < NK; ++k) {
    const int v = k * kSampNT + tid;
    unsigned long long s = v < NV ? vec_fix_sum<T>(trow, drow, V, al_t, al_d, v, pq, pp, mode) : 0;
    s = warp_sum_u64(s);
    if (l == 0) sm.wsum[k][w] = s;
  }
  __syncthreads();
  if (tid < NK) {
    unsigned long long t = 0;
    for (int i = 0; i < kSampNW; ++i) t += sm.wsum[tid][i];
    sm.tile_tot[tid] = t;
  }
  __syncthreads();
  if (tid == 0) {
    unsigned long long Z = 0;
    for (int k = 0; k < NK; ++k) Z += sm.tile_tot[k];
    int kstar = -1;
    unsigned long long tgt = 0, base = 0;
    if (Z > 0) {
      const unsigned long long ku = k24;
      const unsigned long long lo = ku * Z, hi = __umul64hi(ku, Z);
      tgt = (hi << 40) | (lo >> 24);            // floor(k * Z / 2^24) < Z
      unsigned long long cum = 0;
      for (int k = 0; k < NK; ++k) {
        if (tgt < cum + sm.tile_tot[k]) { kstar = k; base = cum; break; }
        cum += sm.tile_tot[k];
      }
    }
    sm.bcast[0] = kstar;
    sm.bcast[1] = -1;
    sm.bcast64[0] = tgt;
    sm.bcast64[1] = base;
  }
  __syncthreads();
  const int kstar = sm.bcast[0];
  if (kstar < 0) return -1;
  const unsigned long long tgt = sm.bcast64[0], base = sm.bcast64[1];
  const int v = kstar * kSampNT + tid;
  const unsigned long long s = v < NV ? vec_fix_sum<T>(trow, drow, V, al_t, al_d, v, pq, pp, mode) : 0;
  unsigned long long dummy;
  const unsigned long long ex = block_exclusive_scan_u64<kSampNT>(s, sm.red64, &dummy);
  const unsigned long long lo_c = base + ex;
  if (s > 0 && lo_c <= tgt && tgt < lo_c + s) {
    // owner: walk the vector element by element with the same arithmetic
    uint32_t bq[EPV], bp[EPV];
    load_bits<T>(trow, V, v, al_t, bq);
    if (mode == 0) load_bits<T>(drow, V, v, al_d, bp);
    unsigned long long c = lo_c;
    int x = v * EPV + EPV - 1;
#pragma unroll
    for (int e = 0; e < EPV; ++e) {
      float r = row_prob<T>(pq, bq[e]);
      if (mode == 0) r = fmaxf(__fsub_rn(r, row_prob<T>(pp, bp[e])), 0.0f);
      c += __float2ull_rz(__fmul_rn(r, kFix));
      if (c > tgt) { x = v * EPV + e; break; }
    }
    sm.bcast[1] = x;
  }
  __syncthreads();
  return sm.bcast[1];
}

__device__ __forceinline__ RowProb make_rowprob(const RowStats &st, float c_hi, float c_lo) {
  RowProb r;
  r.wf = WeightFn{st.lmax, c_hi, c_lo};
  r.tau = st.tau_key;
  const double inv = 1.0 / st.ssum;
  r.inv_hi = static_cast<float>(inv);
  r.inv_lo = static_cast<float>(inv - static_cast<double>(r.inv_hi));
  return r;
}

// Copy block rows 0..n of sequence i to pool rows kv_start + L .. (fused step).
__device__ void append_seq(const SampParams &P, int i, int r0, int n, int L, uint32_t *status) {
  const AppendView &A = P.app;
  int32_t new_len = L;
  const int64_t start = A.kv_start[i];
  if (L + n + 1 > A.kv_cap[i]) {
    if (threadIdx.x == 0) set_status(status, SV_DEV_CAPACITY);
  } else if (start < 0 || start + L + n + 1 > A.pool_rows) {
    if (threadIdx.x == 0) set_status(status, SV_DEV_BAD_LENGTH);
  } else {
    const int64_t nvec = static_cast<int64_t>(n + 1) * A.row_bytes / 16;
    const uint4 *sk = reinterpret_cast<const uint4 *>(static_cast<const char *>(A.k_new) +
                                                      static_cast<int64_t>(r0) * A.row_bytes);
    const uint4 *sv_ = reinterpret_cast<const uint4 *>(static_cast<const char *>(A.v_new) +
                                                       static_cast<int64_t>(r0) * A.row_bytes);
    uint4 *dk = reinterpret_cast<uint4 *>(static_cast<char *>(A.k_cache) +
                                          (start + L) * A.row_bytes);
    uint4 *dv = reinterpret_cast<uint4 *>(static_cast<char *>(A.v_cache) +
                                          (start + L) * A.row_bytes);
    for (int64_t v = threadIdx.x; v < nvec; v += kSampNT) {
      dk[v] = __ldcg(sk + v);
      dv[v] = __ldcg(sv_ + v);
    }
    new_len = L + n + 1;
  }
  if (threadIdx.x == 0) A.new_kv_len[i] = new_len;
}

// --------------------------------------------------------------------------
// Decision for sequence i, run by the last row CTA of i to finish.
// --------------------------------------------------------------------------
template <typename T>
__device__ void decide_sequence(const SampParams &P, int i, SampSmem &sm) {
  const sv_sample_args &a = P.a;
  const int V = a.vocab, R = static_cast<int>(a.num_rows);
  const int r0 = a.cu_q[i], K = a.cu_q[i + 1] - r0 - 1, p0 = r0 - i;
  const int L = a.kv_len[i];
  const long long sid = a.seq_ids ? a.seq_ids[i] : static_cast<long long>(i);
  const int tid = threadIdx.x;
  const T *tgt = static_cast<const T *>(a.target_logits);
  const T *drf = static_cast<const T *>(a.draft_logits);

  // all rows valid?
  int ok = 1;
  if (tid <= K) ok = __ldcg(&P.stats[r0 + tid].valid) != 0;
  if (tid < K) ok = ok && (__ldcg(&P.stats[R + p0 + tid].valid) != 0);
  ok = __syncthreads_and(ok);
  if (!ok || L < 0) {
    if (tid <= K) a.out_tokens[r0 + tid] = -1;
    if (tid == 0) {
      a.num_accepted[i] = -1;
      set_status(a.dev_status, L < 0 ? SV_DEV_BAD_LENGTH : SV_DEV_NONFINITE);
      if (P.do_append) P.app.new_kv_len[i] = L;
    }
    return;
  }
  const uint32_t k0 = static_cast<uint32_t>(a.seed), k1 = static_cast<uint32_t>(a.seed >> 32);
  const uint32_t sid_lo = static_cast<uint32_t>(static_cast<unsigned long long>(sid));
  const uint32_t sid_hi = static_cast<uint32_t>(static_cast<unsigned long long>(sid) >> 32);

  // accept tests, one lane per draft row (K <= 15)
  if (tid < 32) {
    bool rej = false, bad = false;
    if (tid < K) {
      const int d = a.draft_tokens[p0 + tid];
      if (d < 0 || d >= V) {
        rej = bad = true;
      } else {
        RowStats sq, sp;
        sq.lmax = __ldcg(&P.stats[r0 + tid].lmax);
        sq.tau_key = __ldcg(&P.stats[r0 + tid].tau_key);
        sq.ssum = __ldcg(&P.stats[r0 + tid].ssum);
        sp.lmax = __ldcg(&P.stats[R + p0 + tid].lmax);
        sp.tau_key = __ldcg(&P.stats[R + p0 + tid].tau_key);
        sp.ssum = __ldcg(&P.stats[R + p0 + tid].ssum);
        const uint32_t bq = static_cast<uint32_t>(tgt[static_cast<int64_t>(r0 + tid) * V + d]);
        const uint32_t bp = static_cast<uint32_t>(drf[static_cast<int64_t>(p0 + tid) * V + d]);
        const double lq = LT<T>::val(bq), lp = LT<T>::val(bp);
        const double qh = LT<T>::key(bq) >= sq.tau_key
                              ? exp((lq - static_cast<double>(sq.lmax)) * P.inv_T) / sq.ssum
                              : 0.0;
        const double ph = LT<T>::key(bp) >= sp.tau_key
                              ? exp((lp - static_cast<double>(sp.lmax)) * P.inv_T) / sp.ssum
                              : 0.0;
        const U4 w = philox4x32_10(U4{static_cast<uint32_t>(L + tid + 1), sid_lo, sid_hi, 0u}, k0, k1);
        const double u = static_cast<double>(u24(w.x)) * 0x1p-24;
        rej = !(u * ph < qh);
      }
    }
    const unsigned rm = __ballot_sync(0xffffffffu, rej);
    const unsigned bm = __ballot_sync(0xffffffffu, bad);
    if (tid == 0) {
      const int n = rm ? (__ffs(rm) - 1) : K;
      sm.bcast[2] = n;
      if (n < K && ((bm >> n) & 1u)) set_status(a.dev_status, SV_DEV_BAD_TOKEN);
    }
  }
  __syncthreads();
  const int n = sm.bcast[2];

  // draw at row n: residual (n < K) or bonus (n == K)
  const U4 wv = philox4x32_10(U4{static_cast<uint32_t>(L + n + 1), sid_lo, sid_hi, 0u}, k0, k1);
  const uint32_t ks = u24(wv.y);
  RowStats sq;
  sq.lmax = __ldcg(&P.stats[r0 + n].lmax);
  sq.tau_key = __ldcg(&P.stats[r0 + n].tau_key);
  sq.ssum = __ldcg(&P.stats[r0 + n].ssum);
  const RowProb pq = make_rowprob(sq, P.c_hi, P.c_lo);
  const T *trow = tgt + static_cast<int64_t>(r0 + n) * V;
  int x;
  if (n < K) {
    RowStats sp;
    sp.lmax = __ldcg(&P.stats[R + p0 + n].lmax);
    sp.tau_key = __ldcg(&P.stats[R + p0 + n].tau_key);
    sp.ssum = __ldcg(&P.stats[R + p0 + n].ssum);
    const RowProb pp = make_rowprob(sp, P.c_hi, P.c_lo);
    x = block_draw<T>(trow, drf + static_cast<int64_t>(p0 + n) * V, V, pq, pp, 0, ks, sm);
    if (x < 0) {
      if (tid == 0) set_status(a.dev_status, SV_DEV_EMPTY_RESIDUAL);
      x = block_draw<T>(trow, trow, V, pq, pq, 1, ks, sm);
    }
  } else {
    x = block_draw<T>(trow, trow, V, pq, pq, 1, ks, sm);
  }
  if (tid <= K) {
    int tok = -1;
    if (tid < n) tok = a.draft_tokens[p0 + tid];
    else if (tid == n) tok = x;
    a.out_tokens[r0 + tid] = tok;
  }
  if (tid == 0) a.num_accepted[i] = n;
  if (P.do_append) append_seq(P, i, r0, n, L, a.dev_status);
}

template <typename T>
__global__ void __launch_bounds__(kSampNT) sampler_kernel(const SampParams P) {
  if (P.pdl_primary) asm volatile("griddepcontrol.launch_dependents;\n");
  extern __shared__ __align__(16) unsigned char smem_raw[];
  SampSmem &sm = *reinterpret_cast<SampSmem *>(smem_raw);
  const sv_sample_args &a = P.a;
  const int V = a.vocab, R = static_cast<int>(a.num_rows), B = a.batch;
  const int r = blockIdx.x;
  const int tid = threadIdx.x;

  int i;
  const T *row;
  if (r < R) {
    i = seq_of_target_row(a.cu_q, B, r);
    row = static_cast<const T *>(a.target_logits) + static_cast<int64_t>(r) * V;
  } else {
    i = seq_of_draft_row(a.cu_q, B, r - R);
    row = static_cast<const T *>(a.draft_logits) + static_cast<int64_t>(r - R) * V;
  }
  if (!seq_rows_ok(a, i)) {
    if (tid == 0) set_status(a.dev_status, SV_DEV_BAD_LENGTH);
    return;
  }
  constexpr int EPV = LT<T>::EPV;
  const int NV = (V + EPV - 1) / EPV;
  const bool aligned = (reinterpret_cast<uintptr_t>(row) & 15) == 0;

  // pass 1: max and finiteness (streams the row from HBM)
  float mx = -INFINITY;
  int bad = 0;
  for (int v = tid; v < NV; v += kSampNT) {
    uint32_t bits[EPV];
    load_bits<T>(row, V, v, aligned, bits);
#pragma unroll
    for (int e = 0; e < EPV; ++e) {
      const float x = LT<T>::val(bits[e]);
      bad |= (x != x) || (x == INFINITY);
      mx = fmaxf(mx, x);
    }
  }
  bad = __syncthreads_or(bad);
  mx = block_max_f<kSampNT>(mx, sm.redf);
  const bool valid = !bad && mx > -INFINITY;
  uint32_t tau = 0;
  double ssum = 1.0;
  if (valid) {
    const WeightFn wf{mx, P.c_hi, P.c_lo};
    // pass 2: sum of weights (Kahan per thread, fp64 across threads)
    float s = 0.0f, comp = 0.0f;
    for (int v = tid; v < NV; v += kSampNT) {
      uint32_t bits[EPV];
      load_bits<T>(row, V, v, aligned, bits);
#pragma unroll
      for (int e = 0; e < EPV; ++e) {
        const float y = __fsub_rn(wf(LT<T>::val(bits[e])), comp);
        const float t = __fadd_rn(s, y);
        comp = __fsub_rn(__fsub_rn(t, s), y);
        s = t;
      }
    }
    const double S = block_sum_d<kSampNT>(static_cast<double>(s) - static_cast<double>(comp), sm.red);
    if (a.top_p < 1.0f) {
      nucleus_cut<T>(row, V, aligned, wf, S, a.top_p, sm, tau, ssum);
    } else {
      ssum = S;
    }
  }
  if (tid == 0) {
    RowStats st;
    st.lmax = mx;
    st.tau_key = tau;
    st.valid = valid ? 1u : 0u;
    st.pad = 0;
    st.ssum = ssum;
    P.stats[r] = st;
    __threadfence();
    const int nrows = 2 * (a.cu_q[i + 1] - a.cu_q[i]) - 1;
    const unsigned old = atomicInc(&P.counters[i], static_cast<unsigned>(nrows - 1));
    sm.bcast[3] = (old == static_cast<unsigned>(nrows - 1)) ? 1 : 0;
  }
  __syncthreads();
  if (sm.bcast[3]) {
    __threadfence();
    decide_sequence<T>(P, i, sm);
  }
}

}  // namespace

size_t sampler_stats_bytes(const sv_sample_args &a) {
  return static_cast<size_t>(2 * a.num_rows - a.batch) * sizeof(RowStats);
}

int sampler_max_vocab(int dtype) {
  return kMaxTiles * kSampNT * (dtype == SV_BF16 ? 8 : 4);
}

cudaError_t launch_sampler(const SamplerLaunch &L, cudaStream_t s) {
  SampParams P;
  P.a = L.a;
  P.stats = L.stats;
  P.counters = L.counters;
  P.do_append = L.do_append ? 1 : 0;
  P.app = L.app;
  const double c = 1.4426950408889634 / static_cast<double>(L.a.temperature);
  P.c_hi = static_cast<float>(c);
  P.c_lo = static_cast<float>(c - static_cast<double>(P.c_hi));
  P.inv_T = 1.0 / static_cast<double>(L.a.temperature);
  P.pdl_primary = L.pdl_primary ? 1 : 0;
  const int grid = static_cast<int>(2 * L.a.num_rows - L.a.batch);
  if (grid <= 0) return cudaSuccess;
  const size_t smem = sizeof(SampSmem);
  cudaError_t e;
  if (L.a.dtype == SV_BF16) {
    e = cudaFuncSetAttribute(sampler_kernel<uint16_t>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    sampler_kernel<uint16_t><<<grid, kSampNT, smem, s>>>(P);
  } else {
    e = cudaFuncSetAttribute(sampler_kernel<float>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    sampler_kernel<float><<<grid, kSampNT, smem, s>>>(P);
  }
  return cudaGetLastError();
}

}  // namespace sv

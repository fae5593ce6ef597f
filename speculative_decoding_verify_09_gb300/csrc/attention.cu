// Ragged split-KV verify attention (sm_103a).
//
// What is computed: for sequence i, query head h and block row j,
//   out = softmax(scale * q . k) v  over the keys  [kv cache rows of i] ++
//   [block rows 0..j of i]   (KV head h / (Hq/Hkv)),
// i.e. the K_i + 1 rows scored in one target call ("Accelerating Large
// Language Model Decoding with Speculative Sampling", section "Conditional
// scoring"), over a batch with different lengths and no padding (BASS and
// EMS-SD abstracts).  Attention over the KV cache is memory-bound and its cost
// does not grow with K (same section), so the kernel is built to stream KV
// bytes at HBM rate:
//
//  * Work unit: a 64-key tile of one (sequence, KV head) segment.  The
//    (K_i + 1) x (Hq/Hkv) query rows sharing that KV head are packed as the M
//    dimension, so every KV byte is read once for all of them (GQA).
//  * Stream-K split: the global tile sequence (segments in order) is cut into
//    gridDim.x equal contiguous ranges, one per persistent CTA, regardless of
//    segment boundaries.  A CTA that covers a whole segment writes the output
//    directly; otherwise each piece writes a partial (unnormalized O, row max,
//    row sum) and the last piece to arrive (atomic count, no waiting) merges
//    them.  Balance is within one tile per CTA for any length mix.
//  * Tiles are staged with a 3-stage cp.async pipeline (16-byte copies, rows
//    XOR-swizzled in shared memory), which runs across segment boundaries.
//  * Q.K^T and P.V use mma.sync m16n8k16 (bf16 in, fp32 accumulate); the
//    probabilities stay in registers between the two products.  Online softmax
//    per warp uses quad shuffles.  Four warps split each tile's 64 keys; their
//    states are merged in shared memory at the end of a piece.
//
// fp32 inputs use a CUDA-core kernel (one CTA per segment, fp32 FMA).
#include <algorithm>

#include "common.cuh"
#include "kernels.h"

namespace sv {

namespace {

constexpr int kTileKeys = 64;
constexpr int kStages = 3;
constexpr int kKW = 4;            // warps splitting the keys of one tile
constexpr int kMaxBatch = 1024;   // sequences per call (schedule held in smem)
constexpr int kMaxGroups = 256;   // shared-prefix groups per call
constexpr float kLog2e = 1.4426950408889634f;

struct AttnParams {
  int B, Hq, Hkv, g, max_q_rows;
  int64_t num_rows, pool_rows;
  float sl2;                      // scale * log2(e)
  const int32_t *cu_q;
  const uint16_t *q, *k_new, *v_new, *k_cache, *v_cache;
  const int64_t *kv_start;
  const int32_t *kv_len;
  uint16_t *out;
  float *part_o;                  // [slots][rows_m][D]
  float2 *part_ml;                // [slots][rows_m]
  uint32_t *counters;             // [B * Hkv]
  uint32_t *dev_status;
  int64_t tiles_bound;            // host bound on the global tile count
  int pdl_secondary;
  // shared-prefix (bifurcated) arrangement
  int mode;                       // 0 plain; 1 decode partials only; 2 prefix partials
  int G, spb;                     // groups; sequences per prefix row-block
  const int32_t *group;           // [B] non-decreasing
  const int64_t *prefix_start;    // [G]
  const int32_t *prefix_len;      // [G]
};

// ---------------------------------------------------------------- smem layout
// Warps: 4 key slices (16 keys of each 64-key tile) x RS row groups (8*NB
// packed query rows each).  Packed row m = j*g + hg for block row j and query
// head hk*g + hg; a CTA holds up to RS*8*NB rows.
template <int D, int RS, int NB>
struct AttnSmem {
  static constexpr int kWarps = kKW * RS;
  static constexpr int kThreads = kWarps * 32;
  static constexpr int kRowsW = 8 * NB;                        // rows per warp
  static constexpr int kRows = RS * kRowsW;                    // rows per CTA
  static constexpr int kTileBytes = kTileKeys * D * 2;         // one K or V tile
  static constexpr int kStageBytes = 2 * kTileBytes;
  static constexpr int kOStride = D + 4;                       // padded merge rows (floats)
  static constexpr int kMergeO = kRows * kOStride * 4;
  static constexpr int kMergeML = kWarps * kRowsW * 8;         // (m, l) per warp row
  static constexpr int kFinal = kRows * 8;                     // merged (m, l) per row
  static constexpr int kSchedBytes = kMaxBatch * 4 + 4 * kMaxGroups * 4;  // schedule tables
  static constexpr int kOffStages = 0;
  static constexpr int kOffMergeO = kStages * kStageBytes;
  static constexpr int kOffMergeML = kOffMergeO + kMergeO;
  static constexpr int kOffFinal = kOffMergeML + kMergeML;
  static constexpr int kOffSched = kOffFinal + kFinal;
  static constexpr int kOffMisc = kOffSched + kSchedBytes;
  static constexpr int kBytes = kOffMisc + 64;
  static_assert(kMaxBatch * 8 <= kStages * kStageBytes, "sequence bases staged in tile buffers");
};

// Swizzled byte offset of (row, 16-byte chunk) inside a tile: chunk ^ (row % 8)
// makes the 8 rows read by one ldmatrix phase hit 8 different bank groups.
template <int D>
__device__ __forceinline__ uint32_t swz(int row, int chunk) {
  return static_cast<uint32_t>(row * (D * 2) + ((chunk ^ (row & 7)) << 4));
}

// ---------------------------------------------------------------- schedule
// The global tile order walks "units" (mode 0/1: sequences; mode 2: shared-
// prefix groups), each holding ns segments of nt 64-key tiles:
//   mode 0/1: segment hk = (sequence, KV head) over the sequence's cache + block;
//   mode 2:   segment (KV head, row-block) over the group's prefix rows, for
//             the packed query rows of up to spb whole sequences of the group.
struct Sched {
  int32_t *nt;          // [units] tiles per segment
  int32_t *ns;          // [groups] segments per unit (mode 2)
  int32_t *first;       // [groups] first sequence of the group (mode 2)
  int32_t *cnt;         // [groups] sequences in the group (mode 2)
  int32_t *segb;        // [groups] index of the unit's first segment (mode 2)
  int units;
  int mode, Hkv;
  __device__ __forceinline__ int nseg(int u) const { return mode == 2 ? ns[u] : Hkv; }
};

__device__ __forceinline__ Sched sched_view(unsigned char *base, int mode, int Hkv) {
  Sched S;
  S.nt = reinterpret_cast<int32_t *>(base);
  S.ns = S.nt + kMaxBatch;
  S.first = S.ns + kMaxGroups;
  S.cnt = S.first + kMaxGroups;
  S.segb = S.cnt + kMaxGroups;
  S.mode = mode;
  S.Hkv = Hkv;
  S.units = 0;
  return S;
}

// Fill the schedule tables and the per-unit tile offsets `ubase` (block-wide,
// identical in every CTA).  Returns the global tile count W, 0 if there is no
// work, -1 if the inputs are inconsistent (dev_status gets BAD_LENGTH).
template <int NT>
__device__ int64_t build_sched(const AttnParams &P, Sched &S, int64_t *ubase, int64_t *scratch) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int B = P.B;
  int bad = 0;
  for (int i = tid; i < B; i += NT) {
    const int r0 = P.cu_q[i], r1 = P.cu_q[i + 1], L = P.kv_len[i];
    const int64_t kv0 = P.kv_start[i];
    const bool ok = r0 >= 0 && r1 - r0 >= 1 && r1 - r0 <= P.max_q_rows && r1 <= P.num_rows &&
                    L >= 0 && kv0 >= 0 && kv0 + L <= P.pool_rows;
    if (P.mode != 2) S.nt[i] = ok ? (L + (r1 - r0) + kTileKeys - 1) / kTileKeys : 0;
    bad |= !ok;
    if (P.mode != 0) {          // shared-prefix groups: non-decreasing, in range
      const int gi = P.group[i];
      bad |= gi < 0 || gi >= P.G || (i > 0 && P.group[i - 1] > gi);
    }
  }
  if (P.mode == 2) {
    for (int gg = tid; gg < P.G; gg += NT) {
      int lo = 0, hi = B;                          // first i with group[i] >= gg
      while (lo < hi) { const int mid = (lo + hi) >> 1; if (P.group[mid] < gg) lo = mid + 1; else hi = mid; }
      int lo2 = lo, hi2 = B;                       // first i with group[i] > gg
      while (lo2 < hi2) { const int mid = (lo2 + hi2) >> 1; if (P.group[mid] <= gg) lo2 = mid + 1; else hi2 = mid; }
      const int n = lo2 - lo;
      const int64_t ps = P.prefix_start[gg];
      const int pl = P.prefix_len[gg];
      const bool ok = pl >= 0 && ps >= 0 && ps + pl <= P.pool_rows;
      bad |= !ok;
      S.first[gg] = lo;
      S.cnt[gg] = n;
      S.ns[gg] = P.Hkv * ((n + P.spb - 1) / P.spb);
      S.nt[gg] = ok ? (pl + kTileKeys - 1) / kTileKeys : 0;
    }
  }
  bad = __syncthreads_or(bad);
  S.units = P.mode == 2 ? P.G : B;
  if (bad) {
    if (blockIdx.x == 0 && tid == 0) set_status(P.dev_status, SV_DEV_BAD_LENGTH);
    // plain/decode mode skips only the bad sequences (zero tiles); the
    // prefix launch needs every group and sequence consistent
    if (P.mode == 2 || P.mode == 1) return -1;
  }
  if (warp == 0) {
    int64_t carry = 0, segc = 0;
    for (int base = 0; base < S.units; base += 32) {
      const int u = base + lane;
      const int64_t nsu = u < S.units ? S.nseg(u) : 0;
      const int64_t v = u < S.units ? static_cast<int64_t>(S.nt[u]) * nsu : 0;
      int64_t inc = v, sinc = nsu;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int64_t t = __shfl_up_sync(0xffffffffu, inc, o);
        const int64_t t2 = __shfl_up_sync(0xffffffffu, sinc, o);
        if (lane >= o) { inc += t; sinc += t2; }
      }
      if (u < S.units) {
        ubase[u] = carry + inc - v;
        if (P.mode == 2) S.segb[u] = static_cast<int32_t>(segc + sinc - nsu);
      }
      carry += __shfl_sync(0xffffffffu, inc, 31);
      segc += __shfl_sync(0xffffffffu, sinc, 31);
    }
    if (lane == 0) scratch[0] = carry;
  }
  __syncthreads();
  return scratch[0];
}

// Position in the global tile order.
struct Cursor {
  int u, s, lt;        // unit, segment within the unit, tile within the segment
};

// Advance one tile; returns true when a new segment starts.
__device__ __forceinline__ bool cursor_advance(Cursor &c, const Sched &S) {
  if (++c.lt < S.nt[c.u]) return false;
  c.lt = 0;
  if (++c.s < S.nseg(c.u)) return true;
  c.s = 0;
  do { ++c.u; } while (c.u < S.units && S.nt[c.u] * S.nseg(c.u) == 0);
  return true;
}

// CTA whose range [c*W/G, (c+1)*W/G) holds global tile t (requires G <= W).
__device__ __forceinline__ int64_t cta_of_tile(int64_t t, int64_t W, int64_t G) {
  return ((t + 1) * G + W - 1) / W - 1;
}

struct SeqInfo {       // one segment
  int r0;              // first Q row (and first block row in mode 0/1)
  int Ri;              // block rows (keys after the cache rows); 0 for a prefix
  int M;               // packed query rows
  int L;               // cache (or prefix) rows
  int nt;              // tiles
  int hk;              // KV head
  int seg;             // segment index (partial slots)
  int64_t kv0;         // first pool row
};

__device__ __forceinline__ SeqInfo load_seq(const AttnParams &P, const Sched &S, const Cursor &c) {
  SeqInfo s;
  s.nt = S.nt[c.u];
  if (S.mode != 2) {
    const int i = c.u;
    s.r0 = P.cu_q[i];
    s.Ri = P.cu_q[i + 1] - s.r0;
    s.M = s.Ri * P.g;
    s.L = P.kv_len[i];
    s.kv0 = P.kv_start[i];
    s.hk = c.s;
    s.seg = i * P.Hkv + c.s;
  } else {
    const int nrb = S.ns[c.u] / P.Hkv;
    s.hk = c.s / nrb;
    const int rb = c.s - s.hk * nrb;
    const int f = S.first[c.u] + rb * P.spb;
    const int n = min(P.spb, S.cnt[c.u] - rb * P.spb);
    s.r0 = P.cu_q[f];
    s.M = (P.cu_q[f + n] - s.r0) * P.g;
    s.Ri = 0;
    s.L = P.prefix_len[c.u];
    s.kv0 = P.prefix_start[c.u];
    s.seg = S.segb[c.u] + c.s;
  }
  return s;
}

// Issue the cp.async copies of one 64-key K and V tile (threads 0..127).  Keys
// below L come from the pool, the next Ri from the block rows, the rest are
// zero-filled (and masked).  A tile entirely inside the cache takes the
// strided fast path.
template <int D>
__device__ __forceinline__ void issue_tile_loads(const AttnParams &P, const SeqInfo &s, int hk,
                                                 int lt, uint32_t stage_base) {
  constexpr int CH = D / 8;                 // 16-byte chunks per row
  constexpr int RPP = 128 / CH;             // rows per pass of 128 threads
  constexpr int NPASS = kTileKeys / RPP;
  constexpr int kTile = kTileKeys * D * 2;
  const int t = threadIdx.x;
  const int ch = t % CH, rr = t / CH;
  const int key0 = lt * kTileKeys;
  if (key0 + kTileKeys <= s.L) {
    const int64_t off = ((s.kv0 + key0 + rr) * P.Hkv + hk) * D + ch * 8;
    const int64_t step = static_cast<int64_t>(RPP) * P.Hkv * D;
#pragma unroll
    for (int p = 0; p < NPASS; ++p) {
      const int row = rr + p * RPP;
      cp_async16(stage_base + swz<D>(row, ch), P.k_cache + off + p * step, 16);
      cp_async16(stage_base + kTile + swz<D>(row, ch), P.v_cache + off + p * step, 16);
    }
    return;
  }
#pragma unroll
  for (int p = 0; p < NPASS; ++p) {
    const int row = rr + p * RPP;
    const int key = key0 + row;
    int64_t off = 0;
    const uint16_t *kb = P.k_new, *vb = P.v_new;
    int bytes = 0;
    if (key < s.L) {
      off = ((s.kv0 + key) * P.Hkv + hk) * D + ch * 8;
      kb = P.k_cache;
      vb = P.v_cache;
      bytes = 16;
    } else if (key < s.L + s.Ri) {
      off = (static_cast<int64_t>(s.r0 + key - s.L) * P.Hkv + hk) * D + ch * 8;
      bytes = 16;
    }
    cp_async16(stage_base + swz<D>(row, ch), kb + off, bytes);
    cp_async16(stage_base + kTile + swz<D>(row, ch), vb + off, bytes);
  }
}

// ---------------------------------------------------------------------------
// bf16 kernel, operands swapped so keys are the MMA M dimension:
//   S^T (16 keys x 8 rows) = K (16 x D) . Q^T      per n-block of 8 rows
//   O^T (D x 8 rows)      += V^T (D x 16) . P^T   with P^T transposed in
//                                                 registers by movmatrix
// With few packed rows (MHA, K+1 <= 8) this needs half the MMAs of putting the
// rows on M, and keeps O in 32*NB registers per thread.
// ---------------------------------------------------------------------------
template <int D, int RS, int NB>
__device__ __forceinline__ void attn_bf16_body(const AttnParams &P, unsigned char *smem) {
  using SM = AttnSmem<D, RS, NB>;
  constexpr int NT = SM::kThreads;
  constexpr int KS = D / 16;          // k-steps of K.Q^T
  constexpr int DM = D / 16;          // m-tiles of V^T.P^T
  constexpr int RW = SM::kRowsW;
  constexpr int OS = SM::kOStride;
  const uint32_t sbase = smem_u32(smem);
  int64_t *ubase = reinterpret_cast<int64_t *>(smem + SM::kOffStages);  // before the pipeline
  int *misc = reinterpret_cast<int *>(smem + SM::kOffMisc);
  float *merge_o = reinterpret_cast<float *>(smem + SM::kOffMergeO);
  float2 *merge_ml = reinterpret_cast<float2 *>(smem + SM::kOffMergeML);
  float2 *fin = reinterpret_cast<float2 *>(smem + SM::kOffFinal);
  int64_t *misc64 = reinterpret_cast<int64_t *>(misc + 8);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int ks = warp % kKW, rs = warp / kKW;
  const int r = lane >> 2, q = lane & 3;
  const int g = P.g;

  Sched S = sched_view(smem + SM::kOffSched, P.mode, P.Hkv);
  const int64_t W = build_sched<NT>(P, S, ubase, misc64);
  if (W <= 0) return;
  if (W > P.tiles_bound) {
    if (blockIdx.x == 0 && tid == 0) set_status(P.dev_status, SV_DEV_BAD_LENGTH);
    return;
  }
  const int64_t G = W < static_cast<int64_t>(gridDim.x) ? W : static_cast<int64_t>(gridDim.x);
  if (blockIdx.x >= G) return;
  const int64_t t_begin = (static_cast<int64_t>(blockIdx.x) * W) / G;
  const int64_t t_end = (static_cast<int64_t>(blockIdx.x + 1) * W) / G;
  const int ntiles = static_cast<int>(t_end - t_begin);   // >= 1 since G <= W

  Cursor cur;
  {
    int lo = 0, hi = S.units - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (ubase[mid] <= t_begin) lo = mid; else hi = mid - 1;
    }
    while (S.nt[lo] * S.nseg(lo) == 0) ++lo;
    const int64_t rel = t_begin - ubase[lo];
    cur.u = lo;
    cur.s = static_cast<int>(rel / S.nt[lo]);
    cur.lt = static_cast<int>(rel - static_cast<int64_t>(cur.s) * S.nt[lo]);
  }
  int64_t seg_first_tile = t_begin - cur.lt;   // global index of the segment's tile 0
  __syncthreads();                            // ubase dead: tile buffers free

  // ---- prologue: first kStages-1 tiles in flight
  Cursor ld = cur;
  SeqInfo ld_s = load_seq(P, S, ld);
#pragma unroll
  for (int st = 0; st < kStages - 1; ++st) {
    if (st < ntiles) {
      if (tid < 128) issue_tile_loads<D>(P, ld_s, ld_s.hk, ld.lt, sbase + st * SM::kStageBytes);
      if (cursor_advance(ld, S) && st + 1 < ntiles) ld_s = load_seq(P, S, ld);
    }
    cp_async_commit();
  }

  SeqInfo cs = load_seq(P, S, cur);
  uint32_t qf[KS][NB][2];          // Q^T B-fragments of this warp's rows
  float o[DM][NB][4];              // O^T accumulators
  float m_run[NB][2], l_run[NB][2];
  const int row_w0 = rs * RW;      // first packed row of this warp
  bool active = row_w0 < cs.M;

  auto load_q = [&]() {
    const int M = cs.M;
#pragma unroll
    for (int nb = 0; nb < NB; ++nb) {
      const int m = row_w0 + nb * 8 + r;
      const bool ok = m < M;
      const int j = ok ? m / g : 0, hg = ok ? m - j * g : 0;
      const uint16_t *qrow = P.q + (static_cast<int64_t>(cs.r0 + j) * P.Hq + cs.hk * g + hg) * D;
#pragma unroll
      for (int kk = 0; kk < KS; ++kk) {
        qf[kk][nb][0] = ok ? *reinterpret_cast<const uint32_t *>(qrow + kk * 16 + 2 * q) : 0u;
        qf[kk][nb][1] = ok ? *reinterpret_cast<const uint32_t *>(qrow + kk * 16 + 8 + 2 * q) : 0u;
      }
    }
  };
  auto reset_state = [&]() {
#pragma unroll
    for (int dm = 0; dm < DM; ++dm)
#pragma unroll
      for (int nb = 0; nb < NB; ++nb) o[dm][nb][0] = o[dm][nb][1] = o[dm][nb][2] = o[dm][nb][3] = 0.0f;
#pragma unroll
    for (int nb = 0; nb < NB; ++nb) {
      m_run[nb][0] = m_run[nb][1] = -INFINITY;
      l_run[nb][0] = l_run[nb][1] = 0.0f;
    }
  };
  load_q();
  reset_state();

  for (int k = 0; k < ntiles; ++k) {
    cp_async_wait<kStages - 2>();
    __syncthreads();
    {   // refill the stage consumed at k-1
      const int kn = k + kStages - 1;
      if (kn < ntiles) {
        if (tid < 128) issue_tile_loads<D>(P, ld_s, ld_s.hk, ld.lt, sbase + (kn % kStages) * SM::kStageBytes);
        if (cursor_advance(ld, S) && kn + 1 < ntiles) ld_s = load_seq(P, S, ld);
      }
      cp_async_commit();
    }
    if (active) {
      const uint32_t kbase = sbase + (k % kStages) * SM::kStageBytes;
      const uint32_t vbase = kbase + SM::kTileBytes;
      // ---- S^T = K Q^T for this warp's 16 keys
      float sacc[NB][4];
#pragma unroll
      for (int nb = 0; nb < NB; ++nb) sacc[nb][0] = sacc[nb][1] = sacc[nb][2] = sacc[nb][3] = 0.0f;
      {
        const int krow = ks * 16 + (lane & 7) + (((lane >> 3) & 1) << 3);
#pragma unroll
        for (int kk = 0; kk < KS; ++kk) {
          uint32_t a[4];
          ldmatrix_x4(kbase + swz<D>(krow, kk * 2 + (lane >> 4)), a[0], a[1], a[2], a[3]);
#pragma unroll
          for (int nb = 0; nb < NB; ++nb) mma_bf16_16816(sacc[nb], a, qf[kk][nb][0], qf[kk][nb][1]);
        }
      }
      // ---- mask (only in tiles reaching past the cache) + online softmax
      const int key_a = cur.lt * kTileKeys + ks * 16 + r;          // key of sacc[.][0..1]
      const bool need_mask = (cur.lt + 1) * kTileKeys > cs.L;
      uint32_t pb[NB][2];
#pragma unroll
      for (int nb = 0; nb < NB; ++nb) {
        float pv[4];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          float v0 = sacc[nb][e] * P.sl2, v1 = sacc[nb][2 + e] * P.sl2;
          if (need_mask) {
            const int m = row_w0 + nb * 8 + 2 * q + e;
            const int lim = cs.L + (cs.Ri > 0 ? min(m / g, cs.Ri - 1) + 1 : 0);  // keys < lim visible
            v0 = key_a < lim ? v0 : -INFINITY;
            v1 = key_a + 8 < lim ? v1 : -INFINITY;
          }
          float mx = fmaxf(v0, v1);
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
          const float m_new = fmaxf(m_run[nb][e], mx);
          const float m_use = m_new == -INFINITY ? 0.0f : m_new;
          const float alpha = exp2f(m_run[nb][e] - m_use);
          const float p0 = exp2f(v0 - m_use), p1 = exp2f(v1 - m_use);
          l_run[nb][e] = l_run[nb][e] * alpha + (p0 + p1);
          m_run[nb][e] = m_new;
          pv[e] = p0;
          pv[2 + e] = p1;
          if (alpha != 1.0f) {
#pragma unroll
            for (int dm = 0; dm < DM; ++dm) {
              o[dm][nb][e] *= alpha;
              o[dm][nb][2 + e] *= alpha;
            }
          }
        }
        pb[nb][0] = movmatrix_trans(pack_bf16x2(pv[0], pv[1]));   // keys 0-7 of the slice
        pb[nb][1] = movmatrix_trans(pack_bf16x2(pv[2], pv[3]));   // keys 8-15
      }
      // ---- O^T += V^T P^T
      {
        const int vrow = ks * 16 + (lane & 7) + ((lane >> 4) << 3);
#pragma unroll
        for (int dm = 0; dm < DM; ++dm) {
          uint32_t a[4];
          ldmatrix_x4_trans(vbase + swz<D>(vrow, dm * 2 + ((lane >> 3) & 1)), a[0], a[1], a[2], a[3]);
#pragma unroll
          for (int nb = 0; nb < NB; ++nb) mma_bf16_16816(o[dm][nb], a, pb[nb][0], pb[nb][1]);
        }
      }
    }

    const bool seg_end = cur.lt + 1 == cs.nt;
    const bool last = k + 1 == ntiles;
    if (!(seg_end || last)) {
      ++cur.lt;
      continue;
    }
    // ================= end of a piece: merge the key-slice warps =================
    const int Mi = cs.M;
#pragma unroll
    for (int nb = 0; nb < NB; ++nb)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        float lv = l_run[nb][e];
        lv += __shfl_xor_sync(0xffffffffu, lv, 4);
        lv += __shfl_xor_sync(0xffffffffu, lv, 8);
        lv += __shfl_xor_sync(0xffffffffu, lv, 16);
        if (r == 0) merge_ml[warp * RW + nb * 8 + 2 * q + e] = make_float2(m_run[nb][e], lv);
      }
    __syncthreads();
    if (tid < SM::kRows) {            // merged (max, sum) of packed row tid
      const int rg = tid / RW, rl = tid - rg * RW;
      float mm = -INFINITY;
#pragma unroll
      for (int w2 = 0; w2 < kKW; ++w2) mm = fmaxf(mm, merge_ml[(rg * kKW + w2) * RW + rl].x);
      const float mu = mm == -INFINITY ? 0.0f : mm;
      float ll = 0.0f;
#pragma unroll
      for (int w2 = 0; w2 < kKW; ++w2) {
        const float2 v = merge_ml[(rg * kKW + w2) * RW + rl];
        ll += v.y * exp2f(v.x - mu);
      }
      fin[tid] = make_float2(mm, ll);
    }
    __syncthreads();
    // O^T of the 4 key slices into the row-major buffer, in a fixed order
    for (int step = kKW - 1; step >= 0; --step) {
      if (ks == step) {
#pragma unroll
        for (int nb = 0; nb < NB; ++nb)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int m = row_w0 + nb * 8 + 2 * q + e;
            const float mm = fin[m].x;
            const float sc = exp2f(m_run[nb][e] - (mm == -INFINITY ? 0.0f : mm));
            float *dst = merge_o + m * OS;
#pragma unroll
            for (int dm = 0; dm < DM; ++dm) {
              const int d0 = dm * 16 + r;
              const float a0 = o[dm][nb][e] * sc, a1 = o[dm][nb][2 + e] * sc;
              if (step == kKW - 1) {
                dst[d0] = a0;
                dst[d0 + 8] = a1;
              } else {
                dst[d0] += a0;
                dst[d0 + 8] += a1;
              }
            }
          }
      }
      __syncthreads();
    }
    const int seg = cs.seg;
    const int64_t c_first = cta_of_tile(seg_first_tile, W, G);
    const int64_t c_last = cta_of_tile(seg_first_tile + cs.nt - 1, W, G);
    const int npieces = static_cast<int>(c_last - c_first + 1);
    constexpr int rows_m = SM::kRows;
    if (npieces == 1 && P.mode == 0) {   // the whole segment is here: normalize, store
      for (int e = tid; e < Mi * (D / 2); e += NT) {
        const int m = e / (D / 2), d = (e - m * (D / 2)) * 2;
        const float lsum = fin[m].y;
        const float inv = lsum > 0.0f ? 1.0f / lsum : 0.0f;
        const int j = m / g, hg = m - j * g;
        *reinterpret_cast<uint32_t *>(P.out + (static_cast<int64_t>(cs.r0 + j) * P.Hq + cs.hk * g + hg) * D + d) =
            pack_bf16x2(merge_o[m * OS + d] * inv, merge_o[m * OS + d + 1] * inv);
      }
    } else {                          // partial: slot = CTA index + segment index
      const int64_t slot = static_cast<int64_t>(blockIdx.x) + seg;
      for (int e = tid; e < Mi * (D / 2); e += NT) {
        const int m = e / (D / 2), d = (e - m * (D / 2)) * 2;
        *reinterpret_cast<float2 *>(P.part_o + (slot * rows_m + m) * D + d) =
            make_float2(merge_o[m * OS + d], merge_o[m * OS + d + 1]);
      }
      if (tid < Mi) P.part_ml[slot * rows_m + tid] = fin[tid];
    }
    if (npieces > 1 && P.mode == 0) {    // plain mode: the last piece merges
      __threadfence();
      __syncthreads();
      if (tid == 0) {
        const unsigned old = atomicInc(&P.counters[seg], static_cast<unsigned>(npieces - 1));
        misc[0] = old == static_cast<unsigned>(npieces - 1) ? 1 : 0;
      }
      __syncthreads();
      if (misc[0]) {                   // last piece to arrive merges the segment
        __threadfence();
        for (int e = tid; e < Mi * (D / 2); e += NT) {
          const int m = e / (D / 2), d = (e - m * (D / 2)) * 2;
          float mm = -INFINITY;
          for (int c = 0; c < npieces; ++c)
            mm = fmaxf(mm, __ldcg(&P.part_ml[(c_first + c + seg) * rows_m + m].x));
          const float mu = mm == -INFINITY ? 0.0f : mm;
          float n0 = 0.0f, n1 = 0.0f, den = 0.0f;
          for (int c = 0; c < npieces; ++c) {
            const int64_t slot2 = c_first + c + seg;
            const float2 ml = __ldcg(&P.part_ml[slot2 * rows_m + m]);
            const float f = exp2f(ml.x - mu);
            const float2 ov = __ldcg(reinterpret_cast<const float2 *>(P.part_o + (slot2 * rows_m + m) * D + d));
            n0 += f * ov.x;
            n1 += f * ov.y;
            den += f * ml.y;
          }
          const float inv = den > 0.0f ? 1.0f / den : 0.0f;
          const int j = m / g, hg = m - j * g;
          *reinterpret_cast<uint32_t *>(P.out + (static_cast<int64_t>(cs.r0 + j) * P.Hq + cs.hk * g + hg) * D + d) =
              pack_bf16x2(n0 * inv, n1 * inv);
        }
      }
    }
    __syncthreads();                   // merge buffers reusable
    if (last) break;
    seg_first_tile += cs.nt;
    cursor_advance(cur, S);
    cs = load_seq(P, S, cur);
    active = row_w0 < cs.M;
    load_q();
    reset_state();
  }
  cp_async_wait<0>();
}

template <int D, int RS, int NB>
__global__ void __launch_bounds__(AttnSmem<D, RS, NB>::kThreads)
    attn_bf16_kernel(const AttnParams P) {
  extern __shared__ __align__(128) unsigned char smem[];
  attn_bf16_body<D, RS, NB>(P, smem);
  // A dependent launch (fused step) must not complete before its primary.
  if (P.pdl_secondary) asm volatile("griddepcontrol.wait;\n" ::: "memory");
}

// ---------------------------------------------------------------------------
// Shared-prefix merge: out(i, h, j) combines the decode partials of (i, hk)
// (cache + block keys, causal) with the prefix partials of the row-block that
// holds sequence i's rows (the group's prefill keys), as one softmax over the
// concatenated keys -- the bifurcated attention abstract's "precise" split.
// One CTA per (sequence, KV head); it rebuilds both launches' schedules to
// find the pieces (partial slots) of its two segments.
// ---------------------------------------------------------------------------
constexpr int kMergeNT = 128;

struct MergeParams {
  AttnParams P;                       // mode 1 view of the batch
  const float *dec_o; const float2 *dec_ml; int dec_rows; int dec_grid;
  const float *pre_o; const float2 *pre_ml; int pre_rows; int pre_grid;
};

template <int D>
__global__ void __launch_bounds__(kMergeNT) attn_prefix_merge_kernel(const MergeParams MP) {
  extern __shared__ __align__(16) unsigned char msm[];
  constexpr int kTables = kMaxBatch * 4 + 4 * kMaxGroups * 4;
  Sched Sd = sched_view(msm, 1, MP.P.Hkv);
  Sched Sp = sched_view(msm + kTables, 2, MP.P.Hkv);
  int64_t *ud = reinterpret_cast<int64_t *>(msm + 2 * kTables);
  int64_t *up = ud + kMaxBatch;
  int64_t *scratch = up + kMaxGroups;
  AttnParams P = MP.P;
  P.mode = 1;
  const int64_t Wd = build_sched<kMergeNT>(P, Sd, ud, scratch);
  AttnParams P2 = MP.P;
  P2.mode = 2;
  const int64_t Wp = build_sched<kMergeNT>(P2, Sp, up, scratch + 1);
  if (Wd <= 0 || Wp < 0) return;
  const int i = blockIdx.x / P.Hkv, hk = blockIdx.x - i * P.Hkv;
  if (Sd.nt[i] == 0) return;
  const int g = P.g;
  const int r0 = P.cu_q[i], Mi = (P.cu_q[i + 1] - r0) * g;
  // decode pieces
  const int64_t Gd = Wd < MP.dec_grid ? Wd : MP.dec_grid;
  const int seg_d = i * P.Hkv + hk;
  const int64_t td = ud[i] + static_cast<int64_t>(hk) * Sd.nt[i];
  const int64_t cfd = cta_of_tile(td, Wd, Gd), cld = cta_of_tile(td + Sd.nt[i] - 1, Wd, Gd);
  // prefix pieces
  const int gg = P.group[i];
  const int ntp = Wp > 0 ? Sp.nt[gg] : 0;
  int64_t cfp = 0, clp = -1;
  int seg_p = 0, rowoff = 0;
  if (ntp > 0) {
    const int nrb = Sp.ns[gg] / P.Hkv;
    const int rb = (i - Sp.first[gg]) / P.spb;
    const int s_in = hk * nrb + rb;
    seg_p = Sp.segb[gg] + s_in;
    const int64_t tp = up[gg] + static_cast<int64_t>(s_in) * ntp;
    const int64_t Gp = Wp < MP.pre_grid ? Wp : MP.pre_grid;
    cfp = cta_of_tile(tp, Wp, Gp);
    clp = cta_of_tile(tp + ntp - 1, Wp, Gp);
    rowoff = (r0 - P.cu_q[Sp.first[gg] + rb * P.spb]) * g;
  }
  for (int e = threadIdx.x; e < Mi * (D / 2); e += kMergeNT) {
    const int m = e / (D / 2), d = (e - m * (D / 2)) * 2;
    float mm = -INFINITY;
    for (int64_t c = cfd; c <= cld; ++c) mm = fmaxf(mm, __ldcg(&MP.dec_ml[(c + seg_d) * MP.dec_rows + m].x));
    for (int64_t c = cfp; c <= clp; ++c)
      mm = fmaxf(mm, __ldcg(&MP.pre_ml[(c + seg_p) * MP.pre_rows + rowoff + m].x));
    const float mu = mm == -INFINITY ? 0.0f : mm;
    float n0 = 0.0f, n1 = 0.0f, den = 0.0f;
    for (int64_t c = cfd; c <= cld; ++c) {
      const int64_t row = (c + seg_d) * MP.dec_rows + m;
      const float2 ml = __ldcg(&MP.dec_ml[row]);
      const float f = exp2f(ml.x - mu);
      const float2 ov = __ldcg(reinterpret_cast<const float2 *>(MP.dec_o + row * D + d));
      n0 += f * ov.x;
      n1 += f * ov.y;
      den += f * ml.y;
    }
    for (int64_t c = cfp; c <= clp; ++c) {
      const int64_t row = (c + seg_p) * MP.pre_rows + rowoff + m;
      const float2 ml = __ldcg(&MP.pre_ml[row]);
      const float f = exp2f(ml.x - mu);
      const float2 ov = __ldcg(reinterpret_cast<const float2 *>(MP.pre_o + row * D + d));
      n0 += f * ov.x;
      n1 += f * ov.y;
      den += f * ml.y;
    }
    const float inv = den > 0.0f ? 1.0f / den : 0.0f;
    const int j = m / g, hg = m - j * g;
    *reinterpret_cast<uint32_t *>(P.out + (static_cast<int64_t>(r0 + j) * P.Hq + hk * g + hg) * D + d) =
        pack_bf16x2(n0 * inv, n1 * inv);
  }
}

constexpr int kMergeSmem = 2 * (kMaxBatch * 4 + 4 * kMaxGroups * 4) + (kMaxBatch + kMaxGroups + 2) * 8;

// ---------------------------------------------------------------------------
// fp32 kernel (CUDA cores): one CTA per (sequence, KV head), whole segment.
// ---------------------------------------------------------------------------
constexpr int kF32NT = 256;
constexpr int kF32Keys = 32;

template <int D>
struct F32Smem {
  static constexpr int kQ = kMaxRowsM * D;          // floats
  static constexpr int kK = kF32Keys * (D + 1);
  static constexpr int kV = kF32Keys * D;
  static constexpr int kBytes = (kQ + kK + kV) * 4;
};

template <int D>
__global__ void __launch_bounds__(kF32NT) attn_f32_kernel(const AttnParams P, const float *q,
                                                          const float *k_new, const float *v_new,
                                                          const float *k_cache, const float *v_cache,
                                                          float *out) {
  constexpr int DL = D / 32;                  // output columns per lane
  extern __shared__ __align__(16) float fsm[];
  float (*Qs)[D] = reinterpret_cast<float (*)[D]>(fsm);
  float (*Ks)[D + 1] = reinterpret_cast<float (*)[D + 1]>(fsm + F32Smem<D>::kQ);
  float (*Vs)[D] = reinterpret_cast<float (*)[D]>(fsm + F32Smem<D>::kQ + F32Smem<D>::kK);
  const int seg = blockIdx.x;
  const int i = seg / P.Hkv, hk = seg - i * P.Hkv;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int r0 = P.cu_q[i], Ri = P.cu_q[i + 1] - r0, L = P.kv_len[i];
  const int64_t kv0 = P.kv_start[i];
  if (r0 < 0 || Ri < 1 || Ri > P.max_q_rows || r0 + Ri > P.num_rows || L < 0 || kv0 < 0 ||
      kv0 + L > P.pool_rows) {
    if (tid == 0) set_status(P.dev_status, SV_DEV_BAD_LENGTH);
    if (P.pdl_secondary) asm volatile("griddepcontrol.wait;\n" ::: "memory");
    return;
  }
  const int g = P.g, M = Ri * g;
  for (int e = tid; e < M * D; e += kF32NT) {
    const int m = e / D, d = e - m * D, j = m / g, hg = m - j * g;
    Qs[m][d] = q[(static_cast<int64_t>(r0 + j) * P.Hq + hk * g + hg) * D + d];
  }
  constexpr int RPW = kMaxRowsM / (kF32NT / 32);   // rows per warp
  float m_run[RPW], l_run[RPW], o[RPW][DL];
#pragma unroll
  for (int a = 0; a < RPW; ++a) {
    m_run[a] = -INFINITY;
    l_run[a] = 0.0f;
#pragma unroll
    for (int c = 0; c < DL; ++c) o[a][c] = 0.0f;
  }
  const int T = L + Ri;
  for (int k0 = 0; k0 < T; k0 += kF32Keys) {
    __syncthreads();
    for (int e = tid; e < kF32Keys * D; e += kF32NT) {
      const int rr = e / D, d = e - rr * D, key = k0 + rr;
      float kv = 0.0f, vv = 0.0f;
      if (key < L) {
        kv = k_cache[((kv0 + key) * P.Hkv + hk) * D + d];
        vv = v_cache[((kv0 + key) * P.Hkv + hk) * D + d];
      } else if (key < T) {
        kv = k_new[(static_cast<int64_t>(r0 + key - L) * P.Hkv + hk) * D + d];
        vv = v_new[(static_cast<int64_t>(r0 + key - L) * P.Hkv + hk) * D + d];
      }
      Ks[rr][d] = kv;
      Vs[rr][d] = vv;
    }
    __syncthreads();
#pragma unroll
    for (int a = 0; a < RPW; ++a) {
      const int m = warp + a * (kF32NT / 32);
      if (m >= M) continue;
      const int j = m / g;
      const int key = k0 + lane;
      float sc = 0.0f;
#pragma unroll 8
      for (int d = 0; d < D; ++d) sc = fmaf(Qs[m][d], Ks[lane][d], sc);
      const bool vis = key < L + j + 1 && key < T;
      sc = vis ? sc * P.sl2 : -INFINITY;
      const float mx = warp_max(sc);
      const float m_new = fmaxf(m_run[a], mx);
      const float m_use = m_new == -INFINITY ? 0.0f : m_new;
      const float alpha = exp2f(m_run[a] - m_use);
      const float pv = exp2f(sc - m_use);
      l_run[a] = l_run[a] * alpha + warp_sum(pv);
      m_run[a] = m_new;
#pragma unroll
      for (int c = 0; c < DL; ++c) o[a][c] *= alpha;
      for (int kk = 0; kk < kF32Keys; ++kk) {
        const float pk = __shfl_sync(0xffffffffu, pv, kk);
#pragma unroll
        for (int c = 0; c < DL; ++c) o[a][c] = fmaf(pk, Vs[kk][lane + 32 * c], o[a][c]);
      }
    }
  }
#pragma unroll
  for (int a = 0; a < RPW; ++a) {
    const int m = warp + a * (kF32NT / 32);
    if (m >= M) continue;
    const int j = m / g, hg = m - j * g;
    const float inv = l_run[a] > 0.0f ? 1.0f / l_run[a] : 0.0f;
#pragma unroll
    for (int c = 0; c < DL; ++c)
      out[(static_cast<int64_t>(r0 + j) * P.Hq + hk * g + hg) * D + lane + 32 * c] = o[a][c] * inv;
  }
  if (P.pdl_secondary) asm volatile("griddepcontrol.wait;\n" ::: "memory");
}

template <int D, int RS, int NB>
cudaError_t launch_bf16(const AttnParams &P, int grid, cudaStream_t s) {
  using SM = AttnSmem<D, RS, NB>;
  auto kern = attn_bf16_kernel<D, RS, NB>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SM::kBytes);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(SM::kThreads);
  cfg.dynamicSmemBytes = SM::kBytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = P.pdl_secondary ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, P);
}

template <int D, int RS, int NB>
int occupancy_bf16() {
  using SM = AttnSmem<D, RS, NB>;
  auto kern = attn_bf16_kernel<D, RS, NB>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SM::kBytes) != cudaSuccess)
    return 1;
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, SM::kThreads, SM::kBytes) != cudaSuccess)
    return 1;
  return n > 0 ? n : 1;
}

// Row configuration for rows_m packed rows: (RS, NB) with RS*8*NB >= rows_m.
// 0: (1,1) <= 8 rows; 1: (1,2) <= 16; 2: (2,2) <= 32; 3: (3,2) <= 48; 4: (4,2) <= 64.
int row_config(int rows_m) {
  return rows_m <= 8 ? 0 : rows_m <= 16 ? 1 : rows_m <= 32 ? 2 : rows_m <= 48 ? 3 : 4;
}
int config_rows(int rc) { static const int rows[5] = {8, 16, 32, 48, 64}; return rows[rc]; }

template <int D>
int occupancy_d(int rc) {
  switch (rc) {
    case 0: return occupancy_bf16<D, 1, 1>();
    case 1: return occupancy_bf16<D, 1, 2>();
    case 2: return occupancy_bf16<D, 2, 2>();
    case 3: return occupancy_bf16<D, 3, 2>();
    default: return occupancy_bf16<D, 4, 2>();
  }
}

int occupancy_for(int D, int rc) {
  static int cache[2][5] = {{0}};
  const int di = D == 128 ? 1 : 0;
  if (cache[di][rc] == 0) cache[di][rc] = D == 64 ? occupancy_d<64>(rc) : occupancy_d<128>(rc);
  return cache[di][rc];
}

template <int D>
cudaError_t launch_d(const AttnParams &P, int rc, int grid, cudaStream_t s) {
  switch (rc) {
    case 0: return launch_bf16<D, 1, 1>(P, grid, s);
    case 1: return launch_bf16<D, 1, 2>(P, grid, s);
    case 2: return launch_bf16<D, 2, 2>(P, grid, s);
    case 3: return launch_bf16<D, 3, 2>(P, grid, s);
    default: return launch_bf16<D, 4, 2>(P, grid, s);
  }
}

}  // namespace

constexpr int64_t kMaxGrid = 2048;   // bound on persistent attention CTAs
constexpr int kPrefixCfg = 4;        // prefix launches hold 64 packed rows per CTA

AttnPlan plan_attention(const sv_attn_args &a, int num_sms) {
  AttnPlan p;
  const int g = a.num_q_heads / a.num_kv_heads;
  p.rows_m = a.max_q_rows * g;
  p.row_cfg = row_config(p.rows_m);
  p.m_tiles = (config_rows(p.row_cfg) + 15) / 16;
  // sum over sequences of ceil((L_i + R_i) / 64), per KV head
  p.tiles_bound = static_cast<int64_t>(a.num_kv_heads) *
                  ((a.kv_rows_bound + a.num_rows) / kTileKeys + a.batch);
  p.grid = std::min<int64_t>(kMaxGrid, std::max<int64_t>(1, p.tiles_bound));
  if (a.dtype == SV_BF16 && num_sms > 0) {
    const int occ = occupancy_for(a.head_dim, p.row_cfg);
    p.grid = std::min<int64_t>(p.grid, static_cast<int64_t>(num_sms) * occ);
  }
  p.prefix = a.num_groups > 0;
  p.spb = std::max(1, config_rows(kPrefixCfg) / p.rows_m);
  p.pre_grid = p.pre_tiles_bound = p.pre_slots = 0;
  if (p.prefix) {
    const int64_t rb_max = a.batch / p.spb + 1;            // row-blocks of one group
    p.pre_tiles_bound = static_cast<int64_t>(a.num_kv_heads) * rb_max *
                        (a.prefix_rows_bound / kTileKeys + a.num_groups);
    p.pre_grid = std::min<int64_t>(kMaxGrid, std::max<int64_t>(1, p.pre_tiles_bound));
    if (num_sms > 0) {
      const int occ = occupancy_for(a.head_dim, kPrefixCfg);
      p.pre_grid = std::min<int64_t>(p.pre_grid, static_cast<int64_t>(num_sms) * occ);
    }
    p.pre_slots = p.pre_grid + static_cast<int64_t>(a.num_kv_heads) *
                                   (a.batch / p.spb + 1 + a.num_groups);
  }
  return p;
}

int attention_max_batch() { return kMaxBatch; }
int attention_max_groups() { return kMaxGroups; }
int attention_slot_rows(const AttnPlan &p) { return config_rows(p.row_cfg); }
int attention_prefix_rows() { return config_rows(kPrefixCfg); }

cudaError_t launch_attention(const sv_attn_args &a, const AttnPlan &p, const AttnWs &ws,
                             bool pdl_secondary, cudaStream_t s) {
  if (a.batch <= 0) return cudaSuccess;
  AttnParams P;
  P.B = a.batch;
  P.Hq = a.num_q_heads;
  P.Hkv = a.num_kv_heads;
  P.g = a.num_q_heads / a.num_kv_heads;
  P.max_q_rows = a.max_q_rows;
  P.num_rows = a.num_rows;
  P.pool_rows = a.pool_rows;
  const float scale = a.scale != 0.0f ? a.scale : 1.0f / sqrtf(static_cast<float>(a.head_dim));
  P.sl2 = scale * kLog2e;
  P.cu_q = a.cu_q;
  P.q = static_cast<const uint16_t *>(a.q);
  P.k_new = static_cast<const uint16_t *>(a.k_new);
  P.v_new = static_cast<const uint16_t *>(a.v_new);
  P.k_cache = static_cast<const uint16_t *>(a.k_cache);
  P.v_cache = static_cast<const uint16_t *>(a.v_cache);
  P.kv_start = a.kv_start;
  P.kv_len = a.kv_len;
  P.out = static_cast<uint16_t *>(a.out);
  P.part_o = ws.dec_o;
  P.part_ml = reinterpret_cast<float2 *>(ws.dec_ml);
  P.counters = ws.counters;
  P.dev_status = a.dev_status;
  P.tiles_bound = p.tiles_bound;
  P.pdl_secondary = pdl_secondary ? 1 : 0;
  P.mode = 0;
  P.G = a.num_groups;
  P.spb = p.spb;
  P.group = a.group;
  P.prefix_start = a.prefix_start;
  P.prefix_len = a.prefix_len;
  if (a.dtype == SV_F32) {
    const int grid = a.batch * a.num_kv_heads;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kF32NT);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl_secondary ? 1 : 0;
    const float *q = static_cast<const float *>(a.q), *kn = static_cast<const float *>(a.k_new),
                *vn = static_cast<const float *>(a.v_new), *kc = static_cast<const float *>(a.k_cache),
                *vc = static_cast<const float *>(a.v_cache);
    float *out = static_cast<float *>(a.out);
    if (a.head_dim == 64) {
      cfg.dynamicSmemBytes = F32Smem<64>::kBytes;
      cudaError_t e = cudaFuncSetAttribute(attn_f32_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           F32Smem<64>::kBytes);
      if (e != cudaSuccess) return e;
      return cudaLaunchKernelEx(&cfg, attn_f32_kernel<64>, P, q, kn, vn, kc, vc, out);
    }
    cfg.dynamicSmemBytes = F32Smem<128>::kBytes;
    cudaError_t e = cudaFuncSetAttribute(attn_f32_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         F32Smem<128>::kBytes);
    if (e != cudaSuccess) return e;
    return cudaLaunchKernelEx(&cfg, attn_f32_kernel<128>, P, q, kn, vn, kc, vc, out);
  }
  const bool d64 = a.head_dim == 64;
  if (!p.prefix) {
    const int grid = static_cast<int>(p.grid);
    return d64 ? launch_d<64>(P, p.row_cfg, grid, s) : launch_d<128>(P, p.row_cfg, grid, s);
  }
  // shared prefix: prefix row-blocks, then decode segments, then the merge
  AttnParams Pp = P;
  Pp.mode = 2;
  Pp.part_o = ws.pre_o;
  Pp.part_ml = reinterpret_cast<float2 *>(ws.pre_ml);
  Pp.tiles_bound = p.pre_tiles_bound;
  const int pgrid = static_cast<int>(p.pre_grid);
  cudaError_t e = d64 ? launch_d<64>(Pp, kPrefixCfg, pgrid, s) : launch_d<128>(Pp, kPrefixCfg, pgrid, s);
  if (e != cudaSuccess) return e;
  AttnParams Pd = P;
  Pd.mode = 1;
  Pd.pdl_secondary = 0;
  const int grid = static_cast<int>(p.grid);
  e = d64 ? launch_d<64>(Pd, p.row_cfg, grid, s) : launch_d<128>(Pd, p.row_cfg, grid, s);
  if (e != cudaSuccess) return e;
  MergeParams MP;
  MP.P = Pd;
  MP.dec_o = ws.dec_o;
  MP.dec_ml = reinterpret_cast<const float2 *>(ws.dec_ml);
  MP.dec_rows = config_rows(p.row_cfg);
  MP.dec_grid = grid;
  MP.pre_o = ws.pre_o;
  MP.pre_ml = reinterpret_cast<const float2 *>(ws.pre_ml);
  MP.pre_rows = config_rows(kPrefixCfg);
  MP.pre_grid = pgrid;
  auto mk = d64 ? attn_prefix_merge_kernel<64> : attn_prefix_merge_kernel<128>;
  e = cudaFuncSetAttribute(mk, cudaFuncAttributeMaxDynamicSharedMemorySize, kMergeSmem);
  if (e != cudaSuccess) return e;
  mk<<<a.batch * a.num_kv_heads, kMergeNT, kMergeSmem, s>>>(MP);
  return cudaGetLastError();
}

}  // namespace sv

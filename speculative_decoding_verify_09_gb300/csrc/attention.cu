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
//    (K_i + 1) x (Hq/Hkv) query rows sharing that KV head are packed as the N
//    dimension, so every KV byte is read once for all of them (GQA).
//  * Stream-K split: the global tile sequence (segments in order) is cut into
//    gridDim.x contiguous ranges of equal cost (a segment costs its tiles plus
//    kSegCost), one per persistent CTA (two CTAs per SM), regardless of
//    segment boundaries.  A CTA that covers a whole segment writes the output
//    directly; otherwise each piece writes a partial (unnormalized O, row max,
//    row sum) and the last piece to arrive (atomic count, no waiting) folds
//    every piece in CTA order (one routine at every merge site, so the bits do
//    not depend on which piece merges).
//  * Warp specialization: one producer warp walks the CTA's tile range and
//    streams every K and V tile into a ring of shared-memory stages guarded by
//    full / empty mbarriers, running ahead across segment boundaries: 16-byte
//    cp.async copies (cache rows, block rows, zero fill past the end) into
//    XOR-swizzled rows, whose completion arrives on the stage's mbarrier.  (A
//    256-byte bulk copy per row moves the same bytes at about a quarter of the
//    rate: the copy engine's cost is per request.)  It also stages each
//    segment's packed Q rows (bulk copies into 16-byte-padded rows) and a
//    segment header into one of two Q slots.
//  * Consumer warps (4 key slices x RS row groups) compute S^T = K Q^T and
//    O^T += V^T P^T with mma.sync m16n8k16 (bf16 in, or f16 built in registers
//    from E4M3 K/V codes; fp32 accumulate) and an online softmax per warp; no
//    CTA-wide barrier per tile.  At the end of a piece in the middle of a
//    CTA's range the key-slice states are merged in shared memory and a
//    merger warp counts the piece and, if last, folds the pieces; the CTA's
//    final piece is closed by the consumers, with the slices in the (then
//    idle) stages and one folding pass.
//  * Every wait is bounded: a wait that runs out sets SV_DEV_TIMEOUT and the
//    CTA drains its copies in flight and leaves.
//
// fp32 inputs use a CUDA-core kernel (one CTA per segment, fp32 FMA).
#include <algorithm>

#include "common.cuh"
#include "kernels.h"

namespace sv {

namespace {

constexpr int kTileKeys = 64;
constexpr int kKW = 4;            // consumer warps splitting the keys of one tile
constexpr int kMaxBatch = 1024;   // sequences per call
constexpr int kMaxGroups = 256;   // shared-prefix groups per call
constexpr int kMaxStages = 8;
// The split weighs each segment as its tiles plus kSegCost tiles: starting and
// finishing a segment (Q load, epilogue, partial, merge) costs about that much
// time, so CTAs that cross more segments get fewer tiles and all end together.
constexpr int kSegCost = 3;
constexpr uint32_t kSpinLimit = 1u << 22;   // polls of one mbarrier before giving up
constexpr float kLog2e = 1.4426950408889634f;

// Byte offsets of the dynamic shared memory (same on host and device).
struct SmemMap {
  int ns;                  // ring stages
  int units_cap, groups_cap, b_cap;
  int q;                   // two Q slots (header + packed rows)
  int merge_o, merge_ml, fin, jobs, bars, sched, misc, total;
};

// A stream-K merge handed from the consumer warps to the merger warp: the
// piece's partial is in global memory; the merger counts the pieces of the
// segment and, for the last one, combines them into the output.
constexpr int kJobs = 4;
struct MergeJob {
  int seg;              // segment (-1: no more jobs)
  int npieces, Mi, r0, hk;
  int64_t c_first;      // first piece's CTA index
};

struct AttnParams {
  int B, Hq, Hkv, g, max_q_rows;
  int64_t num_rows, pool_rows;
  float sl2;                      // scale * log2(e) (times k_scale for E4M3 K)
  float v_scale;                  // E4M3 V: output scale (1 otherwise)
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
  int pdl_primary;                // let the next launch start at once
  uint32_t spin_limit;            // polls of one mbarrier wait before it gives up
  // shared-prefix (bifurcated) arrangement
  int mode;                       // 0 plain; 1 decode partials only; 2 prefix partials
  int G, spb;                     // groups; sequences per prefix row-block
  const int32_t *group;           // [B] non-decreasing
  const int64_t *prefix_start;    // [G]
  const int32_t *prefix_len;      // [G]
  SmemMap sm;
};

// Bytes of the schedule tables (see Sched): int64 kst, int32 klen, cuq, nt, and
// four int32 group tables.
__host__ __device__ constexpr int sched_bytes(int units_cap, int groups_cap, int b_cap) {
  return 8 * units_cap + 4 * units_cap + 4 * b_cap + 4 * units_cap + 16 * groups_cap;
}

// ---------------------------------------------------------------- smem layout
// Warps: 4 key slices (16 keys of each 64-key tile) x RS row groups (8*NB
// packed query rows each), then the producer warp.  Packed row m = j*g + hg
// for block row j and query head hk*g + hg; a CTA holds up to RS*8*NB rows.
template <int D, int RS, int NB, bool KV8>
struct AttnCfg {
  static constexpr int kKVB = KV8 ? 1 : 2;                      // bytes per K/V element
  static constexpr int kCW = kKW * RS;                          // consumer warps
  static constexpr int kThreads = (kCW + 2) * 32;               // + producer + merger
  static constexpr int kRowsW = 8 * NB;                         // rows per warp
  static constexpr int kRows = RS * kRowsW;                     // rows per CTA
  static constexpr int kRowB = D * 2 + 16;                      // padded Q row
  static constexpr int kTileB = kTileKeys * D * kKVB;           // one K or V tile (swizzled)
  static constexpr int kStageB = 2 * kTileB;
  static constexpr int kQHead = 64;                             // segment header
  static constexpr int kQSlotB = kQHead + kRows * kRowB;
  static constexpr int kOStride = D + 4;                        // padded merge rows (floats)
  static constexpr int kMergeO = 2 * kRows * kOStride * 4;      // two key-slice sums
  static constexpr int kMergeML = kCW * kRowsW * 8;
  static constexpr int kFinal = kRows * 8;
  // The final piece's merge keeps every key slice's O rows in the (then idle)
  // K/V stages: needs kKW row blocks within the smallest ring (2 stages).
  static constexpr bool kFinalFits = kKW * kRows * kOStride * 4 <= 2 * kStageB;
  static_assert(kMaxBatch * 16 <= 2 * kStageB, "unit tile and cost bases staged in the ring");

  static SmemMap map(int ns, int units_cap, int groups_cap, int b_cap) {
    auto up = [](int x, int a) { return (x + a - 1) / a * a; };
    SmemMap m;
    m.ns = ns;
    m.units_cap = up(std::max(units_cap, 1), 4);
    m.groups_cap = up(std::max(groups_cap, 1), 4);
    m.b_cap = up(b_cap + 1, 4);
    int off = ns * kStageB;
    m.q = off;
    off += 2 * kQSlotB;
    m.merge_o = off;
    off += kMergeO;
    m.merge_ml = off;
    off += kMergeML;
    m.fin = off;
    off += kFinal;
    m.jobs = up(off, 16);
    off = m.jobs + kJobs * static_cast<int>(sizeof(MergeJob)) + kRows * 8;   // + merger's row stats
    m.bars = up(off, 8);
    off = m.bars + (2 * ns + 5 + 2 * kJobs) * 8;
    m.sched = up(off, 16);
    off = m.sched + sched_bytes(m.units_cap, m.groups_cap, m.b_cap);
    m.misc = up(off, 16);
    m.total = m.misc + 64;
    return m;
  }
};

// ---------------------------------------------------------------- mbarriers
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_arrive_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(bar), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_test(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ uint32_t lds_u32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.b32 %0, [%1];\n" : "=r"(v) : "r"(addr));
  return v;
}
__device__ __forceinline__ void lds_u64(uint32_t addr, uint32_t &a, uint32_t &b) {
  asm volatile("ld.shared.v2.b32 {%0, %1}, [%2];\n" : "=r"(a), "=r"(b) : "r"(addr));
}

// Output column of O^T accumulator row r (hi = 0) or r + 8 (hi = 1) of m-tile
// dm.  With E4M3 V the A operand is built by transposing 8x8 blocks of V rows
// read four codes at a time, which puts column 16 dm + 4 (r / 2) + r % 2 (+ 2
// for the second block) on row r.
template <bool KV8>
__device__ __forceinline__ int o_col(int dm, int r, int hi) {
  return KV8 ? dm * 16 + 4 * (r >> 1) + (r & 1) + 2 * hi : dm * 16 + r + 8 * hi;
}

// Fold one piece of a split segment -- its (max, row sum) v and four O columns
// ov, relative to that max -- into a running combination (mm, den, acc).  Every
// merge site folds the pieces in CTA order with this one routine, so the bits
// do not depend on which piece happens to merge.
__device__ __forceinline__ void fold_piece(float &mm, float &den, float4 &acc, float2 v,
                                           float4 ov) {
  const float mn = fmaxf(mm, v.x);
  const float mu = mn == -INFINITY ? 0.0f : mn;
  const float fa = fast_exp2(mm - mu), fb = fast_exp2(v.x - mu);
  den = den * fa + v.y * fb;
  acc.x = acc.x * fa + ov.x * fb;
  acc.y = acc.y * fa + ov.y * fb;
  acc.z = acc.z * fa + ov.z * fb;
  acc.w = acc.w * fa + ov.w * fb;
  mm = mn;
}

// Wait for the phase of parity `parity` to complete; false after `limit`
// polls (the launch's wait limit: kSpinLimit unless the host set a smaller one).
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, uint32_t limit) {
  for (uint32_t it = 0; it < limit; ++it)
    if (mbar_test(bar, parity)) return true;
  return false;
}

// One global -> shared bulk copy completing on `bar` (16-byte aligned, bytes % 16 == 0).
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n"
      ::"r"(dst), "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}
__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;\n" : "=l"(p));
  return p;
}

// 16-byte cp.async with an L2 cache-policy hint; src_bytes = 0 zero-fills.
__device__ __forceinline__ void cp_async16_hint(uint32_t dst, const void *src, int src_bytes,
                                                uint64_t policy) {
  asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2, %3;\n" ::"r"(dst),
               "l"(src), "r"(src_bytes), "l"(policy)
               : "memory");
}
// Arrive on `bar` once every cp.async this thread issued so far has landed
// (the barrier's count includes this arrival).
__device__ __forceinline__ void cp_async_arrive(uint32_t bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];\n" ::"r"(bar) : "memory");
}

// Padded Q row address inside a Q slot.
template <int D>
__device__ __forceinline__ uint32_t prow(int row, int chunk) {
  return static_cast<uint32_t>(row * (D * 2 + 16) + (chunk << 4));
}
// Swizzled byte offset of (row, 16-byte chunk) inside a K or V tile: chunk ^
// (row % 8) makes the 8 rows read by one ldmatrix phase hit 8 bank groups.
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
  int64_t *kst;         // [units] first pool row: kv_start (mode 0/1) or prefix_start (mode 2)
  int32_t *klen;        // [units] kv_len (mode 0/1) or prefix_len (mode 2)
  int32_t *cuq;         // [B+1] cu_q
  int32_t *nt;          // [units] tiles per segment
  int32_t *ns;          // [groups] segments per unit (mode 2)
  int32_t *first;       // [groups] first sequence of the group (mode 2)
  int32_t *cnt;         // [groups] sequences in the group (mode 2)
  int32_t *segb;        // [groups] index of the unit's first segment (mode 2)
  int units;
  int mode, Hkv;
  __device__ __forceinline__ int nseg(int u) const { return mode == 2 ? ns[u] : Hkv; }
};

__device__ __forceinline__ Sched sched_view(unsigned char *base, int mode, int Hkv, int units_cap,
                                            int groups_cap, int b_cap) {
  Sched S;
  S.kst = reinterpret_cast<int64_t *>(base);
  S.klen = reinterpret_cast<int32_t *>(S.kst + units_cap);
  S.cuq = S.klen + units_cap;
  S.nt = S.cuq + b_cap;
  S.ns = S.nt + units_cap;
  S.first = S.ns + groups_cap;
  S.cnt = S.first + groups_cap;
  S.segb = S.cnt + groups_cap;
  S.mode = mode;
  S.Hkv = Hkv;
  S.units = 0;
  return S;
}

// Fill the schedule tables, the per-unit tile offsets `ubase` and cost offsets
// `cbase` (a segment costs its tiles + kSegCost; block-wide, identical in every
// CTA).  Returns the global tile count W (scratch[0]; the total cost in
// scratch[1]), 0 if there is no work, -1 if the inputs are inconsistent
// (dev_status gets BAD_LENGTH).
template <int NT>
__device__ int64_t build_sched(const AttnParams &P, Sched &S, int64_t *ubase, int64_t *cbase,
                               int64_t *scratch) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int B = P.B;
  int bad = 0;
  for (int i = tid; i < B; i += NT) {
    const int r0 = P.cu_q[i], r1 = P.cu_q[i + 1], L = P.kv_len[i];
    const int64_t kv0 = P.kv_start[i];
    const bool ok = r0 >= 0 && r1 - r0 >= 1 && r1 - r0 <= P.max_q_rows && r1 <= P.num_rows &&
                    L >= 0 && kv0 >= 0 && kv0 + L <= P.pool_rows;
    S.cuq[i] = r0;
    if (i == B - 1) S.cuq[B] = r1;
    if (P.mode != 2) {
      S.nt[i] = ok ? (L + (r1 - r0) + kTileKeys - 1) / kTileKeys : 0;
      S.klen[i] = L;
      S.kst[i] = kv0;
    }
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
      S.klen[gg] = pl;
      S.kst[gg] = ps;
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
    int64_t carry = 0, segc = 0, costc = 0;
    for (int base = 0; base < S.units; base += 32) {
      const int u = base + lane;
      const int64_t nsu = u < S.units ? S.nseg(u) : 0;
      const int64_t ntu = u < S.units ? S.nt[u] : 0;
      const int64_t v = ntu * nsu;
      const int64_t cv = ntu > 0 ? (ntu + kSegCost) * nsu : 0;
      int64_t inc = v, sinc = nsu, cinc = cv;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int64_t t = __shfl_up_sync(0xffffffffu, inc, o);
        const int64_t t2 = __shfl_up_sync(0xffffffffu, sinc, o);
        const int64_t t3 = __shfl_up_sync(0xffffffffu, cinc, o);
        if (lane >= o) { inc += t; sinc += t2; cinc += t3; }
      }
      if (u < S.units) {
        ubase[u] = carry + inc - v;
        cbase[u] = costc + cinc - cv;
        if (P.mode == 2) S.segb[u] = static_cast<int32_t>(segc + sinc - nsu);
      }
      carry += __shfl_sync(0xffffffffu, inc, 31);
      segc += __shfl_sync(0xffffffffu, sinc, 31);
      costc += __shfl_sync(0xffffffffu, cinc, 31);
    }
    if (lane == 0) {
      scratch[0] = carry;
      scratch[1] = costc;
    }
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

// CTA whose range [c*W/G, (c+1)*W/G) holds position t (requires G <= W).
__device__ __forceinline__ int64_t cta_of_tile(int64_t t, int64_t W, int64_t G) {
  return ((t + 1) * G + W - 1) / W - 1;
}

// Global tile at cost position x (0 <= x <= Wc): the first tile of the segment
// while x is inside the segment's kSegCost lead-in, then one tile per cost unit.
__device__ __forceinline__ int64_t tile_of_cost(int64_t x, const Sched &S, const int64_t *ubase,
                                                const int64_t *cbase, int64_t Wc, int64_t W) {
  if (x >= Wc) return W;
  int lo = 0, hi = S.units - 1;          // largest unit with cbase <= x (it has tiles)
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (cbase[mid] <= x) lo = mid; else hi = mid - 1;
  }
  const int64_t nt = S.nt[lo], per = nt + kSegCost;
  const int64_t rel = x - cbase[lo], sg = rel / per, within = rel - sg * per;
  return ubase[lo] + sg * nt + (within > kSegCost ? within - kSegCost : 0);
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
    s.r0 = S.cuq[i];
    s.Ri = S.cuq[i + 1] - s.r0;
    s.M = s.Ri * P.g;
    s.L = S.klen[i];
    s.kv0 = S.kst[i];
    s.hk = c.s;
    s.seg = i * P.Hkv + c.s;
  } else {
    const int nrb = S.ns[c.u] / P.Hkv;
    s.hk = c.s / nrb;
    const int rb = c.s - s.hk * nrb;
    const int f = S.first[c.u] + rb * P.spb;
    const int n = min(P.spb, S.cnt[c.u] - rb * P.spb);
    s.r0 = S.cuq[f];
    s.M = (S.cuq[f + n] - s.r0) * P.g;
    s.Ri = 0;
    s.L = S.klen[c.u];
    s.kv0 = S.kst[c.u];
    s.seg = S.segb[c.u] + c.s;
  }
  return s;
}


// ---------------------------------------------------------------------------
// bf16 kernel, operands swapped so keys are the MMA M dimension:
//   S^T (16 keys x 8 rows) = K (16 x D) . Q^T      per n-block of 8 rows
//   O^T (D x 8 rows)      += V^T (D x 16) . P^T   with P^T transposed in
//                                                 registers by movmatrix
// With few packed rows (MHA, K+1 <= 8) this needs half the MMAs of putting the
// rows on M, and keeps O in 32*NB registers per thread.
// ---------------------------------------------------------------------------
struct Ring {            // shared-memory addresses of the pipeline
  uint32_t base, q, full, empty, qfull, qempty, ebar, jfull, jempty;
};

// Producer warp: Q slots and K/V stages for the CTA's tiles [0, ntiles).
template <int D, int RS, int NB, bool KV8>
__device__ __forceinline__ void attn_produce(const AttnParams &P, const Sched &S, Cursor ld,
                                             int ntiles, const Ring &rg, unsigned char *smem,
                                             volatile int *abort_flag) {
  using C = AttnCfg<D, RS, NB, KV8>;
  const int lane = threadIdx.x & 31;
  const int NS = P.sm.ns;
  const uint64_t pol = policy_evict_first();
  SeqInfo s = load_seq(P, S, ld);
  int st = 0;
  uint32_t ph = 0;
  int issued = 0, nq = 0;
  bool ok = true;
  for (int k = 0; k < ntiles; ++k) {
    if (*abort_flag) { ok = false; break; }
    if (k == 0 || ld.lt == 0) {              // a segment starts: its header and Q rows
      const int slot = nq & 1;
      if (!mbar_wait(rg.qempty + 8 * slot, ((nq >> 1) & 1) ^ 1, P.spin_limit)) { ok = false; break; }
      const uint32_t qs = rg.q + slot * C::kQSlotB;
      if (lane == 0) {
        *reinterpret_cast<SeqInfo *>(smem + (qs - rg.base)) = s;
        mbar_arrive_tx(rg.qfull + 8 * slot, static_cast<uint32_t>(s.M * D * 2));
      }
      __syncwarp();
      for (int m = lane; m < s.M; m += 32) {
        const int j = m / P.g, hg = m - j * P.g;
        bulk_g2s(qs + C::kQHead + prow<D>(m, 0),
                 P.q + (static_cast<int64_t>(s.r0 + j) * P.Hq + s.hk * P.g + hg) * D, D * 2,
                 rg.qfull + 8 * slot);
      }
      ++nq;
    }
    if (!mbar_wait(rg.empty + 8 * st, ph ^ 1, P.spin_limit)) { ok = false; break; }
    if constexpr (KV8) {
      // E4M3 rows of D bytes: lane owns 16-byte chunk lane % 8 of rows lane / 8
      // + 4 * p; chunk c of row r lands at chunk c ^ (r % 8) (bank spread for
      // the consumers' 4-byte reads)
      constexpr int CH = D / 16, RPP = 32 / CH, NPASS = kTileKeys / RPP;
      const int ch = lane % CH, rr = lane / CH;
      const uint32_t kdst = rg.base + st * C::kStageB, vdst = kdst + C::kTileB;
      const int key0 = ld.lt * kTileKeys;
      const uint8_t *kc = reinterpret_cast<const uint8_t *>(P.k_cache);
      const uint8_t *vc = reinterpret_cast<const uint8_t *>(P.v_cache);
      const uint8_t *kn = reinterpret_cast<const uint8_t *>(P.k_new);
      const uint8_t *vn = reinterpret_cast<const uint8_t *>(P.v_new);
      if (key0 + kTileKeys <= s.L) {            // whole tile inside the cache
        const int64_t off = ((s.kv0 + key0 + rr) * P.Hkv + s.hk) * D + ch * 16;
        const int64_t step = static_cast<int64_t>(RPP) * P.Hkv * D;
#pragma unroll
        for (int p = 0; p < NPASS; ++p) {
          const int row = rr + p * RPP;
          const uint32_t o = static_cast<uint32_t>(row * D + ((ch ^ (row & 7)) << 4));
          cp_async16_hint(kdst + o, kc + off + p * step, 16, pol);
          cp_async16_hint(vdst + o, vc + off + p * step, 16, pol);
        }
      } else
#pragma unroll 4
      for (int p = 0; p < NPASS; ++p) {
        const int row = rr + p * RPP, key = key0 + row;
        const uint32_t o = static_cast<uint32_t>(row * D + ((ch ^ (row & 7)) << 4));
        if (key < s.L) {                        // cache row (read once: evict first)
          const int64_t off = ((s.kv0 + key) * P.Hkv + s.hk) * D + ch * 16;
          cp_async16_hint(kdst + o, kc + off, 16, pol);
          cp_async16_hint(vdst + o, vc + off, 16, pol);
        } else {                                // block row, or zeros past the segment
          const bool blk = key < s.L + s.Ri;
          const int64_t off =
              blk ? (static_cast<int64_t>(s.r0 + key - s.L) * P.Hkv + s.hk) * D + ch * 16 : 0;
          cp_async16(kdst + o, kn + off, blk ? 16 : 0);
          cp_async16(vdst + o, vn + off, blk ? 16 : 0);
        }
      }
      cp_async_arrive(rg.full + 8 * st);
    } else {
      // K and V rows of the tile: lane owns chunk lane % CH of rows lane / CH + RPP * p
      constexpr int CH = D / 8;                 // 16-byte chunks per row
      constexpr int RPP = 32 / CH;              // rows per pass of the warp
      constexpr int NPASS = kTileKeys / RPP;
      const int ch = lane % CH, rr = lane / CH;
      const uint32_t kdst = rg.base + st * C::kStageB, vdst = kdst + C::kTileB;
      const int key0 = ld.lt * kTileKeys;
      if (key0 + kTileKeys <= s.L) {            // whole tile inside the cache
        const int64_t off = ((s.kv0 + key0 + rr) * P.Hkv + s.hk) * D + ch * 8;
        const int64_t step = static_cast<int64_t>(RPP) * P.Hkv * D;
#pragma unroll 8
        for (int p = 0; p < NPASS; ++p) {
          const int row = rr + p * RPP;
          cp_async16_hint(kdst + swz<D>(row, ch), P.k_cache + off + p * step, 16, pol);
          cp_async16_hint(vdst + swz<D>(row, ch), P.v_cache + off + p * step, 16, pol);
        }
      } else {
#pragma unroll 4
        for (int p = 0; p < NPASS; ++p) {
          const int row = rr + p * RPP, key = key0 + row;
          const uint16_t *kb = P.k_new, *vb = P.v_new;
          int64_t off = 0;
          int bytes = 0;
          if (key < s.L) {
            off = ((s.kv0 + key) * P.Hkv + s.hk) * D + ch * 8;
            kb = P.k_cache;
            vb = P.v_cache;
            bytes = 16;
          } else if (key < s.L + s.Ri) {
            off = (static_cast<int64_t>(s.r0 + key - s.L) * P.Hkv + s.hk) * D + ch * 8;
            bytes = 16;
          }
          cp_async16(kdst + swz<D>(row, ch), kb + off, bytes);
          cp_async16(vdst + swz<D>(row, ch), vb + off, bytes);
        }
      }
      cp_async_arrive(rg.full + 8 * st);
    }
    ++issued;
    if (++st == NS) { st = 0; ph ^= 1; }
    if (cursor_advance(ld, S) && k + 1 < ntiles) s = load_seq(P, S, ld);
  }
  if (!ok && lane == 0) {
    set_status(P.dev_status, SV_DEV_TIMEOUT);
    *abort_flag = 1;
  }
  {
    // Before leaving, every copy this warp started must have landed, whatever
    // the launch's wait limit: each lane's own cp.async copies (waited for
    // unconditionally), then the last fill of each stage and Q slot under the
    // full kSpinLimit (all earlier fills completed before the slot could be
    // refilled; the Q rows are bulk copies that complete on their mbarrier).
    asm volatile("cp.async.wait_all;\n" ::: "memory");
    for (int s2 = 0; s2 < NS && s2 < issued; ++s2) {
      const int last = s2 + (issued - 1 - s2) / NS * NS;
      mbar_wait(rg.full + 8 * s2, (last / NS) & 1, kSpinLimit);
    }
    for (int s2 = 0; s2 < 2 && s2 < nq; ++s2) {
      const int last = s2 + (nq - 1 - s2) / 2 * 2;
      mbar_wait(rg.qfull + 8 * s2, (last >> 1) & 1, kSpinLimit);
    }
  }
}

// Merger warp: for every multi-piece segment the consumers finished, count
// the piece (release of the partial at gpu scope, then an atomic increment
// that wraps to zero); the last piece to arrive combines all pieces' partials
// into the output.  Off the consumers' path, so their next segment proceeds.
template <int D, int RS, int NB, bool KV8>
__device__ __forceinline__ void attn_merge_jobs(const AttnParams &P, const Ring &rg,
                                                MergeJob *jobs, float2 *mfin,
                                                volatile int *abort_flag) {
  using C = AttnCfg<D, RS, NB, KV8>;
  constexpr int rows_m = C::kRows;
  const int lane = threadIdx.x & 31, g = P.g;
  for (int nj = 0;; ++nj) {
    const int js = nj % kJobs;
    if (!mbar_wait(rg.jfull + 8 * js, (nj / kJobs) & 1, P.spin_limit)) {
      if (lane == 0) {
        set_status(P.dev_status, SV_DEV_TIMEOUT);
        *abort_flag = 1;
      }
      return;
    }
    const MergeJob jb = jobs[js];
    if (jb.seg < 0) return;
    int last = 0;
    if (lane == 0) {
      __threadfence();              // the consumers' partial writes, visible at gpu scope
      const unsigned old = atomicInc(&P.counters[jb.seg], static_cast<unsigned>(jb.npieces - 1));
      last = old == static_cast<unsigned>(jb.npieces - 1);
    }
    last = __shfl_sync(0xffffffffu, last, 0);
    if (last) {
      __threadfence();
#pragma unroll 2
      for (int e = lane; e < jb.Mi * (D / 4); e += 32) {
        const int m = e / (D / 4), d = (e - m * (D / 4)) * 4;
        float mm = -INFINITY, den = 0.0f;
        float4 acc = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
#pragma unroll 4
        for (int c = 0; c < jb.npieces; ++c) {
          const int64_t slot2 = jb.c_first + c + jb.seg;
          fold_piece(mm, den, acc, __ldcg(&P.part_ml[slot2 * rows_m + m]),
                     __ldcg(reinterpret_cast<const float4 *>(P.part_o + (slot2 * rows_m + m) * D + d)));
        }
        const float inv = den > 0.0f ? 1.0f / den : 0.0f;
        const int j = m / g, hg = m - j * g;
        uint2 pk;
        pk.x = pack_bf16x2(acc.x * inv, acc.y * inv);
        pk.y = pack_bf16x2(acc.z * inv, acc.w * inv);
        *reinterpret_cast<uint2 *>(P.out + (static_cast<int64_t>(jb.r0 + j) * P.Hq + jb.hk * g + hg) * D + d) = pk;
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(rg.jempty + 8 * js);
  }
}

template <int D, int RS, int NB, bool KV8>
__device__ __forceinline__ void attn_bf16_body(const AttnParams &P, unsigned char *smem) {
  using C = AttnCfg<D, RS, NB, KV8>;
  constexpr int KS = D / 16;          // k-steps of K.Q^T
  constexpr int DM = D / 16;          // m-tiles of V^T.P^T
  constexpr int RW = C::kRowsW;
  constexpr int OS = C::kOStride;
  constexpr int NC = C::kCW * 32;     // consumer threads
  const SmemMap &Mp = P.sm;
  const int NS = Mp.ns;
  Ring rg;
  rg.base = smem_u32(smem);
  rg.q = rg.base + Mp.q;
  rg.full = rg.base + Mp.bars;
  rg.empty = rg.full + 8 * NS;
  rg.qfull = rg.empty + 8 * NS;
  rg.qempty = rg.qfull + 16;
  rg.ebar = rg.qempty + 16;
  rg.jfull = rg.ebar + 8;
  rg.jempty = rg.jfull + 8 * kJobs;
  MergeJob *jobs = reinterpret_cast<MergeJob *>(smem + Mp.jobs);
  float2 *mfin = reinterpret_cast<float2 *>(smem + Mp.jobs + kJobs * sizeof(MergeJob));
  int64_t *ubase = reinterpret_cast<int64_t *>(smem);     // staged in the ring before it starts
  int64_t *cbase = ubase + Mp.units_cap;
  int *misc = reinterpret_cast<int *>(smem + Mp.misc);
  int64_t *misc64 = reinterpret_cast<int64_t *>(smem + Mp.misc + 16);
  volatile int *abort_flag = misc + 1;
  float *merge_o = reinterpret_cast<float *>(smem + Mp.merge_o);
  float2 *merge_ml = reinterpret_cast<float2 *>(smem + Mp.merge_ml);
  float2 *fin = reinterpret_cast<float2 *>(smem + Mp.fin);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  Sched S = sched_view(smem + Mp.sched, P.mode, P.Hkv, Mp.units_cap, Mp.groups_cap, Mp.b_cap);
  const int64_t W = build_sched<C::kThreads>(P, S, ubase, cbase, misc64);
  if (W <= 0) return;
  if (W > P.tiles_bound) {
    if (blockIdx.x == 0 && tid == 0) set_status(P.dev_status, SV_DEV_BAD_LENGTH);
    return;
  }
  const int64_t Wc = misc64[1];                 // total cost
  const int64_t G = W < static_cast<int64_t>(gridDim.x) ? W : static_cast<int64_t>(gridDim.x);
  if (blockIdx.x >= G) return;
  // equal cost per CTA (tiles + kSegCost per segment started), contiguous in tile order
  const int64_t t_begin = tile_of_cost((static_cast<int64_t>(blockIdx.x) * Wc) / G, S, ubase, cbase, Wc, W);
  const int64_t t_end = tile_of_cost((static_cast<int64_t>(blockIdx.x + 1) * Wc) / G, S, ubase, cbase, Wc, W);
  const int ntiles = static_cast<int>(t_end - t_begin);
  if (ntiles <= 0) return;                      // a range inside a segment's lead-in

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
  // cost position of the current segment's start (its lead-in, then its tiles)
  int64_t seg_cost = cbase[cur.u] + static_cast<int64_t>(cur.s) * (S.nt[cur.u] + kSegCost);
  if (tid == 0) {
    for (int s2 = 0; s2 < NS; ++s2) {
      mbar_init(rg.full + 8 * s2, 32);          // one cp.async arrival per producer lane
      mbar_init(rg.empty + 8 * s2, C::kCW);
    }
    for (int s2 = 0; s2 < 2; ++s2) {
      mbar_init(rg.qfull + 8 * s2, 1);
      mbar_init(rg.qempty + 8 * s2, C::kCW);
    }
    mbar_init(rg.ebar, NC);
    for (int s2 = 0; s2 < kJobs; ++s2) {
      mbar_init(rg.jfull + 8 * s2, NC);         // every consumer thread, after its partial writes
      mbar_init(rg.jempty + 8 * s2, 1);         // the merger, done with the job
    }
    misc[1] = 0;
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
  }
  // the ring held ubase (generic writes): order them before the async copies
  asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
  __syncthreads();

  if (warp == C::kCW) {
    attn_produce<D, RS, NB, KV8>(P, S, cur, ntiles, rg, smem, abort_flag);
    return;
  }
  if (warp == C::kCW + 1) {
    attn_merge_jobs<D, RS, NB, KV8>(P, rg, jobs, mfin, abort_flag);
    return;
  }

  // ================================ consumers ================================
  const int ks = warp % kKW, rs = warp / kKW;
  const int r = lane >> 2, q = lane & 3;
  const int g = P.g;
  const int row_w0 = rs * RW;      // first packed row of this warp
  uint32_t ephase = 0;
  bool ok = true;
  // consumer-group barrier (bounded)
  auto csync = [&]() {
    mbar_arrive(rg.ebar);
    if (!mbar_wait(rg.ebar, ephase, P.spin_limit)) ok = false;
    ephase ^= 1;
  };

  float o[DM][NB][4];              // O^T accumulators
  float m_run[NB][2], l_run[NB][2];
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

  int nq = 0, st = 0;
  uint32_t ph = 0;
  SeqInfo cs;
  uint32_t qslot = 0;
  bool active = false;
  // E4M3 K with one 8-row group: the segment's Q fragments (f16, in the
  // permuted k order of the K operand) are converted once and kept
  constexpr bool kHoldQ = KV8 && NB == 1;
  uint32_t qf[kHoldQ ? KS : 1][2];
  auto begin_segment = [&]() -> bool {
    const int slot = nq & 1;
    if (!mbar_wait(rg.qfull + 8 * slot, (nq >> 1) & 1, P.spin_limit)) return false;
    qslot = rg.q + slot * C::kQSlotB;
    cs = *reinterpret_cast<const SeqInfo *>(smem + (qslot - rg.base));
    active = row_w0 < cs.M;
    reset_state();
    if constexpr (kHoldQ) {
      const uint32_t qrow = qslot + C::kQHead + prow<D>(row_w0 + r, 0) + q * 8;
#pragma unroll
      for (int kk = 0; kk < KS; ++kk) {
        uint32_t q0, q1;
        lds_u64(qrow + kk * 32, q0, q1);
        qf[kk][0] = bf16x2_to_f16x2(q0);
        qf[kk][1] = bf16x2_to_f16x2(q1);
      }
    }
    return true;
  };
  int njob = 0;
  // Hand a merge job to the merger warp (every consumer thread calls this after
  // its partial writes; seg = -1 ends the merger).
  auto post_job = [&](const MergeJob &jb) {
    const int js = njob % kJobs;
    if (!mbar_wait(rg.jempty + 8 * js, ((njob / kJobs) & 1) ^ 1, P.spin_limit)) ok = false;
    if (tid == 0) jobs[js] = jb;
    mbar_arrive(rg.jfull + 8 * js);
    ++njob;
  };
  auto end_segment = [&]() {     // Q slot no longer read by this warp
    __syncwarp();
    if (lane == 0) mbar_arrive(rg.qempty + 8 * (nq & 1));
    ++nq;
  };
  // Thread 0, a split segment's piece with its partial written: counts the
  // piece (release at gpu scope, then an increment that wraps to zero); 1 if
  // it is the last piece to arrive, which then merges every piece.
  auto settle_final = [&](int npieces, int seg) -> int {
    __threadfence();
    const unsigned old = atomicInc(&P.counters[seg], static_cast<unsigned>(npieces - 1));
    return old == static_cast<unsigned>(npieces - 1) ? 1 : 0;
  };
  // The CTA's final piece in plain mode, after its last tile (configurations
  // whose kKW x kRows O rows fit in two stages).  Once every consumer warp is
  // past its last tile (warps trail each other by up to NS tiles), every warp's
  // key-slice state (unnormalized O rows, running max, row sum) goes to the
  // idle K/V stages and one pass folds the slices: the output of a whole
  // segment, else this piece's partial, after which the last piece of the
  // segment to arrive folds every piece in CTA order.
  auto final_piece = [&]() {
    constexpr int R = C::kRows;
    float *fo = reinterpret_cast<float *>(smem);
    const int Mi = cs.M, seg = cs.seg;
    const int64_t c_first = cta_of_tile(seg_cost + kSegCost, Wc, G);
    const int64_t c_last = cta_of_tile(seg_cost + kSegCost + cs.nt - 1, Wc, G);
    const int npieces = static_cast<int>(c_last - c_first + 1);
    csync();                          // every warp is past its last tile: the stages are free
#pragma unroll
    for (int nb = 0; nb < NB; ++nb)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        float lv = l_run[nb][e];
        lv += __shfl_xor_sync(0xffffffffu, lv, 4);
        lv += __shfl_xor_sync(0xffffffffu, lv, 8);
        lv += __shfl_xor_sync(0xffffffffu, lv, 16);
        const int m = row_w0 + nb * 8 + 2 * q + e;
        if (r == 0) merge_ml[ks * R + m] = make_float2(m_run[nb][e], lv);
        float *dst = fo + (ks * R + m) * OS;
#pragma unroll
        for (int dm = 0; dm < DM; ++dm) {
          dst[o_col<KV8>(dm, r, 0)] = o[dm][nb][e] * P.v_scale;
          dst[o_col<KV8>(dm, r, 1)] = o[dm][nb][2 + e] * P.v_scale;
        }
      }
    csync();
    const int64_t own = static_cast<int64_t>(blockIdx.x) + seg;   // this piece's partial slot
    for (int e = tid; e < Mi * (D / 4); e += NC) {
      const int m = e / (D / 4), d = (e - m * (D / 4)) * 4;
      float mm = -INFINITY;
#pragma unroll
      for (int w2 = 0; w2 < kKW; ++w2) mm = fmaxf(mm, merge_ml[w2 * R + m].x);
      const float mu = mm == -INFINITY ? 0.0f : mm;
      float den = 0.0f;
      float4 acc = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
#pragma unroll
      for (int w2 = 0; w2 < kKW; ++w2) {
        const float2 ml = merge_ml[w2 * R + m];
        const float f = fast_exp2(ml.x - mu);
        const float4 v = *reinterpret_cast<const float4 *>(fo + (w2 * R + m) * OS + d);
        den = fmaf(ml.y, f, den);
        acc.x = fmaf(f, v.x, acc.x);
        acc.y = fmaf(f, v.y, acc.y);
        acc.z = fmaf(f, v.z, acc.z);
        acc.w = fmaf(f, v.w, acc.w);
      }
      if (npieces > 1) {
        __stcg(reinterpret_cast<float4 *>(P.part_o + (own * R + m) * D + d), acc);
        if (d == 0) __stcg(&P.part_ml[own * R + m], make_float2(mm, den));
        continue;
      }
      const float inv = den > 0.0f ? 1.0f / den : 0.0f;
      const int j = m / g, hg = m - j * g;
      uint2 pk;
      pk.x = pack_bf16x2(acc.x * inv, acc.y * inv);
      pk.y = pack_bf16x2(acc.z * inv, acc.w * inv);
      *reinterpret_cast<uint2 *>(P.out + (static_cast<int64_t>(cs.r0 + j) * P.Hq + cs.hk * g + hg) * D + d) = pk;
    }
    if (npieces == 1) return;
    csync();                          // every thread's partial writes
    if (tid == 0) misc[0] = settle_final(npieces, seg);
    csync();
    if (!misc[0]) return;
    __threadfence();                  // the other pieces' partials, after their publication
    for (int e = tid; e < Mi * (D / 4); e += NC) {
      const int m = e / (D / 4), d = (e - m * (D / 4)) * 4;
      float mm = -INFINITY, den = 0.0f;
      float4 acc = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
#pragma unroll 4
      for (int64_t c = c_first; c <= c_last; ++c) {
        const int64_t slot = c + seg;
        fold_piece(mm, den, acc, __ldcg(&P.part_ml[slot * R + m]),
                   __ldcg(reinterpret_cast<const float4 *>(P.part_o + (slot * R + m) * D + d)));
      }
      const float inv = den > 0.0f ? 1.0f / den : 0.0f;
      const int j = m / g, hg = m - j * g;
      uint2 pk;
      pk.x = pack_bf16x2(acc.x * inv, acc.y * inv);
      pk.y = pack_bf16x2(acc.z * inv, acc.w * inv);
      *reinterpret_cast<uint2 *>(P.out + (static_cast<int64_t>(cs.r0 + j) * P.Hq + cs.hk * g + hg) * D + d) = pk;
    }
  };

  ok = begin_segment();

  for (int k = 0; k < ntiles && ok; ++k) {
    if (!mbar_wait(rg.full + 8 * st, ph, P.spin_limit)) { ok = false; break; }
    if (active) {
      const uint32_t kbase = rg.base + st * C::kStageB;
      const uint32_t vbase = kbase + C::kTileB;
      const uint32_t qrows = qslot + C::kQHead;
      // ---- S^T = K Q^T for this warp's 16 keys
      float sacc[NB][4];
#pragma unroll
      for (int nb = 0; nb < NB; ++nb) sacc[nb][0] = sacc[nb][1] = sacc[nb][2] = sacc[nb][3] = 0.0f;
      if constexpr (KV8) {
        // E4M3 K: lane (r, q) reads codes 16 kk + 4q .. +3 of keys r and r + 8
        // of its slice; the head dimension is permuted inside each k-step (the
        // A operand's column pairs 2q, 2q+8 hold d 4q, 4q+2) and Q's B operand
        // is read with the same permutation, so the dot products are unchanged
        const int kr0 = ks * 16 + r, kr1 = kr0 + 8;
#pragma unroll
        for (int kk = 0; kk < KS; ++kk) {
          const uint32_t w0 = lds_u32(kbase + kr0 * D + ((kk ^ (kr0 & 7)) << 4) + 4 * q);
          const uint32_t w1 = lds_u32(kbase + kr1 * D + ((kk ^ (kr1 & 7)) << 4) + 4 * q);
          uint32_t a[4];
          a[0] = e4m3x2_to_f16x2(w0);
          a[1] = e4m3x2_to_f16x2(w1);
          a[2] = e4m3x2_to_f16x2(w0 >> 16);
          a[3] = e4m3x2_to_f16x2(w1 >> 16);
          if constexpr (kHoldQ) {
            mma_f16_16816(sacc[0], a, qf[kk][0], qf[kk][1]);
          } else {
#pragma unroll
            for (int nb = 0; nb < NB; ++nb) {
              uint32_t q0, q1;
              lds_u64(qrows + prow<D>(row_w0 + nb * 8 + r, 0) + kk * 32 + q * 8, q0, q1);
              mma_f16_16816(sacc[nb], a, bf16x2_to_f16x2(q0), bf16x2_to_f16x2(q1));
            }
          }
        }
      } else {
        const int krow = ks * 16 + (lane & 7) + (((lane >> 3) & 1) << 3);
#pragma unroll
        for (int kk = 0; kk < KS; kk += 2) {
          uint32_t qb[NB][4];
#pragma unroll
          for (int nb = 0; nb < NB; ++nb)
            ldmatrix_x4(qrows + prow<D>(row_w0 + nb * 8 + (lane & 7), (kk + (lane >> 4)) * 2 + ((lane >> 3) & 1)),
                        qb[nb][0], qb[nb][1], qb[nb][2], qb[nb][3]);
#pragma unroll
          for (int k2 = 0; k2 < 2; ++k2) {
            uint32_t a[4];
            ldmatrix_x4(kbase + swz<D>(krow, (kk + k2) * 2 + (lane >> 4)), a[0], a[1], a[2], a[3]);
#pragma unroll
            for (int nb = 0; nb < NB; ++nb) mma_bf16_16816(sacc[nb], a, qb[nb][2 * k2], qb[nb][2 * k2 + 1]);
          }
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
          const float alpha = fast_exp2(m_run[nb][e] - m_use);
          const float p0 = fast_exp2(v0 - m_use), p1 = fast_exp2(v1 - m_use);
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
        if constexpr (KV8) {
          pb[nb][0] = movmatrix_trans(pack_f16x2(pv[0], pv[1]));
          pb[nb][1] = movmatrix_trans(pack_f16x2(pv[2], pv[3]));
        } else {
          pb[nb][0] = movmatrix_trans(pack_bf16x2(pv[0], pv[1]));   // keys 0-7 of the slice
          pb[nb][1] = movmatrix_trans(pack_bf16x2(pv[2], pv[3]));   // keys 8-15
        }
      }
      // ---- O^T += V^T P^T
      if constexpr (KV8) {
        // E4M3 V: lane (r, q) reads codes 16 dm + 4q .. +3 of keys r and r + 8;
        // each f16 pair is one lane's share of an 8x8 (key, d) block whose
        // transpose is the A operand's (d, key) fragment (rows: see o_col)
        const int vr0 = ks * 16 + r, vr1 = vr0 + 8;
#pragma unroll
        for (int dm = 0; dm < DM; ++dm) {
          const uint32_t w0 = lds_u32(vbase + vr0 * D + ((dm ^ (vr0 & 7)) << 4) + 4 * q);
          const uint32_t w1 = lds_u32(vbase + vr1 * D + ((dm ^ (vr1 & 7)) << 4) + 4 * q);
          uint32_t a[4];
          a[0] = movmatrix_trans(e4m3x2_to_f16x2(w0));
          a[1] = movmatrix_trans(e4m3x2_to_f16x2(w0 >> 16));
          a[2] = movmatrix_trans(e4m3x2_to_f16x2(w1));
          a[3] = movmatrix_trans(e4m3x2_to_f16x2(w1 >> 16));
#pragma unroll
          for (int nb = 0; nb < NB; ++nb) mma_f16_16816(o[dm][nb], a, pb[nb][0], pb[nb][1]);
        }
      } else {
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
    __syncwarp();
    if (lane == 0) mbar_arrive(rg.empty + 8 * st);    // stage free for the producer
    if (++st == NS) { st = 0; ph ^= 1; }

    const bool seg_end = cur.lt + 1 == cs.nt;
    const bool last = k + 1 == ntiles;
    if (!(seg_end || last)) {
      ++cur.lt;
      continue;
    }
    end_segment();
    if constexpr (C::kFinalFits) {
      if (last && P.mode == 0) {
        final_piece();
        break;
      }
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
    csync();
    if (tid < C::kRows) {             // merged (max, sum) of packed row tid
      const int rg2 = tid / RW, rl = tid - rg2 * RW;
      float mm = -INFINITY;
#pragma unroll
      for (int w2 = 0; w2 < kKW; ++w2) mm = fmaxf(mm, merge_ml[(rg2 * kKW + w2) * RW + rl].x);
      const float mu = mm == -INFINITY ? 0.0f : mm;
      float ll = 0.0f;
#pragma unroll
      for (int w2 = 0; w2 < kKW; ++w2) {
        const float2 v = merge_ml[(rg2 * kKW + w2) * RW + rl];
        ll += v.y * fast_exp2(v.x - mu);
      }
      fin[tid] = make_float2(mm, ll);
    }
    csync();
    // O^T of the 4 key slices in two steps: slices 1 and 3 store into buffers
    // A and B, then slices 0 and 2 add theirs (fixed order: deterministic);
    // the row-major result is A + B.
    static_assert(kKW == 4, "two-step merge of four key slices");
    for (int step = 0; step < 2; ++step) {
      if ((ks & 1) == (step == 0 ? 1 : 0)) {
#pragma unroll
        for (int nb = 0; nb < NB; ++nb)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int m = row_w0 + nb * 8 + 2 * q + e;
            const float mm = fin[m].x;
            const float sc = fast_exp2(m_run[nb][e] - (mm == -INFINITY ? 0.0f : mm)) * P.v_scale;
            float *dst = merge_o + (ks >> 1) * C::kRows * OS + m * OS;
#pragma unroll
            for (int dm = 0; dm < DM; ++dm) {
              const int d0 = o_col<KV8>(dm, r, 0), d1 = o_col<KV8>(dm, r, 1);
              const float a0 = o[dm][nb][e] * sc, a1 = o[dm][nb][2 + e] * sc;
              if (step == 0) {
                dst[d0] = a0;
                dst[d1] = a1;
              } else {
                dst[d0] += a0;
                dst[d1] += a1;
              }
            }
          }
      }
      csync();
    }
    const float *mob = merge_o + C::kRows * OS;   // buffer B; merge_o is A
    const int seg = cs.seg;
    const int64_t c_first = cta_of_tile(seg_cost + kSegCost, Wc, G);
    const int64_t c_last = cta_of_tile(seg_cost + kSegCost + cs.nt - 1, Wc, G);
    const int npieces = static_cast<int>(c_last - c_first + 1);
    constexpr int rows_m = C::kRows;
    if (npieces == 1 && P.mode == 0) {   // the whole segment is here: normalize, store
      for (int e = tid; e < Mi * (D / 4); e += NC) {
        const int m = e / (D / 4), d = (e - m * (D / 4)) * 4;
        const float lsum = fin[m].y;
        const float inv = lsum > 0.0f ? 1.0f / lsum : 0.0f;
        const float4 a = *reinterpret_cast<const float4 *>(merge_o + m * OS + d);
        const float4 b = *reinterpret_cast<const float4 *>(mob + m * OS + d);
        const int j = m / g, hg = m - j * g;
        uint2 pk;
        pk.x = pack_bf16x2((a.x + b.x) * inv, (a.y + b.y) * inv);
        pk.y = pack_bf16x2((a.z + b.z) * inv, (a.w + b.w) * inv);
        *reinterpret_cast<uint2 *>(P.out + (static_cast<int64_t>(cs.r0 + j) * P.Hq + cs.hk * g + hg) * D + d) = pk;
      }
    } else {                          // partial: slot = CTA index + segment index
      const int64_t slot = static_cast<int64_t>(blockIdx.x) + seg;
      for (int e = tid; e < Mi * (D / 4); e += NC) {
        const int m = e / (D / 4), d = (e - m * (D / 4)) * 4;
        const float4 a = *reinterpret_cast<const float4 *>(merge_o + m * OS + d);
        const float4 b = *reinterpret_cast<const float4 *>(mob + m * OS + d);
        __stcg(reinterpret_cast<float4 *>(P.part_o + (slot * rows_m + m) * D + d),
               make_float4(a.x + b.x, a.y + b.y, a.z + b.z, a.w + b.w));
      }
      if (tid < Mi) __stcg(&P.part_ml[slot * rows_m + tid], fin[tid]);
      if (npieces > 1 && P.mode == 0 && !last) {
        // plain mode, mid-range: the merger warp counts the piece; the last merges
        post_job(MergeJob{seg, npieces, Mi, cs.r0, cs.hk, c_first});
      } else if (npieces > 1 && P.mode == 0) {
        // the CTA's final piece: the consumer warps (idle from here on) count
        // it and, if it is the last to arrive, merge with all their threads and
        // every piece's loads in flight together
        csync();
        if (tid == 0) misc[0] = settle_final(npieces, seg);
        csync();
        if (misc[0]) {
          __threadfence();
          for (int e = tid; e < Mi * (D / 4); e += NC) {
            const int m = e / (D / 4), d = (e - m * (D / 4)) * 4;
            float mm = -INFINITY, den = 0.0f;
            float4 acc = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
#pragma unroll 4
            for (int c = 0; c < npieces; ++c) {
              const int64_t slot2 = c_first + c + seg;
              fold_piece(mm, den, acc, __ldcg(&P.part_ml[slot2 * rows_m + m]),
                         __ldcg(reinterpret_cast<const float4 *>(P.part_o + (slot2 * rows_m + m) * D + d)));
            }
            const float inv = den > 0.0f ? 1.0f / den : 0.0f;
            const int j = m / g, hg = m - j * g;
            uint2 pk;
            pk.x = pack_bf16x2(acc.x * inv, acc.y * inv);
            pk.y = pack_bf16x2(acc.z * inv, acc.w * inv);
            *reinterpret_cast<uint2 *>(P.out + (static_cast<int64_t>(cs.r0 + j) * P.Hq + cs.hk * g + hg) * D + d) = pk;
          }
        }
      }
    }
    csync();                           // merge buffers reusable
    if (last || !ok) break;
    seg_cost += cs.nt + kSegCost;
    cursor_advance(cur, S);
    if (!begin_segment()) { ok = false; break; }
  }
  if (!ok && lane == 0) {
    set_status(P.dev_status, SV_DEV_TIMEOUT);
    *abort_flag = 1;
  }
  post_job(MergeJob{-1, 0, 0, 0, 0, 0});
}

template <int D, int RS, int NB, bool KV8>
__global__ void __launch_bounds__(AttnCfg<D, RS, NB, KV8>::kThreads)
    attn_bf16_kernel(const AttnParams P) {
  extern __shared__ __align__(128) unsigned char smem[];
  if (P.pdl_primary) asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
  attn_bf16_body<D, RS, NB, KV8>(P, smem);
}

// The same kernel under a 128-register cap (launch bounds of two 256-thread
// CTAs per SM; it is launched with fewer threads): used for the 16-row
// configuration (bf16 and E4M3 K/V), whose uncapped two CTAs per SM would take
// every register of the SM and leave none for the sampler CTAs the fused step
// runs beside them.
template <int D, int RS, int NB, bool KV8>
__global__ void __launch_bounds__(256, 2) attn_bf16_kernel_cap128(const AttnParams P) {
  extern __shared__ __align__(128) unsigned char smem[];
  if (P.pdl_primary) asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
  attn_bf16_body<D, RS, NB, KV8>(P, smem);
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
  constexpr int kTables = sched_bytes(kMaxBatch, kMaxGroups, kMaxBatch + 4);
  if (MP.P.pdl_primary) asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
  Sched Sd = sched_view(msm, 1, MP.P.Hkv, kMaxBatch, kMaxGroups, kMaxBatch + 4);
  Sched Sp = sched_view(msm + kTables, 2, MP.P.Hkv, kMaxBatch, kMaxGroups, kMaxBatch + 4);
  int64_t *ud = reinterpret_cast<int64_t *>(msm + 2 * kTables);
  int64_t *up = ud + kMaxBatch;
  int64_t *cd = up + kMaxGroups;
  int64_t *cp = cd + kMaxBatch;
  int64_t *scratch = cp + kMaxGroups;
  AttnParams P = MP.P;
  P.mode = 1;
  const int64_t Wd = build_sched<kMergeNT>(P, Sd, ud, cd, scratch);
  AttnParams P2 = MP.P;
  P2.mode = 2;
  const int64_t Wp = build_sched<kMergeNT>(P2, Sp, up, cp, scratch + 2);
  const int64_t Wcd = scratch[1], Wcp = scratch[3];
  if (Wd <= 0 || Wp < 0) return;
  const int i = blockIdx.x / P.Hkv, hk = blockIdx.x - i * P.Hkv;
  if (Sd.nt[i] == 0) return;
  const int g = P.g;
  const int r0 = P.cu_q[i], Mi = (P.cu_q[i + 1] - r0) * g;
  // decode pieces
  const int64_t Gd = Wd < MP.dec_grid ? Wd : MP.dec_grid;
  const int seg_d = i * P.Hkv + hk;
  const int64_t td = cd[i] + static_cast<int64_t>(hk) * (Sd.nt[i] + kSegCost) + kSegCost;
  const int64_t cfd = cta_of_tile(td, Wcd, Gd), cld = cta_of_tile(td + Sd.nt[i] - 1, Wcd, Gd);
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
    const int64_t tp = cp[gg] + static_cast<int64_t>(s_in) * (ntp + kSegCost) + kSegCost;
    const int64_t Gp = Wp < MP.pre_grid ? Wp : MP.pre_grid;
    cfp = cta_of_tile(tp, Wcp, Gp);
    clp = cta_of_tile(tp + ntp - 1, Wcp, Gp);
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

constexpr int kMergeSmem = 2 * sched_bytes(kMaxBatch, kMaxGroups, kMaxBatch + 4) +
                           (2 * kMaxBatch + 2 * kMaxGroups + 4) * 8;

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
  if (P.pdl_primary) asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
  const int seg = blockIdx.x;
  const int i = seg / P.Hkv, hk = seg - i * P.Hkv;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int r0 = P.cu_q[i], Ri = P.cu_q[i + 1] - r0, L = P.kv_len[i];
  const int64_t kv0 = P.kv_start[i];
  if (r0 < 0 || Ri < 1 || Ri > P.max_q_rows || r0 + Ri > P.num_rows || L < 0 || kv0 < 0 ||
      kv0 + L > P.pool_rows) {
    if (tid == 0) set_status(P.dev_status, SV_DEV_BAD_LENGTH);
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
}


template <int D, int RS, int NB, bool KV8>
SmemMap smem_map_for(const AttnParams &P, int ns) {
  using C = AttnCfg<D, RS, NB, KV8>;
  return P.mode == 2 ? C::map(ns, P.G, P.G, P.B) : C::map(ns, P.B, 1, P.B);
}

// Ring stages for a launch: as many as fit in smem_cap (2..kMaxStages).
template <int D, int RS, int NB, bool KV8>
int stages_for(const AttnParams &P, int smem_cap) {
  int ns = kMaxStages;
  while (ns > 2 && smem_map_for<D, RS, NB, KV8>(P, ns).total > smem_cap) --ns;
  return ns;
}

template <int D, int RS, int NB, bool KV8>
cudaError_t launch_bf16(AttnParams P, const AttnLaunchOpts &o, int max_grid, int *grid_used,
                        cudaStream_t s) {
  using C = AttnCfg<D, RS, NB, KV8>;
  AttnLaunchOpts opt = o;
  // a budget that leaves room for another kernel's CTA must still hold 2 stages
  if (opt.smem_min > 0 && smem_map_for<D, RS, NB, KV8>(P, 2).total > opt.smem_cap) {
    opt.smem_cap = kSmemMax;
    opt.smem_min = 0;
  }
  P.sm = smem_map_for<D, RS, NB, KV8>(P, stages_for<D, RS, NB, KV8>(P, opt.smem_cap));
  const int bytes = std::max(P.sm.total, opt.smem_min);
  static_assert(C::kThreads <= 256 || !(RS == 1 && NB == 2), "the capped kernel's bounds");
  auto kern = [] {
    if constexpr (D == 128 && RS == 1 && NB == 2)
      return attn_bf16_kernel_cap128<D, RS, NB, KV8>;
    else
      return attn_bf16_kernel<D, RS, NB, KV8>;
  }();
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemMax);
  if (e != cudaSuccess) return e;
  // all of the SM's unified L1 as shared memory (the loads bypass L1): an SM
  // running this kernel then still has room for another kernel's CTA
  e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                           cudaSharedmemCarveoutMaxShared);
  if (e != cudaSuccess) return e;
  int occ = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, C::kThreads, bytes);
  if (e != cudaSuccess) return e;
  const int grid = std::max(1, std::min(max_grid, std::max(occ, 1) * o.num_sms));
  *grid_used = grid;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(C::kThreads);
  cfg.dynamicSmemBytes = bytes;
  cfg.stream = s;
  return cudaLaunchKernelEx(&cfg, kern, P);
}

// Row configuration for rows_m packed rows: (RS, NB) with RS*8*NB >= rows_m.
// 0: (1,1) <= 8 rows; 1: (1,2) <= 16; 2: (2,2) <= 32; 3: (3,2) <= 48; 4: (4,2) <= 64.
int row_config(int rows_m) {
  return rows_m <= 8 ? 0 : rows_m <= 16 ? 1 : rows_m <= 32 ? 2 : rows_m <= 48 ? 3 : 4;
}
int config_rows(int rc) { static const int rows[5] = {8, 16, 32, 48, 64}; return rows[rc]; }

template <int D>
cudaError_t launch_d(const AttnParams &P, const AttnLaunchOpts &o, int rc, int max_grid, int *grid,
                     cudaStream_t s) {
  switch (rc) {
    case 0: return launch_bf16<D, 1, 1, false>(P, o, max_grid, grid, s);
    case 1: return launch_bf16<D, 1, 2, false>(P, o, max_grid, grid, s);
    case 2: return launch_bf16<D, 2, 2, false>(P, o, max_grid, grid, s);
    case 3: return launch_bf16<D, 3, 2, false>(P, o, max_grid, grid, s);
    default: return launch_bf16<D, 4, 2, false>(P, o, max_grid, grid, s);
  }
}

// E4M3 K/V: D = 128 and one row group (up to 16 packed rows).
cudaError_t launch_e4m3(const AttnParams &P, const AttnLaunchOpts &o, int rc, int max_grid,
                        int *grid, cudaStream_t s) {
  return rc == 0 ? launch_bf16<128, 1, 1, true>(P, o, max_grid, grid, s)
                 : launch_bf16<128, 1, 2, true>(P, o, max_grid, grid, s);
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
  // persistent CTAs: the launch takes min(grid, SMs x resident CTAs per SM)
  p.grid = std::min<int64_t>(kMaxGrid, std::max<int64_t>(1, p.tiles_bound));
  (void)num_sms;
  p.prefix = a.num_groups > 0;
  p.spb = std::max(1, config_rows(kPrefixCfg) / p.rows_m);
  p.pre_grid = p.pre_tiles_bound = p.pre_slots = 0;
  if (p.prefix) {
    const int64_t rb_max = a.batch / p.spb + 1;            // row-blocks of one group
    p.pre_tiles_bound = static_cast<int64_t>(a.num_kv_heads) * rb_max *
                        (a.prefix_rows_bound / kTileKeys + a.num_groups);
    p.pre_grid = std::min<int64_t>(kMaxGrid, std::max<int64_t>(1, p.pre_tiles_bound));
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
                             const AttnLaunchOpts &opts, cudaStream_t s) {
  if (a.batch <= 0) return cudaSuccess;
  AttnParams P{};
  P.B = a.batch;
  P.Hq = a.num_q_heads;
  P.Hkv = a.num_kv_heads;
  P.g = a.num_q_heads / a.num_kv_heads;
  P.max_q_rows = a.max_q_rows;
  P.num_rows = a.num_rows;
  P.pool_rows = a.pool_rows;
  const float scale = a.scale != 0.0f ? a.scale : 1.0f / sqrtf(static_cast<float>(a.head_dim));
  P.sl2 = scale * kLog2e;
  P.v_scale = 1.0f;
  const bool kv8 = a.kv_dtype == SV_E4M3;
  if (kv8) {                      // code * k_scale in the scores, code * v_scale in the output
    P.sl2 *= a.k_scale != 0.0f ? a.k_scale : 1.0f;
    P.v_scale = a.v_scale != 0.0f ? a.v_scale : 1.0f;
  }
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
  P.pdl_primary = 0;
  P.spin_limit = attention_wait_limit();
  if (P.spin_limit == 0 || P.spin_limit > kSpinLimit) P.spin_limit = kSpinLimit;
  P.mode = 0;
  P.G = a.num_groups;
  P.spb = p.spb;
  P.group = a.group;
  P.prefix_start = a.prefix_start;
  P.prefix_len = a.prefix_len;
  if (a.dtype == SV_F32) {
    P.pdl_primary = opts.pdl_primary ? 1 : 0;
    const int grid = a.batch * a.num_kv_heads;
    const float *q = static_cast<const float *>(a.q), *kn = static_cast<const float *>(a.k_new),
                *vn = static_cast<const float *>(a.v_new), *kc = static_cast<const float *>(a.k_cache),
                *vc = static_cast<const float *>(a.v_cache);
    float *out = static_cast<float *>(a.out);
    if (a.head_dim == 64) {
      cudaError_t e = cudaFuncSetAttribute(attn_f32_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           F32Smem<64>::kBytes);
      if (e != cudaSuccess) return e;
      attn_f32_kernel<64><<<grid, kF32NT, F32Smem<64>::kBytes, s>>>(P, q, kn, vn, kc, vc, out);
      return cudaGetLastError();
    }
    cudaError_t e = cudaFuncSetAttribute(attn_f32_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         F32Smem<128>::kBytes);
    if (e != cudaSuccess) return e;
    attn_f32_kernel<128><<<grid, kF32NT, F32Smem<128>::kBytes, s>>>(P, q, kn, vn, kc, vc, out);
    return cudaGetLastError();
  }
  const bool d64 = a.head_dim == 64;
  int grid = 0, pgrid = 0;
  if (kv8) {                      // head_dim 128, one row group, no prefix (checked on the host)
    P.pdl_primary = opts.pdl_primary ? 1 : 0;
    return launch_e4m3(P, opts, p.row_cfg, static_cast<int>(p.grid), &grid, s);
  }
  if (!p.prefix) {
    P.pdl_primary = opts.pdl_primary ? 1 : 0;
    const int mg = static_cast<int>(p.grid);
    return d64 ? launch_d<64>(P, opts, p.row_cfg, mg, &grid, s)
               : launch_d<128>(P, opts, p.row_cfg, mg, &grid, s);
  }
  // shared prefix: prefix row-blocks, then decode segments, then the merge
  // (only the merge lets a following launch start early)
  AttnLaunchOpts wide = opts;
  wide.smem_min = 0;
  AttnParams Pp = P;
  Pp.mode = 2;
  Pp.part_o = ws.pre_o;
  Pp.part_ml = reinterpret_cast<float2 *>(ws.pre_ml);
  Pp.tiles_bound = p.pre_tiles_bound;
  const int mpg = static_cast<int>(p.pre_grid);
  cudaError_t e = d64 ? launch_d<64>(Pp, wide, kPrefixCfg, mpg, &pgrid, s)
                      : launch_d<128>(Pp, wide, kPrefixCfg, mpg, &pgrid, s);
  if (e != cudaSuccess) return e;
  AttnParams Pd = P;
  Pd.mode = 1;
  const int mg = static_cast<int>(p.grid);
  e = d64 ? launch_d<64>(Pd, wide, p.row_cfg, mg, &grid, s) : launch_d<128>(Pd, wide, p.row_cfg, mg, &grid, s);
  if (e != cudaSuccess) return e;
  MergeParams MP;
  MP.P = Pd;
  MP.P.pdl_primary = opts.pdl_primary ? 1 : 0;
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

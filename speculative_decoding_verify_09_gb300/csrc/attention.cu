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
};

// ---------------------------------------------------------------- smem layout
template <int D, int MT>
struct AttnSmem {
  static constexpr int kTileBytes = kTileKeys * D * 2;          // one K or V tile
  static constexpr int kStageBytes = 2 * kTileBytes;
  static constexpr int kMergeO = MT * 16 * D * 4;                // fp32 merge buffer
  static constexpr int kMergeML = MT * kKW * 16 * 8;             // (m, l) per warp row
  static constexpr int kSchedBytes = kMaxBatch * 4;              // tiles per sequence
  static constexpr int kOffStages = 0;
  static constexpr int kOffMergeO = kStages * kStageBytes;
  static constexpr int kOffMergeML = kOffMergeO + kMergeO;
  static constexpr int kOffSched = kOffMergeML + kMergeML;
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

// Position in the global tile order: sequence i, KV head hk, tile lt of the
// (i, hk) segment.
struct Cursor {
  int i, hk, lt;
};

// Advance one tile; returns true when a new sequence starts.
__device__ __forceinline__ bool cursor_advance(Cursor &c, const int32_t *seq_nt, int Hkv, int B) {
  if (++c.lt < seq_nt[c.i]) return false;
  c.lt = 0;
  if (++c.hk < Hkv) return false;
  c.hk = 0;
  do { ++c.i; } while (c.i < B && seq_nt[c.i] == 0);
  return true;
}

// CTA whose range [c*W/G, (c+1)*W/G) holds global tile t (requires G <= W).
__device__ __forceinline__ int64_t cta_of_tile(int64_t t, int64_t W, int64_t G) {
  return ((t + 1) * G + W - 1) / W - 1;
}

struct SeqInfo {
  int r0, Ri, L, nt;   // first block row, block rows, cache rows, tiles
  int64_t kv0;         // first pool row
};

__device__ __forceinline__ SeqInfo load_seq(const AttnParams &P, const int32_t *seq_nt, int i) {
  SeqInfo s;
  s.r0 = P.cu_q[i];
  s.Ri = P.cu_q[i + 1] - s.r0;
  s.L = P.kv_len[i];
  s.kv0 = P.kv_start[i];
  s.nt = seq_nt[i];
  return s;
}

template <int D>
__device__ __forceinline__ void issue_tile_loads(const AttnParams &P, const SeqInfo &s, int hk,
                                                 int lt, uint32_t stage_base, int nthreads) {
  constexpr int CH = D / 8;                        // 16-byte chunks per row
  const int key0 = lt * kTileKeys;
  for (int idx = threadIdx.x; idx < 2 * kTileKeys * CH; idx += nthreads) {
    const int which = idx / (kTileKeys * CH);      // 0: K, 1: V
    const int rem = idx - which * kTileKeys * CH;
    const int row = rem / CH, ch = rem - row * CH;
    const int key = key0 + row;
    const uint16_t *src = P.k_new;                 // any valid address when zero-filling
    int bytes = 0;
    if (key < s.L) {
      src = (which ? P.v_cache : P.k_cache) + ((s.kv0 + key) * P.Hkv + hk) * D + ch * 8;
      bytes = 16;
    } else if (key < s.L + s.Ri) {
      src = (which ? P.v_new : P.k_new) +
            (static_cast<int64_t>(s.r0 + key - s.L) * P.Hkv + hk) * D + ch * 8;
      bytes = 16;
    }
    cp_async16(stage_base + which * (kTileKeys * D * 2) + swz<D>(row, ch), src, bytes);
  }
}

// ---------------------------------------------------------------------------
// bf16 kernel.  MT m-tiles of 16 packed query rows (row m = j*g + hg for block
// row j and head hk*g + hg); 4*MT warps: warp w works on m-tile w/4 and on
// keys (w%4)*16 .. +16 of every 64-key tile.
// ---------------------------------------------------------------------------
template <int D, int MT>
__device__ __forceinline__ void attn_bf16_body(const AttnParams &P, unsigned char *smem) {
  using SM = AttnSmem<D, MT>;
  constexpr int NT = MT * kKW * 32;
  constexpr int KS = D / 16;          // k-steps of Q.K^T
  constexpr int NB = D / 8;           // n-blocks of P.V
  const uint32_t sbase = smem_u32(smem);
  int32_t *seq_nt = reinterpret_cast<int32_t *>(smem + SM::kOffSched);
  int64_t *seq_base = reinterpret_cast<int64_t *>(smem + SM::kOffStages);  // before the pipeline
  int *misc = reinterpret_cast<int *>(smem + SM::kOffMisc);
  float *merge_o = reinterpret_cast<float *>(smem + SM::kOffMergeO);
  float2 *merge_ml = reinterpret_cast<float2 *>(smem + SM::kOffMergeML);
  int64_t *misc64 = reinterpret_cast<int64_t *>(misc + 8);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int mt = warp / kKW, kw = warp % kKW;
  const int B = P.B, Hkv = P.Hkv, g = P.g;

  // ---- schedule (identical in every CTA): tiles per sequence and prefix
  int bad = 0;
  for (int i = tid; i < B; i += NT) {
    const int r0 = P.cu_q[i], r1 = P.cu_q[i + 1], L = P.kv_len[i];
    const int64_t kv0 = P.kv_start[i];
    const bool ok = r0 >= 0 && r1 - r0 >= 1 && r1 - r0 <= P.max_q_rows && r1 <= P.num_rows &&
                    L >= 0 && kv0 >= 0 && kv0 + L <= P.pool_rows;
    bad |= !ok;
    seq_nt[i] = ok ? (L + (r1 - r0) + kTileKeys - 1) / kTileKeys : 0;
  }
  bad = __syncthreads_or(bad);
  if (bad && blockIdx.x == 0 && tid == 0) set_status(P.dev_status, SV_DEV_BAD_LENGTH);
  if (warp == 0) {
    int64_t carry = 0;
    for (int base = 0; base < B; base += 32) {
      const int i = base + lane;
      const int64_t v = i < B ? static_cast<int64_t>(seq_nt[i]) * Hkv : 0;
      int64_t inc = v;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int64_t t = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += t;
      }
      if (i < B) seq_base[i] = carry + inc - v;
      carry += __shfl_sync(0xffffffffu, inc, 31);
    }
    if (lane == 0) misc64[0] = carry;
  }
  __syncthreads();
  const int64_t W = misc64[0];
  if (W == 0) return;
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
    int lo = 0, hi = B - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (seq_base[mid] <= t_begin) lo = mid; else hi = mid - 1;
    }
    while (seq_nt[lo] == 0) ++lo;
    const int64_t rel = t_begin - seq_base[lo];
    cur.i = lo;
    cur.hk = static_cast<int>(rel / seq_nt[lo]);
    cur.lt = static_cast<int>(rel - static_cast<int64_t>(cur.hk) * seq_nt[lo]);
  }
  int64_t seg_first_tile = t_begin - cur.lt;   // global index of the segment's tile 0
  __syncthreads();                            // seq_base dead: tile buffers free

  // ---- prologue: first kStages-1 tiles in flight
  Cursor ld = cur;
  SeqInfo ld_s = load_seq(P, seq_nt, ld.i);
#pragma unroll
  for (int st = 0; st < kStages - 1; ++st) {
    if (st < ntiles) {
      issue_tile_loads<D>(P, ld_s, ld.hk, ld.lt, sbase + st * SM::kStageBytes, NT);
      if (cursor_advance(ld, seq_nt, Hkv, B) && st + 1 < ntiles) ld_s = load_seq(P, seq_nt, ld.i);
    }
    cp_async_commit();
  }

  SeqInfo cs = load_seq(P, seq_nt, cur.i);
  uint32_t qf[KS][4];
  float o[NB][4];
  float m_run[2], l_run[2];
  const int r = lane >> 2, c2 = (lane & 3) * 2;

  auto load_q = [&]() {
    const int M = cs.Ri * g;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int m = mt * 16 + r + h * 8;
      const bool ok = m < M;
      const int j = ok ? m / g : 0, hg = ok ? m - j * g : 0;
      const uint16_t *qrow = P.q + (static_cast<int64_t>(cs.r0 + j) * P.Hq + cur.hk * g + hg) * D;
#pragma unroll
      for (int ks = 0; ks < KS; ++ks) {
        qf[ks][h] = ok ? *reinterpret_cast<const uint32_t *>(qrow + ks * 16 + c2) : 0u;
        qf[ks][2 + h] = ok ? *reinterpret_cast<const uint32_t *>(qrow + ks * 16 + 8 + c2) : 0u;
      }
    }
  };
  auto reset_state = [&]() {
#pragma unroll
    for (int nb = 0; nb < NB; ++nb) o[nb][0] = o[nb][1] = o[nb][2] = o[nb][3] = 0.0f;
    m_run[0] = m_run[1] = -INFINITY;
    l_run[0] = l_run[1] = 0.0f;
  };
  load_q();
  reset_state();

  for (int k = 0; k < ntiles; ++k) {
    cp_async_wait<kStages - 2>();
    __syncthreads();
    {   // refill the stage consumed at k-1
      const int kn = k + kStages - 1;
      if (kn < ntiles) {
        issue_tile_loads<D>(P, ld_s, ld.hk, ld.lt, sbase + (kn % kStages) * SM::kStageBytes, NT);
        if (cursor_advance(ld, seq_nt, Hkv, B) && kn + 1 < ntiles) ld_s = load_seq(P, seq_nt, ld.i);
      }
      cp_async_commit();
    }
    const uint32_t kbase = sbase + (k % kStages) * SM::kStageBytes;
    const uint32_t vbase = kbase + SM::kTileBytes;
    const int mi = lane >> 3;                    // 8x8 matrix this lane addresses

    // ---- S = Q K^T over this warp's 16 keys
    float s[2][4];
#pragma unroll
    for (int nb = 0; nb < 2; ++nb) s[nb][0] = s[nb][1] = s[nb][2] = s[nb][3] = 0.0f;
    {
      const int krow = kw * 16 + ((mi >> 1) << 3) + (lane & 7);
#pragma unroll
      for (int ks = 0; ks < KS; ++ks) {
        uint32_t b0, b1, b2, b3;
        ldmatrix_x4(kbase + swz<D>(krow, ks * 2 + (mi & 1)), b0, b1, b2, b3);
        mma_bf16_16816(s[0], qf[ks], b0, b1);
        mma_bf16_16816(s[1], qf[ks], b2, b3);
      }
    }
    // ---- mask + online softmax for rows r and r+8
    const int key_w0 = cur.lt * kTileKeys + kw * 16;
    float p[2][4];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int m = mt * 16 + r + h * 8;
      const int j = min(m / g, cs.Ri - 1);
      const int lim = cs.L + j + 1;              // keys < lim are visible to row m
      float mx = -INFINITY;
#pragma unroll
      for (int nb = 0; nb < 2; ++nb)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int key = key_w0 + nb * 8 + c2 + e;
          const float v = key < lim ? s[nb][h * 2 + e] * P.sl2 : -INFINITY;
          s[nb][h * 2 + e] = v;
          mx = fmaxf(mx, v);
        }
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
      const float m_new = fmaxf(m_run[h], mx);
      const float m_use = m_new == -INFINITY ? 0.0f : m_new;
      const float alpha = exp2f(m_run[h] - m_use);
      float rs = 0.0f;
#pragma unroll
      for (int nb = 0; nb < 2; ++nb)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const float pv = exp2f(s[nb][h * 2 + e] - m_use);
          p[nb][h * 2 + e] = pv;
          rs += pv;
        }
      l_run[h] = l_run[h] * alpha + rs;
      m_run[h] = m_new;
#pragma unroll
      for (int nb = 0; nb < NB; ++nb) {
        o[nb][h * 2] *= alpha;
        o[nb][h * 2 + 1] *= alpha;
      }
    }
    // ---- O += P V (P stays in registers as the A operand)
    uint32_t pa[4];
    pa[0] = pack_bf16x2(p[0][0], p[0][1]);
    pa[1] = pack_bf16x2(p[0][2], p[0][3]);
    pa[2] = pack_bf16x2(p[1][0], p[1][1]);
    pa[3] = pack_bf16x2(p[1][2], p[1][3]);
    {
      const int vrow = kw * 16 + ((mi & 1) << 3) + (lane & 7);
#pragma unroll
      for (int nb = 0; nb < NB; nb += 2) {
        uint32_t b0, b1, b2, b3;
        ldmatrix_x4_trans(vbase + swz<D>(vrow, nb + (mi >> 1)), b0, b1, b2, b3);
        mma_bf16_16816(o[nb], pa, b0, b1);
        mma_bf16_16816(o[nb + 1], pa, b2, b3);
      }
    }

    const bool seg_end = cur.lt + 1 == cs.nt;
    const bool last = k + 1 == ntiles;
    if (!(seg_end || last)) {
      ++cur.lt;
      continue;
    }
    // ================= end of a piece =================
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      l_run[h] += __shfl_xor_sync(0xffffffffu, l_run[h], 1);
      l_run[h] += __shfl_xor_sync(0xffffffffu, l_run[h], 2);
    }
    if ((lane & 3) == 0) {
      merge_ml[(mt * kKW + kw) * 16 + r] = make_float2(m_run[0], l_run[0]);
      merge_ml[(mt * kKW + kw) * 16 + r + 8] = make_float2(m_run[1], l_run[1]);
    }
    __syncthreads();
    float mrow[2], lrow[2], sc[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      float mm = -INFINITY;
#pragma unroll
      for (int w2 = 0; w2 < kKW; ++w2) mm = fmaxf(mm, merge_ml[(mt * kKW + w2) * 16 + r + h * 8].x);
      const float mu = mm == -INFINITY ? 0.0f : mm;
      float ll = 0.0f;
#pragma unroll
      for (int w2 = 0; w2 < kKW; ++w2) {
        const float2 v = merge_ml[(mt * kKW + w2) * 16 + r + h * 8];
        ll += v.y * exp2f(v.x - mu);
      }
      mrow[h] = mm;
      lrow[h] = ll;
      sc[h] = exp2f(m_run[h] - mu);
    }
    // O of the 4 key-slice warps: kw = 3, 2, 1 accumulate into the buffer in
    // a fixed order, kw = 0 adds its own and owns the result.
    float *ob = merge_o + mt * 16 * D;
    for (int step = kKW - 1; step >= 1; --step) {
      if (kw == step) {
#pragma unroll
        for (int nb = 0; nb < NB; ++nb)
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            float2 *dst = reinterpret_cast<float2 *>(ob + (r + h * 8) * D + nb * 8 + c2);
            float2 a = make_float2(o[nb][h * 2] * sc[h], o[nb][h * 2 + 1] * sc[h]);
            if (step != kKW - 1) {
              const float2 b = *dst;
              a.x += b.x;
              a.y += b.y;
            }
            *dst = a;
          }
      }
      __syncthreads();
    }
    const int seg = cur.i * Hkv + cur.hk;
    const int64_t c_first = cta_of_tile(seg_first_tile, W, G);
    const int64_t c_last = cta_of_tile(seg_first_tile + cs.nt - 1, W, G);
    const int npieces = static_cast<int>(c_last - c_first + 1);
    const int Mi = cs.Ri * g;
    constexpr int rows_m = MT * 16;
    if (kw == 0) {
#pragma unroll
      for (int nb = 0; nb < NB; ++nb)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const float2 b = *reinterpret_cast<const float2 *>(ob + (r + h * 8) * D + nb * 8 + c2);
          o[nb][h * 2] = o[nb][h * 2] * sc[h] + b.x;
          o[nb][h * 2 + 1] = o[nb][h * 2 + 1] * sc[h] + b.y;
        }
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int m = mt * 16 + r + h * 8;
        if (m >= Mi) continue;
        if (npieces == 1) {            // whole segment here: normalize, store
          const int j = m / g, hg = m - j * g;
          const float inv = lrow[h] > 0.0f ? 1.0f / lrow[h] : 0.0f;
          uint16_t *orow = P.out + (static_cast<int64_t>(cs.r0 + j) * P.Hq + cur.hk * g + hg) * D;
#pragma unroll
          for (int nb = 0; nb < NB; ++nb)
            *reinterpret_cast<uint32_t *>(orow + nb * 8 + c2) =
                pack_bf16x2(o[nb][h * 2] * inv, o[nb][h * 2 + 1] * inv);
        } else {                       // partial: slot = CTA index + segment index
          const int64_t slot = static_cast<int64_t>(blockIdx.x) + seg;
          float *po = P.part_o + (slot * rows_m + m) * D;
#pragma unroll
          for (int nb = 0; nb < NB; ++nb)
            *reinterpret_cast<float2 *>(po + nb * 8 + c2) = make_float2(o[nb][h * 2], o[nb][h * 2 + 1]);
          if ((lane & 3) == 0) P.part_ml[slot * rows_m + m] = make_float2(mrow[h], lrow[h]);
        }
      }
    }
    if (npieces > 1) {
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
            const int64_t slot = c_first + c + seg;
            const float2 ml = __ldcg(&P.part_ml[slot * rows_m + m]);
            const float f = exp2f(ml.x - mu);
            const float2 ov = __ldcg(reinterpret_cast<const float2 *>(P.part_o + (slot * rows_m + m) * D + d));
            n0 += f * ov.x;
            n1 += f * ov.y;
            den += f * ml.y;
          }
          const float inv = den > 0.0f ? 1.0f / den : 0.0f;
          const int j = m / g, hg = m - j * g;
          *reinterpret_cast<uint32_t *>(P.out + (static_cast<int64_t>(cs.r0 + j) * P.Hq + cur.hk * g + hg) * D + d) =
              pack_bf16x2(n0 * inv, n1 * inv);
        }
      }
    }
    __syncthreads();                   // merge buffers reusable
    if (last) break;
    seg_first_tile += cs.nt;
    if (cursor_advance(cur, seq_nt, Hkv, B)) cs = load_seq(P, seq_nt, cur.i);
    load_q();
    reset_state();
  }
  cp_async_wait<0>();
}

template <int D, int MT>
__global__ void __launch_bounds__(MT * kKW * 32) attn_bf16_kernel(const AttnParams P) {
  extern __shared__ __align__(128) unsigned char smem[];
  attn_bf16_body<D, MT>(P, smem);
  // A dependent launch (fused step) must not complete before its primary.
  if (P.pdl_secondary) asm volatile("griddepcontrol.wait;\n" ::: "memory");
}

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

template <int D, int MT>
cudaError_t launch_bf16(const AttnParams &P, int grid, cudaStream_t s) {
  using SM = AttnSmem<D, MT>;
  auto kern = attn_bf16_kernel<D, MT>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SM::kBytes);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(MT * kKW * 32);
  cfg.dynamicSmemBytes = SM::kBytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = P.pdl_secondary ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, P);
}

template <int D, int MT>
int occupancy_bf16() {
  using SM = AttnSmem<D, MT>;
  auto kern = attn_bf16_kernel<D, MT>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SM::kBytes) != cudaSuccess)
    return 1;
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, MT * kKW * 32, SM::kBytes) != cudaSuccess)
    return 1;
  return n > 0 ? n : 1;
}

int occupancy_for(int D, int MT) {
  static int cache[2][5] = {{0}};
  const int di = D == 128 ? 1 : 0;
  if (cache[di][MT] == 0) {
    int n = 1;
    if (D == 64) {
      switch (MT) { case 1: n = occupancy_bf16<64, 1>(); break; case 2: n = occupancy_bf16<64, 2>(); break;
                    case 3: n = occupancy_bf16<64, 3>(); break; default: n = occupancy_bf16<64, 4>(); }
    } else {
      switch (MT) { case 1: n = occupancy_bf16<128, 1>(); break; case 2: n = occupancy_bf16<128, 2>(); break;
                    case 3: n = occupancy_bf16<128, 3>(); break; default: n = occupancy_bf16<128, 4>(); }
    }
    cache[di][MT] = n;
  }
  return cache[di][MT];
}

}  // namespace

AttnPlan plan_attention(const sv_attn_args &a, int num_sms) {
  AttnPlan p;
  const int g = a.num_q_heads / a.num_kv_heads;
  p.rows_m = a.max_q_rows * g;
  p.m_tiles = (p.rows_m + 15) / 16;
  // sum over sequences of ceil((L_i + R_i) / 64), per KV head
  p.tiles_bound = static_cast<int64_t>(a.num_kv_heads) *
                  ((a.kv_rows_bound + a.num_rows) / kTileKeys + a.batch);
  p.grid = 1;
  if (a.dtype == SV_BF16 && num_sms > 0) {
    const int occ = occupancy_for(a.head_dim, p.m_tiles);
    p.grid = std::max<int64_t>(1, std::min<int64_t>(static_cast<int64_t>(num_sms) * occ, p.tiles_bound));
  }
  return p;
}

int attention_max_batch() { return kMaxBatch; }

size_t attention_partials_bytes(const sv_attn_args &a, const AttnPlan &p) {
  if (a.dtype != SV_BF16) return 0;
  // slot = CTA index + segment index < grid + B * Hkv
  const int64_t slots = p.grid + static_cast<int64_t>(a.batch) * a.num_kv_heads;
  const int64_t rows = static_cast<int64_t>(p.m_tiles) * 16;
  return static_cast<size_t>(slots * rows * a.head_dim * 4 + slots * rows * 8);
}

cudaError_t launch_attention(const sv_attn_args &a, const AttnPlan &p, float *part_o,
                             float *part_ml, uint32_t *counters, bool pdl_secondary,
                             cudaStream_t s) {
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
  P.part_o = part_o;
  P.part_ml = reinterpret_cast<float2 *>(part_ml);
  P.counters = counters;
  P.dev_status = a.dev_status;
  P.tiles_bound = p.tiles_bound;
  P.pdl_secondary = pdl_secondary ? 1 : 0;
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
  const int grid = static_cast<int>(p.grid);
  if (a.head_dim == 64) {
    switch (p.m_tiles) {
      case 1: return launch_bf16<64, 1>(P, grid, s);
      case 2: return launch_bf16<64, 2>(P, grid, s);
      case 3: return launch_bf16<64, 3>(P, grid, s);
      default: return launch_bf16<64, 4>(P, grid, s);
    }
  }
  switch (p.m_tiles) {
    case 1: return launch_bf16<128, 1>(P, grid, s);
    case 2: return launch_bf16<128, 2>(P, grid, s);
    case 3: return launch_bf16<128, 3>(P, grid, s);
    default: return launch_bf16<128, 4>(P, grid, s);
  }
}

}  // namespace sv

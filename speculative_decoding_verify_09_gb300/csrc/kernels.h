// Internal interface between the C-ABI layer (api.cu) and the kernels.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "spec_verify.h"

namespace sv {

constexpr int kMaxQRows = 16;   // bound on K_i + 1 block rows per sequence
constexpr int kMaxRowsM = 64;   // bound on (K_i + 1) * (Hq / Hkv) packed query rows
constexpr int kSmemMax = 227 * 1024;   // dynamic shared memory one CTA may ask for

// Per logits row statistics written by the sampler's first phase.
struct RowStats {
  float lmax;         // largest logit of the row
  uint32_t tau_key;   // nucleus threshold as an order-preserving key (0: keep all)
  uint32_t valid;     // 0: NaN / +inf / only -inf in the row
  float inv_hi;       // 1 / ssum as a float-float pair
  float inv_lo;
  int32_t amax;       // greedy row (temperature 0): index of the one-hot; else -1
  float c_hi, c_lo;   // log2(e) / T of the row's sequence as a float pair
  float acc_hi, acc_lo;   // sum over the kept set of exp((l - lmax) / T) from float-float
                          // weights (~1e-13), for residual draws
  float it_hi, it_lo;     // 1 / T of the row's sequence as a float pair
};

// Partial (max, sum) of one chunk of a row (chunked statistics).
struct ChunkPart {
  float m;            // chunk max
  float s_hi, s_lo;   // sum of exp((l - m) / T) over the chunk, float-float
  uint32_t bad;       // NaN / +inf seen
  float a_hi, a_lo;   // the same sum from float-float weights
};

// Sampler workspace regions (device pointers).
struct SamplerWs {
  RowStats *stats;          // [2R - B]
  uint32_t *row_cnt;        // [2R - B] chunk arrivals per row (zero between calls)
  uint32_t *seq_cnt1;       // [B] row arrivals per sequence (zero between calls)
  uint32_t *seq_cnt2;       // [B] draw-chunk arrivals per sequence (zero between calls)
  ChunkPart *parts;         // [(2R - B) * stat_chunks]
  unsigned __int128 *draw_parts;    // [B * draw_chunks] fixed-point (2^-116) chunk sums
  unsigned __int128 *draw_thr;      // [B * draw_chunks * draw_threads] the chunks' per-thread
                                    // run sums (runs in vocabulary order)
};

struct SamplerPlan {
  int stat_chunks;          // CTAs per row in the statistics phase (1: nucleus path)
  int draw_chunks;          // CTAs per sequence in the draw phase (<= 128; one run per thread)
  int draw_threads;         // threads per draw CTA (one run of the chunk each)
  bool cluster;             // one CTA cluster per sequence (no nucleus, rows fit in smem)
  int cluster_nvt;          // 16-byte vectors per thread and row in the cluster kernel (1, 2)
  int win_stats;            // bf16 rows off the cluster path: the window-histogram
                            // statistics kernel (0: the f32 kernels)
};

struct AppendView {   // what the fused step's append needs (all device pointers)
  const void *k_new, *v_new;
  void *k_cache, *v_cache;
  int64_t pool_rows;
  const int64_t *kv_start;
  const int32_t *kv_cap;
  int32_t *new_kv_len;
  int32_t row_bytes;  // Hkv * D * element size
};

struct SamplerLaunch {
  sv_sample_args a;
  SamplerWs ws;
  SamplerPlan plan;
  bool do_append;
  AppendView app;
  bool pdl_secondary;       // launched early behind the attention: wait for it at the end
  uint32_t philox_stream;   // 0: the verify step's uniforms; 1: draft-token draws
};

SamplerPlan plan_sampler(const sv_sample_args &a);
int sampler_max_vocab(int dtype);
cudaError_t launch_sampler(const SamplerLaunch &L, cudaStream_t s);

cudaError_t launch_append(int32_t B, int32_t row_bytes, int32_t max_q_rows, int64_t num_rows,
                          const int32_t *cu_q, const void *k_new, const void *v_new,
                          void *k_cache, void *v_cache, int64_t pool_rows,
                          const int64_t *kv_start, const int32_t *kv_len, const int32_t *kv_cap,
                          const int32_t *num_accepted, int32_t *new_kv_len,
                          uint32_t *dev_status, cudaStream_t s);

// Attention split plan: chosen on the host from the bounds.
struct AttnPlan {
  int rows_m;           // packed query rows per (sequence, KV head): max_q_rows * Hq/Hkv
  int row_cfg;          // kernel row configuration (rows per CTA: 8, 16, 32, 48, 64)
  int m_tiles;          // partial-slot rows / 16
  int64_t grid;         // bound on the persistent CTAs (bf16 path; sizes the partials)
  int64_t tiles_bound;  // bound on the global count of 64-key tiles
  // shared-prefix arrangement (num_groups > 0)
  bool prefix;
  int spb;              // whole sequences per prefix row-block
  int64_t pre_grid, pre_tiles_bound, pre_slots;
};

// Device regions of the attention workspace.
struct AttnWs {
  uint32_t *counters;   // [B * Hkv]
  float *dec_o, *dec_ml;      // decode partials
  float *pre_o, *pre_ml;      // prefix partials
};

// Polls of one attention pipeline wait before it gives up with SV_DEV_TIMEOUT
// (0: the built-in bound); set by sv_set_wait_limit, read at each launch.
uint32_t attention_wait_limit();

// num_sms = 0: device-independent plan (grids at their upper bound).
AttnPlan plan_attention(const sv_attn_args &a, int num_sms);
int attention_max_batch();
int attention_max_groups();
int attention_slot_rows(const AttnPlan &p);   // rows per decode partial slot
int attention_prefix_rows();                  // rows per prefix partial slot
// How one attention call is launched.
struct AttnLaunchOpts {
  bool pdl_primary;     // the next launch on the stream may start at once
  int smem_cap;         // shared memory budget of one CTA (sets the ring depth)
  int smem_min;         // ask for at least this much (0: no floor)
  int num_sms;          // SMs of the device (grid = SMs x resident CTAs per SM)
};
cudaError_t launch_attention(const sv_attn_args &a, const AttnPlan &p, const AttnWs &ws,
                             const AttnLaunchOpts &opts, cudaStream_t s);
// Shared memory the cluster sampler asks for per CTA (0 if it is not used).
int sampler_cluster_smem(const SamplerPlan &p);

}  // namespace sv

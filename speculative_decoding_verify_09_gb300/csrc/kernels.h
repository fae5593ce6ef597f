// Internal interface between the C-ABI layer (api.cu) and the kernels.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "spec_verify.h"

namespace sv {

constexpr int kMaxQRows = 16;   // bound on K_i + 1 block rows per sequence
constexpr int kMaxRowsM = 64;   // bound on (K_i + 1) * (Hq / Hkv) packed query rows

// Per logits row statistics written by the sampler's row pass.
struct RowStats {
  float lmax;         // largest logit of the row
  uint32_t tau_key;   // nucleus threshold as an order-preserving key (0: keep all)
  uint32_t valid;     // 0: NaN / +inf / only -inf in the row
  uint32_t pad;
  double ssum;        // sum over the kept set of exp((l - lmax) / T)
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
  RowStats *stats;          // [2R - B]
  uint32_t *counters;       // [B], zero between calls
  bool do_append;
  AppendView app;
  bool pdl_primary;         // trigger dependent launch at kernel start
};

// Sizes of the sampler's workspace parts.
size_t sampler_stats_bytes(const sv_sample_args &a);
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
  int m_tiles;          // ceil(rows_m / 16)
  int64_t grid;         // persistent CTAs (bf16 path)
  int64_t tiles_bound;  // bound on the global count of 64-key tiles
};

AttnPlan plan_attention(const sv_attn_args &a, int num_sms);
size_t attention_partials_bytes(const sv_attn_args &a, const AttnPlan &p);
int attention_max_batch();
cudaError_t launch_attention(const sv_attn_args &a, const AttnPlan &p, float *part_o,
                             float *part_ml, uint32_t *counters, bool pdl_secondary,
                             cudaStream_t s);

}  // namespace sv

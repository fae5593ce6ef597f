// Ragged append of the accepted K/V rows (sm_103a).
//
// "EMS-SD: Efficient Multi-sample Speculative Decoding" (abstract): samples
// accept different numbers of tokens and no padding tokens are added.  Here
// block rows 0..n_i of sequence i (pending token + accepted drafts) are
// copied to pool rows kv_start_i + L_i .. + n_i; rows of one sequence are
// contiguous on both sides, so each sequence is two flat copies done with
// 16-byte vector loads and stores.
#include "common.cuh"
#include "kernels.h"

namespace sv {

namespace {

constexpr int kAppNT = 256;

struct AppParams {
  int32_t B, row_bytes, max_q_rows;
  int64_t num_rows, pool_rows;
  const int32_t *cu_q;
  const char *k_new, *v_new;
  char *k_cache, *v_cache;
  const int64_t *kv_start;
  const int32_t *kv_len, *kv_cap, *num_accepted;
  int32_t *new_kv_len;
  uint32_t *dev_status;
};

// grid: (B, slices); slice y copies every gridDim.y-th 16-byte vector.
__global__ void __launch_bounds__(kAppNT) append_kernel(const AppParams P) {
  const int i = blockIdx.x;
  const int r0 = P.cu_q[i], Ri = P.cu_q[i + 1] - r0;
  const int n = P.num_accepted[i];
  const int L = P.kv_len[i];
  const bool first = blockIdx.y == 0 && threadIdx.x == 0;
  if (r0 < 0 || Ri < 1 || Ri > P.max_q_rows || r0 + Ri > P.num_rows || L < 0) {
    if (first) {
      set_status(P.dev_status, SV_DEV_BAD_LENGTH);
      P.new_kv_len[i] = L;
    }
    return;
  }
  if (n < 0 || n >= Ri) {            // failed sequence: nothing to append
    if (first) P.new_kv_len[i] = L;
    return;
  }
  if (L + n + 1 > P.kv_cap[i]) {
    if (first) {
      set_status(P.dev_status, SV_DEV_CAPACITY);
      P.new_kv_len[i] = L;
    }
    return;
  }
  const int64_t start = P.kv_start[i];
  if (start < 0 || start + L + n + 1 > P.pool_rows) {
    if (first) {
      set_status(P.dev_status, SV_DEV_BAD_LENGTH);
      P.new_kv_len[i] = L;
    }
    return;
  }
  const int64_t nvec = static_cast<int64_t>(n + 1) * P.row_bytes / 16;
  const uint4 *sk = reinterpret_cast<const uint4 *>(P.k_new + static_cast<int64_t>(r0) * P.row_bytes);
  const uint4 *sv_ = reinterpret_cast<const uint4 *>(P.v_new + static_cast<int64_t>(r0) * P.row_bytes);
  uint4 *dk = reinterpret_cast<uint4 *>(P.k_cache + (start + L) * P.row_bytes);
  uint4 *dv = reinterpret_cast<uint4 *>(P.v_cache + (start + L) * P.row_bytes);
  for (int64_t v = static_cast<int64_t>(blockIdx.y) * kAppNT + threadIdx.x; v < nvec;
       v += static_cast<int64_t>(gridDim.y) * kAppNT) {
    dk[v] = __ldg(sk + v);
    dv[v] = __ldg(sv_ + v);
  }
  if (first) P.new_kv_len[i] = L + n + 1;
}

}  // namespace

cudaError_t launch_append(int32_t B, int32_t row_bytes, int32_t max_q_rows, int64_t num_rows,
                          const int32_t *cu_q, const void *k_new, const void *v_new,
                          void *k_cache, void *v_cache, int64_t pool_rows,
                          const int64_t *kv_start, const int32_t *kv_len, const int32_t *kv_cap,
                          const int32_t *num_accepted, int32_t *new_kv_len,
                          uint32_t *dev_status, cudaStream_t s) {
  if (B <= 0) return cudaSuccess;
  AppParams P;
  P.B = B;
  P.row_bytes = row_bytes;
  P.max_q_rows = max_q_rows;
  P.num_rows = num_rows;
  P.pool_rows = pool_rows;
  P.cu_q = cu_q;
  P.k_new = static_cast<const char *>(k_new);
  P.v_new = static_cast<const char *>(v_new);
  P.k_cache = static_cast<char *>(k_cache);
  P.v_cache = static_cast<char *>(v_cache);
  P.kv_start = kv_start;
  P.kv_len = kv_len;
  P.kv_cap = kv_cap;
  P.num_accepted = num_accepted;
  P.new_kv_len = new_kv_len;
  P.dev_status = dev_status;
  const int64_t max_vec = static_cast<int64_t>(max_q_rows) * row_bytes / 16;
  const int slices = static_cast<int>(std::min<int64_t>(8, (max_vec + kAppNT * 4 - 1) / (kAppNT * 4)));
  append_kernel<<<dim3(B, slices > 0 ? slices : 1), kAppNT, 0, s>>>(P);
  return cudaGetLastError();
}

}  // namespace sv

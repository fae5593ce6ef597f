// C ABI of the verify step: argument checks, workspace layout, launches.
// See include/spec_verify.h for the contract of every entry point.
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>

#include <cuda.h>

#include "kernels.h"

namespace {

thread_local std::string g_err;

sv_status fail(sv_status st, const char *fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_err = buf;
  return st;
}

sv_status cuda_fail(cudaError_t e, const char *what) {
  return fail(SV_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

constexpr size_t kAlign = 256;

size_t round_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

sv_status check_attn(const sv_attn_args *a) {
  if (!a) return fail(SV_ERR_INVALID, "attention args: null");
  if (a->batch < 0 || a->batch > sv::attention_max_batch())
    return fail(SV_ERR_INVALID, "attention: batch %d outside [0, %d]", a->batch,
                sv::attention_max_batch());
  if (a->num_q_heads < 1 || a->num_kv_heads < 1 || a->num_q_heads % a->num_kv_heads)
    return fail(SV_ERR_INVALID, "attention: heads Hq=%d Hkv=%d (need Hq %% Hkv == 0)",
                a->num_q_heads, a->num_kv_heads);
  if (a->head_dim != 64 && a->head_dim != 128)
    return fail(SV_ERR_UNSUPPORTED, "attention: head_dim %d (built: 64, 128)", a->head_dim);
  if (a->dtype != SV_F32 && a->dtype != SV_BF16)
    return fail(SV_ERR_INVALID, "attention: dtype %d", a->dtype);
  if (a->max_q_rows < 1 || a->max_q_rows > sv::kMaxQRows)
    return fail(SV_ERR_INVALID, "attention: max_q_rows %d outside [1, %d]", a->max_q_rows,
                sv::kMaxQRows);
  const int g = a->num_q_heads / a->num_kv_heads;
  if (a->max_q_rows * g > sv::kMaxRowsM)
    return fail(SV_ERR_UNSUPPORTED, "attention: max_q_rows * Hq/Hkv = %d > %d",
                a->max_q_rows * g, sv::kMaxRowsM);
  if (a->num_rows < a->batch || a->num_rows > static_cast<int64_t>(a->batch) * a->max_q_rows)
    return fail(SV_ERR_INVALID, "attention: num_rows %lld inconsistent with batch %d and max_q_rows %d",
                static_cast<long long>(a->num_rows), a->batch, a->max_q_rows);
  if (a->kv_rows_bound < 0 || a->pool_rows < 0)
    return fail(SV_ERR_INVALID, "attention: negative kv_rows_bound or pool_rows");
  if (!std::isfinite(a->scale) || a->scale < 0.0f)
    return fail(SV_ERR_INVALID, "attention: scale must be finite and >= 0");
  if (a->num_groups < 0 || a->num_groups > sv::attention_max_groups())
    return fail(SV_ERR_INVALID, "attention: num_groups %d outside [0, %d]", a->num_groups,
                sv::attention_max_groups());
  if (a->kv_dtype != 0 && a->kv_dtype != SV_E4M3)
    return fail(SV_ERR_INVALID, "attention: kv_dtype %d", a->kv_dtype);
  if (a->kv_dtype == SV_E4M3) {
    if (a->dtype != SV_BF16 || a->head_dim != 128 || a->num_groups > 0 ||
        a->max_q_rows * g > 16)
      return fail(SV_ERR_UNSUPPORTED,
                  "attention: E4M3 K/V built for bf16 q/out, head_dim 128, no shared prefix, "
                  "(Hq/Hkv)*max_q_rows <= 16");
    if (!std::isfinite(a->k_scale) || a->k_scale < 0.0f || !std::isfinite(a->v_scale) ||
        a->v_scale < 0.0f)
      return fail(SV_ERR_INVALID, "attention: k_scale / v_scale must be finite and >= 0");
  }
  if (a->num_groups > 0) {
    if (a->dtype != SV_BF16)
      return fail(SV_ERR_UNSUPPORTED, "attention: shared prefix built for bf16 only");
    if (a->prefix_rows_bound < 0)
      return fail(SV_ERR_INVALID, "attention: negative prefix_rows_bound");
    if (a->batch > 0 && (!a->group || !a->prefix_start || !a->prefix_len))
      return fail(SV_ERR_INVALID, "attention: null shared-prefix pointer");
  }
  if (a->batch > 0) {
    if (!a->cu_q || !a->q || !a->k_new || !a->v_new || !a->kv_start || !a->kv_len || !a->out)
      return fail(SV_ERR_INVALID, "attention: null device pointer");
    if (a->pool_rows > 0 && (!a->k_cache || !a->v_cache))
      return fail(SV_ERR_INVALID, "attention: null cache pointer");
    if (!aligned16(a->q) || !aligned16(a->k_new) || !aligned16(a->v_new) || !aligned16(a->out) ||
        !aligned16(a->k_cache) || !aligned16(a->v_cache))
      return fail(SV_ERR_INVALID, "attention: tensors must be 16-byte aligned");
  }
  return SV_OK;
}

sv_status check_sample(const sv_sample_args *a) {
  if (!a) return fail(SV_ERR_INVALID, "sampling args: null");
  if (a->batch < 0) return fail(SV_ERR_INVALID, "sampling: batch %d", a->batch);
  if (a->vocab < 1 || a->vocab > sv::sampler_max_vocab(a->dtype))
    return fail(SV_ERR_UNSUPPORTED, "sampling: vocab %d outside [1, %d]", a->vocab,
                sv::sampler_max_vocab(a->dtype));
  if (a->dtype != SV_F32 && a->dtype != SV_BF16)
    return fail(SV_ERR_INVALID, "sampling: dtype %d", a->dtype);
  if (a->max_q_rows < 1 || a->max_q_rows > sv::kMaxQRows)
    return fail(SV_ERR_INVALID, "sampling: max_q_rows %d outside [1, %d]", a->max_q_rows,
                sv::kMaxQRows);
  if (a->num_rows < a->batch || a->num_rows > static_cast<int64_t>(a->batch) * a->max_q_rows)
    return fail(SV_ERR_INVALID, "sampling: num_rows %lld inconsistent with batch %d and max_q_rows %d",
                static_cast<long long>(a->num_rows), a->batch, a->max_q_rows);
  if (!(a->temperature >= 0.0f) || !std::isfinite(a->temperature))
    return fail(SV_ERR_INVALID, "sampling: temperature must be finite and >= 0 (0 = greedy)");
  if (a->top_k < 0) return fail(SV_ERR_INVALID, "sampling: top_k must be >= 0");
  if (!(a->top_p > 0.0f) || std::isnan(a->top_p))
    return fail(SV_ERR_INVALID, "sampling: top_p must be > 0");
  if (a->batch > 0) {
    if (!a->cu_q || !a->target_logits || !a->kv_len || !a->num_accepted || !a->out_tokens)
      return fail(SV_ERR_INVALID, "sampling: null device pointer");
    if (a->num_rows > a->batch && (!a->draft_logits || !a->draft_tokens))
      return fail(SV_ERR_INVALID, "sampling: null draft pointer");
  }
  return SV_OK;
}

sv_status check_draft(const sv_draft_args *d) {
  if (!d) return fail(SV_ERR_INVALID, "draft args: null");
  if (d->batch < 0) return fail(SV_ERR_INVALID, "draft: batch %d", d->batch);
  if (d->dtype != SV_F32 && d->dtype != SV_BF16)
    return fail(SV_ERR_INVALID, "draft: dtype %d", d->dtype);
  if (d->vocab < 1 || d->vocab > sv::sampler_max_vocab(d->dtype))
    return fail(SV_ERR_UNSUPPORTED, "draft: vocab %d outside [1, %d]", d->vocab,
                sv::sampler_max_vocab(d->dtype));
  if (!(d->temperature >= 0.0f) || !std::isfinite(d->temperature))
    return fail(SV_ERR_INVALID, "draft: temperature must be finite and >= 0 (0 = greedy)");
  if (d->top_k < 0) return fail(SV_ERR_INVALID, "draft: top_k must be >= 0");
  if (!(d->top_p > 0.0f) || std::isnan(d->top_p))
    return fail(SV_ERR_INVALID, "draft: top_p must be > 0");
  if (d->batch > 0 && (!d->draft_logits || !d->kv_len || !d->draft_tokens))
    return fail(SV_ERR_INVALID, "draft: null device pointer");
  return SV_OK;
}

// A draft draw as a sampling call: one block row per sequence (null cu_q, so
// the kernels take cu_q[i] = i), the draft logits in the target-row slot, no
// draft rows; every sequence then takes the bonus draw on its row.
sv_sample_args draft_as_sample(const sv_draft_args *d) {
  sv_sample_args s{};
  s.batch = d->batch;
  s.vocab = d->vocab;
  s.dtype = d->dtype;
  s.max_q_rows = 1;
  s.num_rows = d->batch;
  s.temperature = d->temperature;
  s.top_p = d->top_p;
  s.seed = d->seed;
  s.target_logits = d->draft_logits;
  s.draft_logits = d->draft_logits;   // never read (no draft rows); keeps row pointers non-null
  s.kv_len = d->kv_len;
  s.seq_ids = d->seq_ids;
  s.out_tokens = d->draft_tokens;
  s.dev_status = d->dev_status;
  s.top_k = d->top_k;
  s.temperatures = d->temperatures;
  s.top_ps = d->top_ps;
  s.top_ks = d->top_ks;
  return s;
}

struct Layout {
  size_t cnt_attn, row_cnt, seq_cnt1, seq_cnt2, stats, parts, draw_parts;
  size_t part_o, part_ml, pre_o, pre_ml, total;
  sv::AttnPlan plan;
  sv::SamplerPlan splan;
};

// Workspace: [attention counters | sampler counters | row stats | partials].
// The counter regions must be zero before a call and are left zero after it.
Layout layout(const sv_attn_args *a, const sv_sample_args *s) {
  Layout L{};
  size_t off = 0;
  if (a) {
    L.cnt_attn = off;
    off += round_up(static_cast<size_t>(a->batch) * a->num_kv_heads * 4);
  }
  if (s) {
    const size_t rows = static_cast<size_t>(2 * s->num_rows - s->batch);
    L.splan = sv::plan_sampler(*s);
    L.row_cnt = off;                      // counters first: zeroed once, left zero
    off += round_up(rows * 4);
    L.seq_cnt1 = off;
    off += round_up(static_cast<size_t>(s->batch) * 4);
    L.seq_cnt2 = off;
    off += round_up(static_cast<size_t>(s->batch) * 4);
    L.stats = off;
    off += round_up(rows * sizeof(sv::RowStats));
    L.parts = off;
    off += round_up(rows * L.splan.stat_chunks * sizeof(sv::ChunkPart));
    L.draw_parts = off;
    off += round_up(static_cast<size_t>(s->batch) * L.splan.draw_chunks *
                    (1 + static_cast<size_t>(L.splan.draw_threads)) * 16);
  }
  if (a) {
    // size the partials for the largest grids any device could get
    L.plan = sv::plan_attention(*a, 0);
    const bool bf = a->dtype == SV_BF16;
    const int64_t slots = L.plan.grid + static_cast<int64_t>(a->batch) * a->num_kv_heads;
    const int64_t rows = sv::attention_slot_rows(L.plan);
    L.part_o = off;
    off += round_up(bf ? static_cast<size_t>(slots * rows * a->head_dim * 4) : 0);
    L.part_ml = off;
    off += round_up(bf ? static_cast<size_t>(slots * rows * 8) : 0);
    const int64_t prows = sv::attention_prefix_rows();
    L.pre_o = off;
    off += round_up(L.plan.prefix ? static_cast<size_t>(L.plan.pre_slots * prows * a->head_dim * 4) : 0);
    L.pre_ml = off;
    off += round_up(L.plan.prefix ? static_cast<size_t>(L.plan.pre_slots * prows * 8) : 0);
  }
  L.total = off;
  return L;
}

int num_sms_current() {
  static int cache[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  if (cache[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    cache[dev] = n;
  }
  return cache[dev];
}

sv_status check_ws(void *ws, size_t ws_bytes, size_t need) {
  if (need == 0) return SV_OK;
  if (!ws) return fail(SV_ERR_WORKSPACE, "workspace: null (need %zu bytes)", need);
  if (!aligned16(ws)) return fail(SV_ERR_WORKSPACE, "workspace: not 16-byte aligned");
  if (ws_bytes < need)
    return fail(SV_ERR_WORKSPACE, "workspace: %zu bytes given, %zu needed", ws_bytes, need);
  return SV_OK;
}

template <typename T>
T *at(void *ws, size_t off) {
  return reinterpret_cast<T *>(static_cast<char *>(ws) + off);
}

// Per-device shared-memory facts used to size the attention ring.
struct SmemFacts {
  int per_sm;          // shared memory of one SM
  int reserved;        // shared memory the system keeps per CTA
};

SmemFacts smem_facts() {
  static SmemFacts cache[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return SmemFacts{0, 0};
  if (cache[dev].per_sm == 0) {
    int a = 0, b = 0;
    if (cudaDeviceGetAttribute(&a, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&b, cudaDevAttrReservedSharedMemoryPerBlock, dev) != cudaSuccess)
      return SmemFacts{0, 0};
    cache[dev] = SmemFacts{a, b};
  }
  return cache[dev];
}

// Attention alone: two persistent CTAs per SM (two independent load streams
// and twice the consumer warps to hide MMA latency), each with the deepest
// ring that fits half an SM.
sv::AttnLaunchOpts opts_alone() {
  const SmemFacts f = smem_facts();
  const int half = f.per_sm > 0 ? f.per_sm / 2 - f.reserved : sv::kSmemMax;
  return sv::AttnLaunchOpts{false, std::min(half, sv::kSmemMax), 0, num_sms_current()};
}

// Attention ahead of the sampler in the fused step; the sampling launch may
// start at once.  With the cluster sampler (one CTA per SM, small shared
// memory) each SM keeps room for one sampler CTA beside two attention CTAs, so
// the latency-bound sampling runs under the bandwidth-bound attention: the
// attention CTAs take at most (SM - sampler CTA) / 2 and more than a third of
// the SM (so three of them never share one SM).
sv::AttnLaunchOpts opts_step(const sv::SamplerPlan &sp) {
  sv::AttnLaunchOpts o = opts_alone();
  o.pdl_primary = true;
  const SmemFacts f = smem_facts();
  const int samp = sv::sampler_cluster_smem(sp);
  if (f.per_sm <= 0 || samp <= 0) return o;
  const int cap = (f.per_sm - samp - 3 * f.reserved) / 2;
  const int floor3 = f.per_sm / 3 - f.reserved + 16;
  if (cap > floor3) {
    o.smem_cap = cap;
    o.smem_min = floor3;
  }
  return o;
}

sv_status run_attention(const sv_attn_args *a, const Layout &L, void *ws,
                        const sv::AttnLaunchOpts &opts, cudaStream_t s) {
  if (a->batch == 0) return SV_OK;
  const int sms = num_sms_current();
  if (sms <= 0) return fail(SV_ERR_CUDA, "no CUDA device");
  sv::AttnPlan plan = sv::plan_attention(*a, sms);   // grids never exceed the sized ones
  sv::AttnWs w;
  w.counters = at<uint32_t>(ws, L.cnt_attn);
  w.dec_o = at<float>(ws, L.part_o);
  w.dec_ml = at<float>(ws, L.part_ml);
  w.pre_o = at<float>(ws, L.pre_o);
  w.pre_ml = at<float>(ws, L.pre_ml);
  cudaError_t e = sv::launch_attention(*a, plan, w, opts, s);
  if (e != cudaSuccess) return cuda_fail(e, "attention launch");
  return SV_OK;
}

sv::SamplerLaunch sampler_launch(const sv_sample_args *sample, const Layout &L, void *ws) {
  sv::SamplerLaunch SL{};
  SL.a = *sample;
  SL.plan = L.splan;
  SL.ws.stats = at<sv::RowStats>(ws, L.stats);
  SL.ws.row_cnt = at<uint32_t>(ws, L.row_cnt);
  SL.ws.seq_cnt1 = at<uint32_t>(ws, L.seq_cnt1);
  SL.ws.seq_cnt2 = at<uint32_t>(ws, L.seq_cnt2);
  SL.ws.parts = at<sv::ChunkPart>(ws, L.parts);
  SL.ws.draw_parts = at<unsigned __int128>(ws, L.draw_parts);
  SL.ws.draw_thr = SL.ws.draw_parts + static_cast<size_t>(SL.a.batch) * L.splan.draw_chunks;
  return SL;
}

}  // namespace

// Scratch of spec_verify_attn_static: a fixed array in the library's own device
// image instead of a caller workspace.  It exists for callers that may not
// allocate device memory at call time -- an embedder whose device memory is
// owned by another allocator, or a serving runtime that forbids allocation once
// it has started -- and so cannot supply the workspace the other entry points
// take.  One copy per device (per CUDA context that loads the library).
static __device__ __align__(256) unsigned char g_static_scratch[SV_STATIC_SCRATCH_BYTES];

namespace {

std::atomic<uint32_t> g_wait_limit{0};

}  // namespace

namespace sv {
uint32_t attention_wait_limit() { return g_wait_limit.load(std::memory_order_relaxed); }
}  // namespace sv

namespace {

// Front zone of g_static_scratch that holds only merge counters (B * Hkv words).
constexpr size_t kStaticCounterBytes = 64 * 1024;

// The array's device address belongs to a CUDA context, not to a device
// ordinal: after cudaDeviceReset, or under a context that a driver-API caller
// created and made current, the same ordinal has a new context with its own
// copy of the array.  So the looked-up address and the "cleared" state are
// kept per context, keyed by the driver's context id (unique for the life of
// the process, never reused).  The two driver calls are fetched through the
// runtime, so the library does not link the driver library itself.
typedef CUresult (*CtxGetCurrentFn)(CUcontext *);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long *);

struct StaticEntry {
  unsigned long long ctx_id;
  void *ptr;
};

std::mutex g_static_mu;
constexpr int kStaticCtxCap = 64;
StaticEntry g_static_tab[kStaticCtxCap] = {};
int g_static_used = 0, g_static_next = 0;
CtxGetCurrentFn g_ctx_current = nullptr;
CtxGetIdFn g_ctx_id = nullptr;

sv_status current_context_id(unsigned long long *id) {
  if (!g_ctx_current || !g_ctx_id) {
    void *f0 = nullptr, *f1 = nullptr;
    cudaDriverEntryPointQueryResult q0{}, q1{};
    cudaError_t e = cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f0, 12000,
                                                     cudaEnableDefault, &q0);
    if (e == cudaSuccess)
      e = cudaGetDriverEntryPointByVersion("cuCtxGetId", &f1, 12000, cudaEnableDefault, &q1);
    if (e != cudaSuccess) return cuda_fail(e, "static scratch: driver entry points");
    if (q0 != cudaDriverEntryPointSuccess || q1 != cudaDriverEntryPointSuccess || !f0 || !f1)
      return fail(SV_ERR_CUDA, "static scratch: cuCtxGetCurrent / cuCtxGetId not available");
    g_ctx_current = reinterpret_cast<CtxGetCurrentFn>(f0);
    g_ctx_id = reinterpret_cast<CtxGetIdFn>(f1);
  }
  CUcontext ctx = nullptr;
  if (g_ctx_current(&ctx) != CUDA_SUCCESS || !ctx)
    return fail(SV_ERR_CUDA, "static scratch: no current CUDA context");
  if (g_ctx_id(ctx, id) != CUDA_SUCCESS) return fail(SV_ERR_CUDA, "static scratch: cuCtxGetId");
  return SV_OK;
}

// Device address of g_static_scratch in the current context.  The first call
// in each context makes the runtime current on it, looks the symbol up and
// clears the array (synchronously, before returning); later calls in that
// context only read the cached address.
sv_status static_scratch(void **out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);   // also initializes the runtime's context
  if (e != cudaSuccess) return cuda_fail(e, "static scratch: cudaGetDevice");
  e = cudaFree(nullptr);                 // binds the primary context if none is current
  if (e != cudaSuccess) return cuda_fail(e, "static scratch: context setup");
  std::lock_guard<std::mutex> lock(g_static_mu);
  unsigned long long id = 0;
  sv_status st = current_context_id(&id);
  if (st != SV_OK) return st;
  for (int k = 0; k < g_static_used; ++k)
    if (g_static_tab[k].ctx_id == id) {
      *out = g_static_tab[k].ptr;
      return SV_OK;
    }
  void *p = nullptr;
  e = cudaGetSymbolAddress(&p, g_static_scratch);
  if (e != cudaSuccess) return cuda_fail(e, "static scratch: cudaGetSymbolAddress");
  e = cudaMemset(p, 0, SV_STATIC_SCRATCH_BYTES);
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return cuda_fail(e, "static scratch: clearing");
  // a full table drops its oldest entry (a context that long ago went away)
  const int slot = g_static_used < kStaticCtxCap ? g_static_used++ : g_static_next;
  if (slot == g_static_next) g_static_next = (g_static_next + 1) % kStaticCtxCap;
  g_static_tab[slot] = StaticEntry{id, p};
  *out = p;
  return SV_OK;
}

}  // namespace

extern "C" {

SV_API size_t sv_workspace_bytes(const sv_attn_args *attn, const sv_sample_args *sample) {
  if (!attn && !sample) return 0;
  if (attn && check_attn(attn) != SV_OK) return 0;
  if (sample && check_sample(sample) != SV_OK) return 0;
  const size_t t = layout(attn, sample).total;
  return t > 0 ? t : kAlign;
}

SV_API sv_status sv_workspace_init(void *ws, size_t ws_bytes, void *stream) {
  if (!ws || ws_bytes == 0) return fail(SV_ERR_WORKSPACE, "workspace_init: empty workspace");
  cudaError_t e = cudaMemsetAsync(ws, 0, ws_bytes, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "workspace_init");
  return SV_OK;
}

SV_API sv_status spec_verify_attn(const sv_attn_args *attn, void *ws, size_t ws_bytes,
                                  void *stream) {
  sv_status st = check_attn(attn);
  if (st != SV_OK) return st;
  const Layout L = layout(attn, nullptr);
  if ((st = check_ws(ws, ws_bytes, L.total)) != SV_OK) return st;
  return run_attention(attn, L, ws, opts_alone(), static_cast<cudaStream_t>(stream));
}

SV_API sv_status spec_verify_attn_static(const sv_attn_args *attn, void *stream) {
  sv_status st = check_attn(attn);
  if (st != SV_OK) return st;
  // The merge counters keep a fixed zone at the front of the array that no call
  // uses for anything else: the workspace layout puts partials right after the
  // counters of *this* call's shape, so without the zone a smaller earlier
  // call's partials would sit where a larger later call expects zeroed counters.
  Layout L = layout(attn, nullptr);
  const size_t counters = L.part_o - L.cnt_attn;
  if (counters > kStaticCounterBytes)
    return fail(SV_ERR_WORKSPACE,
                "spec_verify_attn_static: %zu bytes of merge counters (batch x kv heads x 4), "
                "the static array reserves %zu",
                counters, kStaticCounterBytes);
  L.part_o += kStaticCounterBytes;
  L.part_ml += kStaticCounterBytes;
  L.pre_o += kStaticCounterBytes;
  L.pre_ml += kStaticCounterBytes;
  L.total += kStaticCounterBytes;
  if (L.total > SV_STATIC_SCRATCH_BYTES)
    return fail(SV_ERR_WORKSPACE,
                "spec_verify_attn_static: needs %zu bytes of scratch, the static array holds %zu "
                "(use spec_verify_attn with a workspace)",
                L.total, static_cast<size_t>(SV_STATIC_SCRATCH_BYTES));
  void *ws = nullptr;
  if ((st = static_scratch(&ws)) != SV_OK) return st;
  return run_attention(attn, L, ws, opts_alone(), static_cast<cudaStream_t>(stream));
}

SV_API sv_status sv_static_scratch_reset(void *stream) {
  void *ws = nullptr;
  sv_status st = static_scratch(&ws);
  if (st != SV_OK) return st;
  cudaError_t e = cudaMemsetAsync(ws, 0, kStaticCounterBytes, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "static scratch reset");
  return SV_OK;
}

SV_API sv_status spec_reject_sample(const sv_sample_args *sample, void *ws, size_t ws_bytes,
                                    void *stream) {
  sv_status st = check_sample(sample);
  if (st != SV_OK) return st;
  const Layout L = layout(nullptr, sample);
  if ((st = check_ws(ws, ws_bytes, L.total)) != SV_OK) return st;
  if (sample->batch == 0) return SV_OK;
  sv::SamplerLaunch SL = sampler_launch(sample, L, ws);
  SL.do_append = false;
  SL.pdl_secondary = false;
  cudaError_t e = sv::launch_sampler(SL, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "sampler launch");
  return SV_OK;
}

SV_API size_t sv_draft_workspace_bytes(const sv_draft_args *draft) {
  if (check_draft(draft) != SV_OK) return 0;
  const sv_sample_args s = draft_as_sample(draft);
  const size_t t = layout(nullptr, &s).total + round_up(static_cast<size_t>(draft->batch) * 4);
  return t > 0 ? t : kAlign;
}

SV_API sv_status spec_draft_sample(const sv_draft_args *draft, void *ws, size_t ws_bytes,
                                   void *stream) {
  sv_status st = check_draft(draft);
  if (st != SV_OK) return st;
  const sv_sample_args s = draft_as_sample(draft);
  const Layout L = layout(nullptr, &s);
  const size_t acc = L.total;     // [B] scratch for the (always 0) accepted counts
  if ((st = check_ws(ws, ws_bytes, acc + round_up(static_cast<size_t>(draft->batch) * 4))) !=
      SV_OK)
    return st;
  if (draft->batch == 0) return SV_OK;
  sv::SamplerLaunch SL = sampler_launch(&s, L, ws);
  SL.a.num_accepted = at<int32_t>(ws, acc);
  SL.do_append = false;
  SL.pdl_secondary = false;
  SL.philox_stream = 1;
  cudaError_t e = sv::launch_sampler(SL, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "draft sampler launch");
  return SV_OK;
}

SV_API size_t sv_draft_step_workspace_bytes(const sv_attn_args *attn, const sv_draft_args *draft) {
  if (!attn || check_attn(attn) != SV_OK || check_draft(draft) != SV_OK) return 0;
  const sv_sample_args s = draft_as_sample(draft);
  const size_t t = layout(attn, &s).total + round_up(static_cast<size_t>(draft->batch) * 4);
  return t > 0 ? t : kAlign;
}

SV_API sv_status spec_draft_step(const sv_attn_args *attn, const sv_draft_args *draft,
                                 const int32_t *kv_cap, int32_t *new_kv_len, void *ws,
                                 size_t ws_bytes, void *stream) {
  sv_status st = check_attn(attn);
  if (st != SV_OK) return st;
  if ((st = check_draft(draft)) != SV_OK) return st;
  if (attn->batch != draft->batch || attn->num_rows != attn->batch || attn->max_q_rows != 1 ||
      attn->kv_len != draft->kv_len || attn->dtype != draft->dtype)
    return fail(SV_ERR_INVALID,
                "draft step: the attention must have one block row per sequence (cu_q = 0..B, "
                "max_q_rows 1) and share kv_len and dtype with the draw");
  if (attn->batch > 0) {
    if (!kv_cap || !new_kv_len) return fail(SV_ERR_INVALID, "draft step: null kv_cap / new_kv_len");
    if (new_kv_len == attn->kv_len)
      return fail(SV_ERR_INVALID, "draft step: new_kv_len aliases kv_len");
    if (!attn->k_cache || !attn->v_cache) return fail(SV_ERR_INVALID, "draft step: null cache");
  }
  const sv_sample_args sa = draft_as_sample(draft);
  const Layout L = layout(attn, &sa);
  const size_t acc = L.total;     // [B] scratch for the (always 0) accepted counts
  if ((st = check_ws(ws, ws_bytes, acc + round_up(static_cast<size_t>(draft->batch) * 4))) != SV_OK)
    return st;
  if (attn->batch == 0) return SV_OK;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  // The position's attention launches first; the draw (Philox stream 1) and the
  // append of the position's own K/V row start beside it as its programmatic
  // dependent launch: neither reads the attention's output, and the append
  // writes only the pool row at kv_len[i], which the attention does not read.
  sv::SamplerLaunch SL = sampler_launch(&sa, L, ws);
  SL.a.num_accepted = at<int32_t>(ws, acc);
  SL.do_append = true;
  SL.pdl_secondary = true;
  SL.philox_stream = 1;
  const int esz = attn->kv_dtype == SV_E4M3 ? 1 : attn->dtype == SV_F32 ? 4 : 2;
  SL.app.k_new = attn->k_new;
  SL.app.v_new = attn->v_new;
  SL.app.k_cache = const_cast<void *>(attn->k_cache);
  SL.app.v_cache = const_cast<void *>(attn->v_cache);
  SL.app.pool_rows = attn->pool_rows;
  SL.app.kv_start = attn->kv_start;
  SL.app.kv_cap = kv_cap;
  SL.app.new_kv_len = new_kv_len;
  SL.app.row_bytes = attn->num_kv_heads * attn->head_dim * esz;
  if (SL.app.row_bytes % 16)
    return fail(SV_ERR_UNSUPPORTED, "draft step: K/V row bytes not a multiple of 16");
  if ((st = run_attention(attn, L, ws, opts_step(L.splan), s)) != SV_OK) return st;
  cudaError_t e = sv::launch_sampler(SL, s);
  if (e != cudaSuccess) return cuda_fail(e, "draft sampler launch");
  return SV_OK;
}

SV_API sv_status kv_append_ragged(int32_t batch, int32_t num_kv_heads, int32_t head_dim,
                                  int32_t dtype, int32_t max_q_rows, int64_t num_rows,
                                  const int32_t *cu_q, const void *k_new, const void *v_new,
                                  void *k_cache, void *v_cache, int64_t pool_rows,
                                  const int64_t *kv_start, const int32_t *kv_len,
                                  const int32_t *kv_cap, const int32_t *num_accepted,
                                  int32_t *new_kv_len, uint32_t *dev_status, void *stream) {
  if (batch < 0) return fail(SV_ERR_INVALID, "append: batch %d", batch);
  if (num_kv_heads < 1 || head_dim < 1 || (dtype != SV_F32 && dtype != SV_BF16 && dtype != SV_E4M3))
    return fail(SV_ERR_INVALID, "append: bad shape or dtype");
  const int esz = dtype == SV_F32 ? 4 : dtype == SV_E4M3 ? 1 : 2;
  const int64_t row_bytes = static_cast<int64_t>(num_kv_heads) * head_dim * esz;
  if (row_bytes % 16 || row_bytes > (1 << 30))
    return fail(SV_ERR_UNSUPPORTED, "append: row bytes %lld not a multiple of 16",
                static_cast<long long>(row_bytes));
  if (max_q_rows < 1 || max_q_rows > sv::kMaxQRows)
    return fail(SV_ERR_INVALID, "append: max_q_rows %d", max_q_rows);
  if (num_rows < batch || num_rows > static_cast<int64_t>(batch) * max_q_rows || pool_rows < 0)
    return fail(SV_ERR_INVALID, "append: num_rows / pool_rows");
  if (batch == 0) return SV_OK;
  if (!cu_q || !k_new || !v_new || !k_cache || !v_cache || !kv_start || !kv_len || !kv_cap ||
      !num_accepted || !new_kv_len)
    return fail(SV_ERR_INVALID, "append: null device pointer");
  if (new_kv_len == kv_len) return fail(SV_ERR_INVALID, "append: new_kv_len aliases kv_len");
  if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(k_cache) || !aligned16(v_cache))
    return fail(SV_ERR_INVALID, "append: tensors must be 16-byte aligned");
  cudaError_t e = sv::launch_append(batch, static_cast<int32_t>(row_bytes), max_q_rows, num_rows,
                                    cu_q, k_new, v_new, k_cache, v_cache, pool_rows, kv_start,
                                    kv_len, kv_cap, num_accepted, new_kv_len, dev_status,
                                    static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "append launch");
  return SV_OK;
}

SV_API sv_status spec_verify_step(const sv_attn_args *attn, const sv_sample_args *sample,
                                  const int32_t *kv_cap, int32_t *new_kv_len, void *ws,
                                  size_t ws_bytes, void *stream) {
  sv_status st = check_attn(attn);
  if (st != SV_OK) return st;
  if ((st = check_sample(sample)) != SV_OK) return st;
  if (attn->batch != sample->batch || attn->num_rows != sample->num_rows ||
      attn->cu_q != sample->cu_q || attn->kv_len != sample->kv_len ||
      attn->max_q_rows != sample->max_q_rows)
    return fail(SV_ERR_INVALID, "step: attention and sampling describe different batches");
  if (attn->batch > 0) {
    if (!kv_cap || !new_kv_len) return fail(SV_ERR_INVALID, "step: null kv_cap / new_kv_len");
    if (new_kv_len == attn->kv_len) return fail(SV_ERR_INVALID, "step: new_kv_len aliases kv_len");
    if (!attn->k_cache || !attn->v_cache) return fail(SV_ERR_INVALID, "step: null cache");
  }
  const Layout L = layout(attn, sample);
  if ((st = check_ws(ws, ws_bytes, L.total)) != SV_OK) return st;
  if (attn->batch == 0) return SV_OK;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  // The attention launches first and lets the sampling launch (with the append
  // of accepted rows) start at once beside it; the sampling waits for the
  // attention before it exits.  The append writes pool rows at or beyond
  // kv_len[i], which the attention never reads.
  sv::SamplerLaunch SL = sampler_launch(sample, L, ws);
  SL.do_append = true;
  SL.pdl_secondary = true;
  const int esz = attn->kv_dtype == SV_E4M3 ? 1 : attn->dtype == SV_F32 ? 4 : 2;
  SL.app.k_new = attn->k_new;
  SL.app.v_new = attn->v_new;
  SL.app.k_cache = const_cast<void *>(attn->k_cache);
  SL.app.v_cache = const_cast<void *>(attn->v_cache);
  SL.app.pool_rows = attn->pool_rows;
  SL.app.kv_start = attn->kv_start;
  SL.app.kv_cap = kv_cap;
  SL.app.new_kv_len = new_kv_len;
  SL.app.row_bytes = attn->num_kv_heads * attn->head_dim * esz;
  if (SL.app.row_bytes % 16)
    return fail(SV_ERR_UNSUPPORTED, "step: K/V row bytes not a multiple of 16");
  if ((st = run_attention(attn, L, ws, opts_step(L.splan), s)) != SV_OK) return st;
  cudaError_t e = sv::launch_sampler(SL, s);
  if (e != cudaSuccess) return cuda_fail(e, "sampler launch");
  return SV_OK;
}

SV_API sv_status sv_set_wait_limit(uint32_t polls) {
  g_wait_limit.store(polls, std::memory_order_relaxed);
  return SV_OK;
}

SV_API const char *sv_last_error(void) { return g_err.c_str(); }

SV_API int32_t sv_abi_version(void) { return SV_ABI_VERSION; }

SV_API size_t sv_struct_size(int32_t which) {
  return which == 0 ? sizeof(sv_attn_args) : which == 1 ? sizeof(sv_sample_args)
         : which == 2 ? sizeof(sv_draft_args) : 0;
}

}  // extern "C"

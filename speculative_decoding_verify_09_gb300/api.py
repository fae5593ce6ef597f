"""Torch-facing calls of the verify step: same names as the C ABI.

Each function only collects data pointers of CUDA tensors and the current
torch stream and calls libspecverify.so; the tensors must stay alive until the
stream has run the call (the argument structs keep references to them).
"""
import ctypes

import torch

from ._binding import (AttnArgs, DraftArgs, SampleArgs, SV_BF16, SV_E4M3, SV_F32, _check, lib)


def _ptr(t):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("tensor must live on a CUDA device")
    if not t.is_contiguous():
        raise ValueError("tensor must be contiguous")
    return t.data_ptr()


def _dt(t):
    if t.dtype == torch.bfloat16:
        return SV_BF16
    if t.dtype == torch.float32:
        return SV_F32
    if t.dtype == torch.uint8:          # E4M3 codes (an 8-bit KV cache)
        return SV_E4M3
    raise ValueError(f"unsupported dtype {t.dtype} (bfloat16, float32 or uint8 E4M3 codes)")


def _stream(stream):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def attn_args(q, k_new, v_new, k_cache, v_cache, cu_q, kv_start, kv_len, out, *, max_q_rows,
              kv_rows_bound, scale=0.0, dev_status=None, group=None, prefix_start=None,
              prefix_len=None, prefix_rows_bound=0, k_scale=0.0, v_scale=0.0):
    """sv_attn_args for q [R, Hq, D], k_new / v_new [R, Hkv, D], caches
    [P, Hkv, D], cu_q [B+1] int32, kv_start [B] int64, kv_len [B] int32,
    out [R, Hq, D]; max_q_rows / kv_rows_bound are host bounds.  Shared
    prefixes: group [B] int32 (non-decreasing), prefix_start [G] int64,
    prefix_len [G] int32 and the host bound prefix_rows_bound.  uint8 K/V
    tensors are E4M3 codes read as code * k_scale / code * v_scale."""
    a = AttnArgs()
    R, Hq, D = q.shape
    a.batch = cu_q.shape[0] - 1
    a.num_q_heads, a.num_kv_heads, a.head_dim = Hq, k_new.shape[1], D
    a.dtype = _dt(q)
    a.max_q_rows = int(max_q_rows)
    a.num_rows = R
    a.kv_rows_bound = int(kv_rows_bound)
    a.pool_rows = k_cache.shape[0]
    a.scale = float(scale)
    a.num_groups = 0 if group is None else prefix_len.shape[0]
    a.prefix_rows_bound = int(prefix_rows_bound)
    a.cu_q, a.q, a.k_new, a.v_new = _ptr(cu_q), _ptr(q), _ptr(k_new), _ptr(v_new)
    a.k_cache, a.v_cache = _ptr(k_cache), _ptr(v_cache)
    a.kv_start, a.kv_len, a.out = _ptr(kv_start), _ptr(kv_len), _ptr(out)
    a.dev_status = _ptr(dev_status)
    a.kv_dtype = SV_E4M3 if k_cache.dtype == torch.uint8 else 0
    a.k_scale, a.v_scale = float(k_scale), float(v_scale)
    a.group, a.prefix_start, a.prefix_len = _ptr(group), _ptr(prefix_start), _ptr(prefix_len)
    a._keep = (q, k_new, v_new, k_cache, v_cache, cu_q, kv_start, kv_len, out, dev_status,
               group, prefix_start, prefix_len)
    return a


def sample_args(target_logits, draft_logits, draft_tokens, cu_q, kv_len, num_accepted,
                out_tokens, *, max_q_rows, temperature, top_p, seed, seq_ids=None,
                dev_status=None, top_k=0, temperatures=None, top_ps=None, top_ks=None):
    """sv_sample_args for target_logits [R, V], draft_logits [R-B, V],
    draft_tokens [R-B] int32, cu_q [B+1], kv_len [B], outputs num_accepted [B]
    and out_tokens [R] (int32), seq_ids [B] int64 or None.  temperature 0 is
    greedy; top_k 0 disables top-k; temperatures / top_ps ([B] float32) and
    top_ks ([B] int32) override the scalars per sequence."""
    s = SampleArgs()
    R, V = target_logits.shape
    s.batch = cu_q.shape[0] - 1
    s.vocab = V
    s.dtype = _dt(target_logits)
    s.max_q_rows = int(max_q_rows)
    s.num_rows = R
    s.temperature = float(temperature)
    s.top_p = float(top_p)
    s.seed = int(seed) & 0xFFFFFFFFFFFFFFFF
    s.cu_q, s.target_logits = _ptr(cu_q), _ptr(target_logits)
    s.draft_logits = _ptr(draft_logits) if draft_logits.numel() else None
    s.draft_tokens = _ptr(draft_tokens) if draft_tokens.numel() else None
    s.kv_len, s.seq_ids = _ptr(kv_len), _ptr(seq_ids)
    s.num_accepted, s.out_tokens = _ptr(num_accepted), _ptr(out_tokens)
    s.dev_status = _ptr(dev_status)
    s.top_k = int(top_k)
    s.temperatures, s.top_ps, s.top_ks = _ptr(temperatures), _ptr(top_ps), _ptr(top_ks)
    s._keep = (target_logits, draft_logits, draft_tokens, cu_q, kv_len, seq_ids, num_accepted,
               out_tokens, dev_status, temperatures, top_ps, top_ks)
    return s


def draft_args(draft_logits, kv_len, draft_tokens, *, temperature, top_p, seed, seq_ids=None,
               dev_status=None, top_k=0, temperatures=None, top_ps=None, top_ks=None):
    """sv_draft_args for draft_logits [B, V] (one row per sequence), kv_len [B]
    (cache lengths before this position's append: row i's token sits at index
    kv_len[i] + 1), output draft_tokens [B] int32; parameters as in
    sample_args."""
    d = DraftArgs()
    B, V = draft_logits.shape
    d.batch, d.vocab, d.dtype = B, V, _dt(draft_logits)
    d.top_k = int(top_k)
    d.temperature, d.top_p = float(temperature), float(top_p)
    d.seed = int(seed) & 0xFFFFFFFFFFFFFFFF
    d.draft_logits, d.kv_len, d.seq_ids = _ptr(draft_logits), _ptr(kv_len), _ptr(seq_ids)
    d.temperatures, d.top_ps, d.top_ks = _ptr(temperatures), _ptr(top_ps), _ptr(top_ks)
    d.draft_tokens, d.dev_status = _ptr(draft_tokens), _ptr(dev_status)
    d._keep = (draft_logits, kv_len, seq_ids, temperatures, top_ps, top_ks, draft_tokens,
               dev_status)
    return d


def spec_draft_step(attn, draft, kv_cap, new_kv_len, ws, stream=None):
    """One draft position: single-row attention, append of the position's row
    and the draft-token draw, the last two beside the attention."""
    _check(lib.spec_draft_step(ctypes.byref(attn), ctypes.byref(draft), _ptr(kv_cap),
                               _ptr(new_kv_len), ctypes.c_void_p(ws.ptr), ws.nbytes,
                               _stream(stream)))


def draft_step_workspace_bytes(attn, draft):
    n = lib.sv_draft_step_workspace_bytes(ctypes.byref(attn), ctypes.byref(draft))
    if n == 0:
        _check(1)
    return n


def draft_workspace_bytes(draft):
    n = lib.sv_draft_workspace_bytes(ctypes.byref(draft))
    if n == 0:
        _check(1)
    return n


def workspace_bytes(attn=None, sample=None):
    n = lib.sv_workspace_bytes(ctypes.byref(attn) if attn is not None else None,
                               ctypes.byref(sample) if sample is not None else None)
    if n == 0:
        _check(1)
    return n


class Workspace:
    """A device workspace for the verify calls, zeroed once on creation."""

    def __init__(self, nbytes, device=None, stream=None):
        self.nbytes = int(nbytes)
        self.buf = torch.empty(self.nbytes + 256, dtype=torch.uint8, device=device or "cuda")
        base = self.buf.data_ptr()
        self.ptr = (base + 255) // 256 * 256
        _check(lib.sv_workspace_init(ctypes.c_void_p(self.ptr), self.nbytes, _stream(stream)))

    def zero(self, stream=None):
        """Zero the workspace again (after a call that reported SV_DEV_TIMEOUT)."""
        _check(lib.sv_workspace_init(ctypes.c_void_p(self.ptr), self.nbytes, _stream(stream)))

    @classmethod
    def for_args(cls, attn=None, sample=None, device=None, stream=None):
        return cls(workspace_bytes(attn, sample), device, stream)


def spec_verify_attn(attn, ws, stream=None):
    _check(lib.spec_verify_attn(ctypes.byref(attn), ctypes.c_void_p(ws.ptr), ws.nbytes,
                                _stream(stream)))


def spec_verify_attn_static(attn, stream=None):
    """spec_verify_attn with the library's static device scratch instead of a
    workspace, for callers that may not allocate device memory; nothing is
    allocated (the first call on a device sets the scratch up)."""
    _check(lib.spec_verify_attn_static(ctypes.byref(attn), _stream(stream)))


def sv_static_scratch_reset(stream=None):
    """Zero the static scratch's merge counters on `stream` (after a static call
    reported SV_DEV_TIMEOUT); allocates nothing."""
    _check(lib.sv_static_scratch_reset(_stream(stream)))


def sv_set_wait_limit(polls):
    """Bound on the polls of one attention pipeline wait (0: the built-in
    bound); a small bound makes waits run out on purpose (SV_DEV_TIMEOUT)."""
    _check(lib.sv_set_wait_limit(int(polls)))


def spec_reject_sample(sample, ws, stream=None):
    _check(lib.spec_reject_sample(ctypes.byref(sample), ctypes.c_void_p(ws.ptr), ws.nbytes,
                                  _stream(stream)))


def spec_draft_sample(draft, ws, stream=None):
    _check(lib.spec_draft_sample(ctypes.byref(draft), ctypes.c_void_p(ws.ptr), ws.nbytes,
                                 _stream(stream)))


def kv_append_ragged(cu_q, k_new, v_new, k_cache, v_cache, kv_start, kv_len, kv_cap,
                     num_accepted, new_kv_len, *, max_q_rows, dev_status=None, stream=None):
    B = cu_q.shape[0] - 1
    R, Hkv, D = k_new.shape
    _check(lib.kv_append_ragged(B, Hkv, D, _dt(k_new), int(max_q_rows), R, _ptr(cu_q),
                                _ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache),
                                k_cache.shape[0], _ptr(kv_start), _ptr(kv_len), _ptr(kv_cap),
                                _ptr(num_accepted), _ptr(new_kv_len), _ptr(dev_status),
                                _stream(stream)))


def spec_verify_step(attn, sample, kv_cap, new_kv_len, ws, stream=None):
    _check(lib.spec_verify_step(ctypes.byref(attn), ctypes.byref(sample), _ptr(kv_cap),
                                _ptr(new_kv_len), ctypes.c_void_p(ws.ptr), ws.nbytes,
                                _stream(stream)))

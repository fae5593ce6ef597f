"""Device buffers for one verify step, built from host arrays.

Convenience for callers that hold a step's inputs as numpy arrays (bfloat16
as uint16 bit patterns): copies them to the current CUDA device, allocates
the outputs and a workspace, and fills the C-ABI argument structs.
"""
import numpy as np
import torch


def dev(x, dtype=None):
    """numpy -> CUDA tensor; uint16 arrays are bfloat16 bit patterns."""
    if x.dtype == np.uint16:
        return torch.from_numpy(x.view(np.int16)).cuda().view(torch.bfloat16)
    t = torch.from_numpy(np.ascontiguousarray(x)).cuda()
    return t if dtype is None else t.to(dtype)


def host_bits(t):
    """CUDA tensor -> numpy (bfloat16 as uint16 bits)."""
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).cpu().numpy().view(np.uint16)
    return t.cpu().numpy()


def to_f32(t):
    return t.float().cpu().numpy()


class StepBuffers:
    """Device copies of one step's inputs (a dict of host arrays, bf16 as
    uint16 bits), its output tensors, the C-ABI argument structs and a
    workspace.  The KV pool copies are the live caches the step appends to."""

    def __init__(self, inp, api, seed=None):
        self.inp = inp
        self.api = api
        R = int(inp["cu_q"][-1])
        B = inp["B"]
        K = np.diff(inp["cu_q"]) - 1
        self.max_q_rows = int(K.max()) + 1 if B else 1
        self.cu_q = dev(inp["cu_q"])
        self.kv_start = dev(inp["kv_start"])
        self.kv_len = dev(inp["kv_len"])
        self.kv_cap = dev(inp["kv_cap"])
        self.seq_ids = dev(inp["seq_ids"])
        self.status = torch.zeros(1, dtype=torch.int32, device="cuda")
        self.num_accepted = torch.full((B,), -7, dtype=torch.int32, device="cuda")
        self.out_tokens = torch.full((R,), -7, dtype=torch.int32, device="cuda")
        self.new_kv_len = torch.full((B,), -7, dtype=torch.int32, device="cuda")
        if "q" in inp:
            self.q, self.k_new, self.v_new = dev(inp["q"]), dev(inp["k_new"]), dev(inp["v_new"])
            self.k_cache, self.v_cache = dev(inp["k_cache"]), dev(inp["v_cache"])
            self.out = torch.full_like(self.q, float("nan"))
            pre = {}
            if inp.get("group") is not None:
                self.group = dev(inp["group"])
                self.prefix_start = dev(inp["prefix_start"])
                self.prefix_len = dev(inp["prefix_len"])
                pre = dict(group=self.group, prefix_start=self.prefix_start,
                           prefix_len=self.prefix_len,
                           prefix_rows_bound=int(np.sum(inp["prefix_len"])))
            self.attn = api.attn_args(self.q, self.k_new, self.v_new, self.k_cache, self.v_cache,
                                      self.cu_q, self.kv_start, self.kv_len, self.out,
                                      max_q_rows=self.max_q_rows,
                                      kv_rows_bound=int(np.sum(inp["kv_len"])),
                                      scale=inp.get("scale") or 0.0, dev_status=self.status,
                                      k_scale=inp.get("k_scale", 0.0),
                                      v_scale=inp.get("v_scale", 0.0), **pre)
        else:
            self.attn = None
        if "target_logits" in inp:
            self.tgt, self.drf = dev(inp["target_logits"]), dev(inp["draft_logits"])
            self.drafts = dev(inp["draft_tokens"])
            per = {k: dev(np.asarray(inp[k])) for k in ("temperatures", "top_ps", "top_ks")
                   if inp.get(k) is not None}
            self.per_seq = per
            self.sample = api.sample_args(self.tgt, self.drf, self.drafts, self.cu_q, self.kv_len,
                                          self.num_accepted, self.out_tokens,
                                          max_q_rows=self.max_q_rows,
                                          temperature=inp["temperature"], top_p=inp["top_p"],
                                          seed=inp["seed"] if seed is None else seed,
                                          seq_ids=self.seq_ids, dev_status=self.status,
                                          top_k=inp.get("top_k", 0), **per)
        else:
            self.sample = None
        self.ws = api.Workspace.for_args(self.attn, self.sample)

    def status_bits(self):
        return int(self.status.item()) & 0xFFFFFFFF


def _torch_dtype(a):
    return {np.dtype(np.uint16): torch.bfloat16, np.dtype(np.float32): torch.float32,
            np.dtype(np.int32): torch.int32, np.dtype(np.int64): torch.int64}[a.dtype]


class StagedStep:
    """A step's per-step inputs and outputs in two contiguous device arenas,
    each with a pinned host mirror, so that a step is one host-to-device copy,
    the fused call and one device-to-host copy.  The KV pools, the workspace and
    the argument structs are those of `base` (a StepBuffers), which stay
    resident on the device.

    Inputs: q, k_new, v_new, target / draft logits, draft tokens, cu_q, kv_len,
    kv_start, kv_cap, seq_ids.  Outputs: out, num_accepted, out_tokens,
    new_kv_len.  Write a step's inputs with `pack` (or into `host_in` views),
    then `upload`, run the step on `base`'s structs, `download`."""

    IN = ("q", "k_new", "v_new", "target_logits", "draft_logits", "draft_tokens", "cu_q",
          "kv_len", "kv_start", "kv_cap", "seq_ids")
    OUT = ("out", "num_accepted", "out_tokens", "new_kv_len")

    def __init__(self, base):
        self.base = base
        ins = {"q": base.q, "k_new": base.k_new, "v_new": base.v_new,
               "target_logits": base.tgt, "draft_logits": base.drf,
               "draft_tokens": base.drafts, "cu_q": base.cu_q, "kv_len": base.kv_len,
               "kv_start": base.kv_start, "kv_cap": base.kv_cap, "seq_ids": base.seq_ids}
        outs = {"out": base.out, "num_accepted": base.num_accepted,
                "out_tokens": base.out_tokens, "new_kv_len": base.new_kv_len}
        self.in_bytes, self.host_in, self.dev_in, self._in = self._arena(ins)
        self.out_bytes, self.host_out, self.dev_out, self._out = self._arena(outs)
        # the step's structs point into the device arenas from now on
        for name, t in self._in[1].items():
            setattr(base, {"target_logits": "tgt", "draft_logits": "drf",
                           "draft_tokens": "drafts"}.get(name, name), t)
        for name, t in self._out[1].items():
            setattr(base, name, t)
        self._rebind()

    @staticmethod
    def _arena(tensors):
        offs, off = {}, 0
        for name, t in tensors.items():
            offs[name] = off
            off += (t.numel() * t.element_size() + 255) // 256 * 256
        host = torch.empty(off, dtype=torch.uint8).pin_memory()
        devb = torch.empty(off, dtype=torch.uint8, device="cuda")
        hv, dv = {}, {}
        for name, t in tensors.items():
            n = t.numel() * t.element_size()
            hv[name] = host[offs[name]:offs[name] + n].view(t.dtype).view(t.shape)
            dv[name] = devb[offs[name]:offs[name] + n].view(t.dtype).view(t.shape)
            dv[name].copy_(t)
        return off, host, devb, (hv, dv)

    def _rebind(self):
        b, api = self.base, self.base.api
        pre = {}
        if getattr(b, "group", None) is not None:
            pre = dict(group=b.group, prefix_start=b.prefix_start, prefix_len=b.prefix_len,
                       prefix_rows_bound=b.attn.prefix_rows_bound)
        self.attn = b.attn = api.attn_args(
            b.q, b.k_new, b.v_new, b.k_cache, b.v_cache, b.cu_q, b.kv_start, b.kv_len, b.out,
            max_q_rows=b.attn.max_q_rows, kv_rows_bound=b.attn.kv_rows_bound,
            scale=b.attn.scale, dev_status=b.status, k_scale=b.attn.k_scale,
            v_scale=b.attn.v_scale, **pre)
        s = b.sample
        self.sample = b.sample = api.sample_args(
            b.tgt, b.drf, b.drafts, b.cu_q, b.kv_len, b.num_accepted, b.out_tokens,
            max_q_rows=s.max_q_rows, temperature=s.temperature, top_p=s.top_p, seed=s.seed,
            seq_ids=b.seq_ids, dev_status=b.status, top_k=s.top_k,
            **getattr(b, "per_seq", {}))

    def pack(self, inp):
        """Write a host input dict (bf16 as uint16 bits) into the pinned arena."""
        hv = self._in[0]
        for name in self.IN:
            a = np.ascontiguousarray(inp[name])
            if a.dtype == np.uint16:
                a = a.view(np.int16)
            hv[name].view(torch.int16 if hv[name].dtype == torch.bfloat16 else hv[name].dtype) \
                .copy_(torch.from_numpy(a).view(hv[name].shape))

    def upload(self):
        self.dev_in.copy_(self.host_in, non_blocking=True)

    def download(self):
        self.host_out.copy_(self.dev_out, non_blocking=True)

    def result(self, name):
        return self._out[0][name]


def _arena(specs):
    """One device buffer and a pinned host mirror holding tensors of the given
    (name, shape, torch dtype), each at a 256-byte aligned offset.  Returns
    (bytes, device buffer, host buffer, device views, host views)."""
    offs, off = {}, 0
    for name, shape, dt in specs:
        n = int(np.prod(shape)) * torch.empty(0, dtype=dt).element_size()
        offs[name] = (off, n)
        off += (n + 255) // 256 * 256
    devb = torch.empty(max(off, 256), dtype=torch.uint8, device="cuda")
    host = torch.empty(max(off, 256), dtype=torch.uint8).pin_memory()
    dv, hv = {}, {}
    for name, shape, dt in specs:
        o, n = offs[name]
        dv[name] = devb[o:o + n].view(dt).view(shape)
        hv[name] = host[o:o + n].view(dt).view(shape)
    return off, devb, host, dv, hv


def _put(t, a):
    """Copy host array `a` (bf16 as uint16 bits) into tensor `t`."""
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        t.view(torch.int16).copy_(torch.from_numpy(a.view(np.int16)).view(t.shape))
    else:
        t.copy_(torch.from_numpy(a).view(t.shape))


class DraftBuffers:
    """Device state for `positions` consecutive draft positions of a batch:
    the draft model's single-row attention (spec_verify_attn with cu_q =
    0..B), the append of that row (kv_append_ragged with num_accepted all 0)
    and the draft-token draw (spec_draft_sample).  `base` is position 0's host
    input dict (bf16 as uint16 bits); `steps` holds every position's q,
    k_new, v_new and draft_logits (default: base's for all).

    Per-position inputs (q, k_new, v_new, draft_logits) sit in one device
    arena and the outputs (out, tokens, the lengths each position writes) in
    another, each with a pinned host mirror (`upload` / `download` copy them
    whole).  Position t reads kv_lens[t] and writes kv_lens[t + 1]; kv_lens[0]
    holds the starting lengths and is never written, so `rewind` restarts the
    chain and nothing but the library's kernels runs between positions.  The
    KV pool copies are the live caches the positions append to."""

    def __init__(self, base, api, seed=None, positions=1, steps=None):
        self.api = api
        B, P = base["B"], int(positions)
        self.B, self.positions = B, P
        steps = steps if steps is not None else [base] * P
        dt = torch.bfloat16 if base["q"].dtype == np.uint16 else torch.float32
        kvdt = torch.uint8 if base["k_new"].dtype == np.uint8 else dt      # E4M3 codes
        Hq, Hkv, D, V = base["num_q_heads"], base["num_kv_heads"], base["head_dim"], base["V"]
        self.in_bytes, self.dev_in, self.host_in, self.inputs, self.host_inputs = _arena([
            ("q", (P, B, Hq, D), dt), ("k_new", (P, B, Hkv, D), kvdt),
            ("v_new", (P, B, Hkv, D), kvdt), ("draft_logits", (P, B, V), dt)])
        self.out_bytes, self.dev_out, self.host_out, self.outputs, self.host_outputs = _arena([
            ("out", (P, B, Hq, D), dt), ("tokens", (P, B), torch.int32),
            ("new_len", (P, B), torch.int32)])
        for t, st in enumerate(steps[:P]):
            for name in ("q", "k_new", "v_new", "draft_logits"):
                _put(self.inputs[name][t], st[name])
        self.outputs["out"].fill_(float("nan"))
        self.outputs["tokens"].fill_(-7)
        self.outputs["new_len"].fill_(-7)
        self.q, self.k_new, self.v_new = (self.inputs[k] for k in ("q", "k_new", "v_new"))
        self.logits = self.inputs["draft_logits"]
        self.out, self.tokens = self.outputs["out"], self.outputs["tokens"]
        self.cu_q = dev(np.arange(B + 1, dtype=np.int32))
        self.kv_start = dev(base["kv_start"])
        self.kv_lens = [dev(base["kv_len"])] + [self.outputs["new_len"][t] for t in range(P)]
        self.kv_cap = dev(base["kv_cap"])
        self.seq_ids = dev(base["seq_ids"])
        self.zeros = torch.zeros(B, dtype=torch.int32, device="cuda")
        self.status = torch.zeros(1, dtype=torch.int32, device="cuda")
        self.k_cache, self.v_cache = dev(base["k_cache"]), dev(base["v_cache"])
        self.per_seq = {k: dev(np.asarray(base[k])) for k in ("temperatures", "top_ps", "top_ks")
                        if base.get(k) is not None}
        self.rows_bound = int(np.sum(base["kv_cap"]))      # no length grows past its cap
        self.attn, self.draft = [], []
        for t in range(P):
            kv = self.kv_lens[t]
            self.attn.append(api.attn_args(
                self.q[t], self.k_new[t], self.v_new[t], self.k_cache, self.v_cache, self.cu_q,
                self.kv_start, kv, self.out[t], max_q_rows=1, kv_rows_bound=self.rows_bound,
                scale=base.get("scale") or 0.0, dev_status=self.status,
                k_scale=base.get("k_scale", 0.0), v_scale=base.get("v_scale", 0.0)))
            self.draft.append(api.draft_args(
                self.logits[t], kv, self.tokens[t], temperature=base["temperature"],
                top_p=base["top_p"], seed=base["seed"] if seed is None else seed,
                seq_ids=self.seq_ids, dev_status=self.status, top_k=base.get("top_k", 0),
                **self.per_seq))
        self.ws_attn = api.Workspace.for_args(self.attn[0])
        self.ws_draft = api.Workspace(api.draft_workspace_bytes(self.draft[0]))
        self.ws_step = api.Workspace(api.draft_step_workspace_bytes(self.attn[0], self.draft[0]))
        self.cur = 0

    @property
    def kv_len(self):
        """The cache lengths the next position starts from."""
        return self.kv_lens[self.cur]

    def rewind(self):
        self.cur = 0

    def stage(self, steps):
        """Write every position's inputs into the pinned host arena."""
        for t, st in enumerate(steps[:self.positions]):
            for name in ("q", "k_new", "v_new", "draft_logits"):
                _put(self.host_inputs[name][t], st[name])

    def upload(self):
        self.dev_in.copy_(self.host_in, non_blocking=True)

    def download(self):
        self.host_out.copy_(self.dev_out, non_blocking=True)

    def run(self, stream=None):
        """The next draft position on the current stream: attention, append,
        draw."""
        c = self.cur
        if c >= self.positions:
            raise IndexError(f"all {self.positions} draft positions have run; rewind first")
        api = self.api
        api.spec_verify_attn(self.attn[c], self.ws_attn, stream)
        api.kv_append_ragged(self.cu_q, self.k_new[c], self.v_new[c], self.k_cache, self.v_cache,
                             self.kv_start, self.kv_lens[c], self.kv_cap, self.zeros,
                             self.kv_lens[c + 1], max_q_rows=1, dev_status=self.status,
                             stream=stream)
        api.spec_draft_sample(self.draft[c], self.ws_draft, stream)
        self.cur = c + 1

    def run_fused(self, stream=None):
        """The next draft position as one call (spec_draft_step): the draw and
        the append start beside the attention."""
        c = self.cur
        if c >= self.positions:
            raise IndexError(f"all {self.positions} draft positions have run; rewind first")
        self.api.spec_draft_step(self.attn[c], self.draft[c], self.kv_cap, self.kv_lens[c + 1],
                                 self.ws_step, stream)
        self.cur = c + 1

    def run_all(self, stream=None, fused=False):
        """Every position from the starting lengths (one draft-side step), as
        three calls per position or (fused) one."""
        self.rewind()
        for _ in range(self.positions):
            self.run_fused(stream) if fused else self.run(stream)

    def status_bits(self):
        return int(self.status.item()) & 0xFFFFFFFF

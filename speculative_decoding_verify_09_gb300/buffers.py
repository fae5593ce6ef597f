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
                                      **pre)
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
            scale=b.attn.scale, dev_status=b.status, **pre)
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

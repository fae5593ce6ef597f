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
            self.sample = api.sample_args(self.tgt, self.drf, self.drafts, self.cu_q, self.kv_len,
                                          self.num_accepted, self.out_tokens,
                                          max_q_rows=self.max_q_rows,
                                          temperature=inp["temperature"], top_p=inp["top_p"],
                                          seed=inp["seed"] if seed is None else seed,
                                          seq_ids=self.seq_ids, dev_status=self.status)
        else:
            self.sample = None
        self.ws = api.Workspace.for_args(self.attn, self.sample)

    def status_bits(self):
        return int(self.status.item()) & 0xFFFFFFFF

"""Helpers for the GPU tests: move workload inputs to the device, run the
C-ABI calls through the binding, compare with the oracle under the near-tie
rules.  Imports the oracle only to compute expected values."""
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


class DeviceStep:
    """All device tensors + argument structs for one verify step."""

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
            self.attn = api.attn_args(self.q, self.k_new, self.v_new, self.k_cache, self.v_cache,
                                      self.cu_q, self.kv_start, self.kv_len, self.out,
                                      max_q_rows=self.max_q_rows,
                                      kv_rows_bound=int(np.sum(inp["kv_len"])),
                                      scale=inp.get("scale") or 0.0, dev_status=self.status)
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


def compare_sampling(ref, num_accepted, out_tokens, cu_q):
    """Bit-exact comparison outside the oracle's near-tie windows.

    Returns (n_checked_sequences, n_tie_sequences).  Raises AssertionError with
    details on a mismatch."""
    B = len(cu_q) - 1
    ties = 0
    for i in range(B):
        r0, r1 = int(cu_q[i]), int(cu_q[i + 1])
        n_ref, n_gpu = int(ref["num_accepted"][i]), int(num_accepted[i])
        kind, row = int(ref["tie_kind"][i]), int(ref["tie_row"][i])
        if kind == 0:
            assert n_gpu == n_ref, f"seq {i}: num_accepted {n_gpu} != {n_ref}"
            assert list(out_tokens[r0:r1]) == list(ref["out_tokens"][r0:r1]), \
                f"seq {i}: tokens {list(out_tokens[r0:r1])} != {list(ref['out_tokens'][r0:r1])}"
            continue
        ties += 1
        if kind == 1:     # accept-level tie at `row`: rows before it still exact
            assert n_gpu >= row, f"seq {i}: gpu rejected at {n_gpu} before the tie row {row}"
            assert list(out_tokens[r0:r0 + row]) == list(ref["out_tokens"][r0:r0 + row])
        else:             # draw-level tie: n and accepted drafts exact, token a neighbour
            assert n_gpu == n_ref, f"seq {i}: num_accepted {n_gpu} != {n_ref} (draw tie)"
            assert list(out_tokens[r0:r0 + n_ref]) == list(ref["out_tokens"][r0:r0 + n_ref])
            alts = ref["tie_alts"].get(i)
            tok = int(out_tokens[r0 + n_ref])
            if alts is not None:
                assert tok in alts, f"seq {i}: drawn {tok} not in tie set {alts}"
            assert list(out_tokens[r0 + n_ref + 1:r1]) == [-1] * (r1 - r0 - n_ref - 1)
    return B, ties

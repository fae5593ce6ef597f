"""GPU parity of kv_append_ragged with the oracle (bit-exact pool and
lengths; EMS-SD abstract: per-sample accepted counts, no padding)."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from gpu_util import dev, host_bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def api():
    import speculative_decoding_verify_09_gb300 as pkg
    pkg.build()
    return pkg.load()


@pytest.mark.parametrize("name,kw", [("tiny_f32", {}), ("bass_b8", {}),
                                     ("ragged_gqa_b32", {"B": 40, "L_hi": 600})])
def test_append_matches_oracle(api, name, kw):
    inp = W.make_inputs(W.workload(name, **kw), with_logits=False)
    rng = np.random.default_rng(1)
    K = np.diff(inp["cu_q"]) - 1
    nacc = np.array([rng.integers(0, k + 1) for k in K], dtype=np.int32)
    nacc[0] = -1                                     # failed sequence: no append
    cap = inp["kv_cap"].copy()
    cap[-1] = inp["kv_len"][-1] + nacc[-1]           # one row short: overflow
    kc, vc = dev(inp["k_cache"]), dev(inp["v_cache"])
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    new_len = torch.full((inp["B"],), -5, dtype=torch.int32, device="cuda")
    api.kv_append_ragged(dev(inp["cu_q"]), dev(inp["k_new"]), dev(inp["v_new"]), kc, vc,
                         dev(inp["kv_start"]), dev(inp["kv_len"]), dev(cap), dev(nacc), new_len,
                         max_q_rows=int(K.max()) + 1, dev_status=status)
    torch.cuda.synchronize()
    k2, v2, nl, st = oracle.kv_append(inp["k_cache"], inp["v_cache"], inp["k_new"],
                                      inp["v_new"], inp["cu_q"], inp["kv_start"], inp["kv_len"],
                                      cap, nacc)
    assert np.array_equal(new_len.cpu().numpy(), nl)
    assert np.array_equal(host_bits(kc), k2) and np.array_equal(host_bits(vc), v2)
    assert int(status.item()) == st == oracle.DEV_CAPACITY

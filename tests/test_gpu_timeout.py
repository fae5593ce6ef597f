"""A bounded wait of the attention pipeline that runs out: SV_DEV_TIMEOUT, a
clean return, and a usable context afterwards.

Every wait of the verify attention's copy ring, Q slots, consumer group and
merge hand-off polls an mbarrier a bounded number of times.  sv_set_wait_limit
lowers that bound for later launches; at one poll the first waits run out
while the copies they wait for are still in flight.  The kernel must then set
SV_DEV_TIMEOUT, drain the copies it started and return (the call's stream
synchronizes: nothing hangs); after the bound is restored and the workspace
zeroed again, the same call gives the oracle's outputs with a clean status.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from gpu_util import DeviceStep

pytestmark = pytest.mark.gpu

SV_DEV_TIMEOUT = 32


@pytest.fixture(scope="module")
def api():
    import speculative_decoding_verify_09_gb300 as pkg
    pkg.build()
    return pkg.load()


@pytest.mark.parametrize("name,kw", [
    ("bass_b8", {}),
    ("ragged_gqa_b32", dict(B=12, gen_seed=91)),
])
def test_wait_limit_runs_out_then_recovers(api, name, kw):
    inp = W.make_inputs(W.workload(name, **kw), with_logits=False)
    d = DeviceStep(inp, api)
    seen = False
    try:
        api.sv_set_wait_limit(1)
        for _ in range(3):
            d.status.zero_()
            api.spec_verify_attn(d.attn, d.ws)
            torch.cuda.synchronize()                  # returns: no wait is endless
            if d.status_bits() & SV_DEV_TIMEOUT:
                seen = True
                break
    finally:
        api.sv_set_wait_limit(0)
    assert seen, "a one-poll bound never ran out"
    # merge counters may have been left nonzero: zero the workspace, run again
    d.ws.zero()
    d.status.zero_()
    d.out.fill_(float("nan"))
    api.spec_verify_attn(d.attn, d.ws)
    torch.cuda.synchronize()
    assert d.status_bits() == 0
    got = d.out.float().cpu().numpy()
    ref = oracle.verify_attention(inp["q"], inp["k_new"], inp["v_new"], inp["k_cache"],
                                  inp["v_cache"], inp["cu_q"], inp["kv_start"], inp["kv_len"],
                                  inp["num_kv_heads"])
    assert np.all(np.isfinite(got))
    assert float(np.max(np.abs(got - ref))) < 2e-2

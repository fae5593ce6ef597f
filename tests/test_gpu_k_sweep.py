"""Acceptance efficiency of the CUDA sampler against K on bass_b8's shapes.

For every K the mean number of tokens a verify step emits per sequence must
match the closed form sum_{j=0..K} prod_{t<j} beta_t, beta_t = sum_x
min(p_hat_t(x), q_hat_t(x)) (speculative-sampling paper: Theorem 1's
acceptance, and the section on the trade-off between draft length and scoring
frequency, Figure 1 middle), within 5 standard errors over fresh inputs and
drafts; drafts come from p_hat (workloads.py draws them from softmax(p / T)).
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from gpu_util import DeviceStep
from test_oracle_k_sweep import emitted_moments

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def api():
    import speculative_decoding_verify_09_gb300 as pkg
    pkg.build()
    return pkg.load()


@pytest.mark.parametrize("K", [1, 4, 8])
def test_mean_emitted_matches_closed_form(api, K):
    dev_sum = var_sum = 0.0
    n = 0
    for inst in range(5):
        w = W.workload("bass_b8", B=32, K_lo=K, K_hi=K, gen_seed=1000 + 10 * K + inst,
                       philox_seed=inst)
        inp = W.make_inputs(w, with_attention=False)
        d = DeviceStep(inp, api)
        api.spec_reject_sample(d.sample, d.ws)
        torch.cuda.synchronize()
        assert d.status_bits() == 0
        emitted = d.num_accepted.cpu().numpy() + 1
        cu = inp["cu_q"]
        for i in range(w.B):
            r0, p0 = int(cu[i]), int(cu[i]) - i
            betas = []
            for j in range(K):
                q = oracle.process_row(oracle.to_f64(inp["target_logits"][r0 + j]), 1.0, 1.0).probs
                p = oracle.process_row(oracle.to_f64(inp["draft_logits"][p0 + j]), 1.0, 1.0).probs
                betas.append(float(np.minimum(p, q).sum()))
            mean, var = emitted_moments(betas)
            dev_sum += emitted[i] - mean
            var_sum += var
            n += 1
    z = dev_sum / np.sqrt(var_sum)
    assert abs(z) < 5, (K, dev_sum / n, z)

"""spec_verify_attn_static against spec_verify_attn.

spec_verify_attn_static keeps its split-KV scratch in a static array inside the
library's device image, for callers that may not allocate device memory when
they call (their memory belongs to another allocator, or their runtime forbids
allocation once serving).  Each call here goes through the C ABI and must give
the workspace entry point's output bit for bit (same kernels, same fold order
of the split-KV pieces), and so lies within the attention tolerance (2e-2 for
bf16, 1e-4 for fp32) of it too, on two calls in a row: the second call also
checks that the first left the shared merge counters at zero.  This file sorts
last so that it runs alone or after every other GPU test.
"""
import ctypes

import pytest
import torch

import workloads as W
from gpu_util import DeviceStep

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def api():
    import speculative_decoding_verify_09_gb300 as pkg
    pkg.build()
    return pkg.load()


def _tol(inp):
    return 1e-4 if inp["dtype"] == "f32" else 2e-2


def _reference(api, inp):
    d = DeviceStep(inp, api)
    api.spec_verify_attn(d.attn, d.ws)
    torch.cuda.synchronize()
    assert d.status_bits() == 0
    return d, d.out.float().clone()


def _static_call_matches(api, d, ref, tol):
    d.out.fill_(float("nan"))
    api.spec_verify_attn_static(d.attn)
    torch.cuda.synchronize()
    got = d.out.float()
    assert bool(torch.isfinite(got).all()), "outputs left unwritten"
    err = float((got - ref).abs().max())
    assert err <= tol, err
    assert torch.equal(got, ref), f"static entry differs from the workspace entry (max {err})"
    assert d.status_bits() == 0


@pytest.mark.parametrize("name,kw", [
    ("tiny_f32", {}),
    ("bass_b8", dict(B=5, Hq=8, Hkv=2, L_lo=0, L_hi=700, K_lo=0, K_hi=7, gen_seed=31)),
    ("bass_b8", {}),
])
def test_static_matches_workspace_entry_twice(api, name, kw):
    inp = W.make_inputs(W.workload(name, **kw), with_logits=False)
    d, ref = _reference(api, inp)
    for _ in range(2):
        _static_call_matches(api, d, ref, _tol(inp))


def test_static_alternating_shapes(api):
    """Calls of different shapes share the array: a small call's partials must
    never land where a larger call's merge counters live."""
    cases = [W.workload("bass_b8", B=3, Hq=4, Hkv=4, L_lo=100, L_hi=3000, K_lo=2, K_hi=6,
                        gen_seed=41),
             W.workload("bass_b8", gen_seed=42)]
    runs = [_reference(api, W.make_inputs(w, with_logits=False)) for w in cases]
    for k in (0, 1, 0, 1):
        d, ref = runs[k]
        _static_call_matches(api, d, ref, 2e-2)


def test_static_reset_between_calls(api):
    """sv_static_scratch_reset zeroes the merge counters (what a caller does
    after a call that timed out); calls before and after it give the same bits."""
    inp = W.make_inputs(W.workload("bass_b8", B=6, Hq=8, Hkv=4, L_lo=64, L_hi=2500,
                                   gen_seed=43), with_logits=False)
    d, ref = _reference(api, inp)
    _static_call_matches(api, d, ref, 2e-2)
    api.sv_static_scratch_reset()
    _static_call_matches(api, d, ref, 2e-2)
    api.sv_static_scratch_reset()
    api.sv_static_scratch_reset()
    _static_call_matches(api, d, ref, 2e-2)


def test_static_rejects_oversized_scratch(api):
    """The 8192-row shared-prefix workload needs more scratch than the static
    array holds: refused with SV_ERR_WORKSPACE before anything launches."""
    from speculative_decoding_verify_09_gb300._binding import lib
    inp = W.make_inputs(W.workload("shared_prefix_s32"), with_logits=False)
    d = DeviceStep(inp, api)
    need = lib.sv_workspace_bytes(ctypes.byref(d.attn), None)
    assert need > (16 << 20)
    with pytest.raises(RuntimeError, match="static array holds"):
        api.spec_verify_attn_static(d.attn)
    torch.cuda.synchronize()
    assert bool(torch.isnan(d.out.float()).all())

"""The C-ABI library: it builds, loads without a GPU, exports exactly what
include/*.h declares, and rejects bad host arguments synchronously (these
calls launch nothing, so they run on a GPU-less host)."""
import ctypes
import glob
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def binding():
    from speculative_decoding_verify_09_gb300 import build
    build()
    from speculative_decoding_verify_09_gb300 import _binding
    return _binding


def declared_symbols():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        src = open(h).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        for m in re.finditer(r"SV_API\s+[\w\s\*]+?\b(\w+)\s*\(", src):
            names.add(m.group(1))
    return names


def test_exports_exactly_the_declared_symbols(binding):
    decl = declared_symbols()
    assert {"spec_verify_attn", "spec_reject_sample", "kv_append_ragged",
            "spec_verify_step"} <= decl
    for name in decl:
        assert hasattr(binding.lib, name), name
    out = subprocess.run(["nm", "-D", "--defined-only", binding.LIB_PATH],
                         capture_output=True, text=True, check=True).stdout
    exported = {ln.split()[-1] for ln in out.splitlines() if ln.split() and ln.split()[1] in "TW"}
    exported = {e for e in exported if not e.startswith("_")}
    assert exported == decl


def test_struct_mirrors_and_version(binding):
    assert binding.lib.sv_abi_version() == 5
    assert binding.lib.sv_struct_size(0) == ctypes.sizeof(binding.AttnArgs)
    assert binding.lib.sv_struct_size(1) == ctypes.sizeof(binding.SampleArgs)
    assert binding.lib.sv_struct_size(2) == ctypes.sizeof(binding.DraftArgs)


def _attn(b, **kw):
    a = b.AttnArgs()
    a.batch, a.num_q_heads, a.num_kv_heads, a.head_dim = 2, 8, 2, 128
    a.dtype, a.max_q_rows, a.num_rows, a.kv_rows_bound, a.pool_rows = b.SV_BF16, 5, 10, 100, 200
    for k in ("cu_q", "q", "k_new", "v_new", "k_cache", "v_cache", "kv_start", "kv_len", "out"):
        setattr(a, k, 4096)
    for k, v in kw.items():
        setattr(a, k, v)
    return a


def _sample(b, **kw):
    s = b.SampleArgs()
    s.batch, s.vocab, s.dtype, s.max_q_rows, s.num_rows = 2, 1000, b.SV_BF16, 5, 10
    s.temperature, s.top_p, s.seed = 1.0, 1.0, 0
    for k in ("cu_q", "target_logits", "draft_logits", "draft_tokens", "kv_len", "num_accepted",
              "out_tokens"):
        setattr(s, k, 4096)
    for k, v in kw.items():
        setattr(s, k, v)
    return s


@pytest.mark.parametrize("field,value,status", [
    ("num_kv_heads", 3, 1), ("head_dim", 96, 4), ("max_q_rows", 0, 1), ("max_q_rows", 17, 1),
    ("num_rows", 11, 1), ("num_rows", 1, 1), ("dtype", 7, 1), ("q", 4097, 1), ("out", 0, 1),
    ("num_groups", 1, 1), ("num_groups", 300, 1), ("prefix_rows_bound", -1, 1),
    ("batch", 5000, 1),
])
def test_attention_host_validation(binding, field, value, status):
    a = _attn(binding, **{field: value})
    if field == "prefix_rows_bound":
        a.num_groups, a.group, a.prefix_start, a.prefix_len = 1, 4096, 4096, 4096
    st = binding.lib.spec_verify_attn(ctypes.byref(a), ctypes.c_void_p(4096), 1 << 30, None)
    assert st == status, binding.last_error()
    assert binding.last_error()
    assert binding.lib.sv_workspace_bytes(ctypes.byref(a), None) == 0


def test_shared_prefix_needs_bf16(binding):
    a = _attn(binding, dtype=binding.SV_F32, num_groups=1, group=4096, prefix_start=4096,
              prefix_len=4096)
    st = binding.lib.spec_verify_attn(ctypes.byref(a), ctypes.c_void_p(4096), 1 << 30, None)
    assert st == binding.SV_ERR_UNSUPPORTED


@pytest.mark.parametrize("field,value,status", [
    ("temperature", -1.0, 1), ("temperature", float("inf"), 1), ("temperature", float("nan"), 1),
    ("top_p", 0.0, 1), ("top_k", -1, 1),
    ("vocab", 0, 4), ("vocab", 10 ** 7, 4), ("num_rows", 1, 1), ("target_logits", 0, 1),
])
def test_sampling_host_validation(binding, field, value, status):
    s = _sample(binding, **{field: value})
    st = binding.lib.spec_reject_sample(ctypes.byref(s), ctypes.c_void_p(4096), 1 << 30, None)
    assert st == status, binding.last_error()


def test_workspace_checks(binding):
    a, s = _attn(binding), _sample(binding)
    need = binding.lib.sv_workspace_bytes(ctypes.byref(a), ctypes.byref(s))
    assert need > 0 and need % 256 == 0
    assert binding.lib.sv_workspace_bytes(ctypes.byref(a), None) < need
    st = binding.lib.spec_verify_step(ctypes.byref(a), ctypes.byref(s), ctypes.c_void_p(4096),
                                      ctypes.c_void_p(8192), ctypes.c_void_p(4096), need - 1, None)
    assert st == binding.SV_ERR_WORKSPACE
    st = binding.lib.spec_verify_step(ctypes.byref(a), ctypes.byref(s), ctypes.c_void_p(4096),
                                      ctypes.c_void_p(8192), ctypes.c_void_p(4104), need, None)
    assert st == binding.SV_ERR_WORKSPACE          # misaligned


def test_step_rejects_mismatched_batches_and_aliasing(binding):
    a, s = _attn(binding), _sample(binding, cu_q=8192)
    st = binding.lib.spec_verify_step(ctypes.byref(a), ctypes.byref(s), ctypes.c_void_p(4096),
                                      ctypes.c_void_p(8192), ctypes.c_void_p(4096), 1 << 30, None)
    assert st == binding.SV_ERR_INVALID
    s = _sample(binding)
    st = binding.lib.spec_verify_step(ctypes.byref(a), ctypes.byref(s), ctypes.c_void_p(4096),
                                      ctypes.c_void_p(4096), ctypes.c_void_p(4096), 1 << 30, None)
    assert st == binding.SV_ERR_INVALID            # new_kv_len aliases kv_len


def test_append_host_validation(binding):
    f = binding.lib.kv_append_ragged
    p = ctypes.c_void_p(4096)
    assert f(2, 1, 3, binding.SV_BF16, 5, 10, *([p] * 5), 100, p, p, p, p,
             ctypes.c_void_p(8192), None, None) == binding.SV_ERR_UNSUPPORTED   # 6-byte rows
    assert f(2, 8, 128, binding.SV_BF16, 5, 10, *([p] * 5), 100, p, p, p, p, p, None,
             None) == binding.SV_ERR_INVALID      # new_kv_len aliases kv_len


def test_binding_module_has_no_fallback():
    src = open(os.path.join(ROOT, "speculative_decoding_verify_09_gb300", "_binding.py")).read()
    assert "oracle" not in src and "import numpy" not in src
    for f in glob.glob(os.path.join(ROOT, "speculative_decoding_verify_09_gb300", "*.py")):
        assert "import oracle" not in open(f).read() and "from oracle" not in open(f).read()


def _draft(b, **kw):
    d = b.DraftArgs()
    d.batch, d.vocab, d.dtype = 4, 1000, b.SV_BF16
    d.temperature, d.top_p, d.seed = 1.0, 1.0, 0
    for k in ("draft_logits", "kv_len", "draft_tokens"):
        setattr(d, k, 4096)
    for k, v in kw.items():
        setattr(d, k, v)
    return d


@pytest.mark.parametrize("field,value,status", [
    ("temperature", -1.0, 1), ("temperature", float("nan"), 1), ("top_p", 0.0, 1),
    ("top_k", -2, 1), ("vocab", 0, 4), ("vocab", 10 ** 7, 4), ("dtype", 9, 1),
    ("draft_logits", 0, 1), ("draft_tokens", 0, 1), ("batch", -1, 1),
])
def test_draft_host_validation(binding, field, value, status):
    d = _draft(binding, **{field: value})
    st = binding.lib.spec_draft_sample(ctypes.byref(d), ctypes.c_void_p(4096), 1 << 30, None)
    assert st == status, binding.last_error()
    assert binding.lib.sv_draft_workspace_bytes(ctypes.byref(d)) == 0


def test_draft_workspace_checks(binding):
    d = _draft(binding)
    need = binding.lib.sv_draft_workspace_bytes(ctypes.byref(d))
    assert need > 0 and need % 256 == 0
    st = binding.lib.spec_draft_sample(ctypes.byref(d), ctypes.c_void_p(4096), need - 1, None)
    assert st == binding.SV_ERR_WORKSPACE


@pytest.mark.parametrize("kw,status", [
    (dict(kv_dtype=2, head_dim=64), 4),                  # E4M3 built for head_dim 128
    (dict(kv_dtype=2, dtype=0), 4),                      # E4M3 K/V with fp32 q/out
    (dict(kv_dtype=2, num_q_heads=16, num_kv_heads=2), 4),   # 8 x 5 rows > 16
    (dict(kv_dtype=2, num_groups=1, group=4096, prefix_start=4096, prefix_len=4096), 4),
    (dict(kv_dtype=2, num_q_heads=4, k_scale=float("nan")), 1),
    (dict(kv_dtype=2, num_q_heads=4, v_scale=-1.0), 1),
    (dict(kv_dtype=7), 1),
])
def test_e4m3_attention_host_validation(binding, kw, status):
    a = _attn(binding, **kw)
    st = binding.lib.spec_verify_attn(ctypes.byref(a), ctypes.c_void_p(4096), 1 << 30, None)
    assert st == status, binding.last_error()


def test_e4m3_attention_accepted_shapes_size_a_workspace(binding):
    a = _attn(binding, kv_dtype=2, num_q_heads=4, num_kv_heads=2, k_scale=0.5, v_scale=0.25)
    assert binding.lib.sv_workspace_bytes(ctypes.byref(a), None) > 0


def test_empty_batches_are_no_ops(binding):
    """B = 0 passes every host check and launches nothing (no device needed)."""
    ws = ctypes.c_void_p(4096)
    a = binding.AttnArgs()
    a.batch, a.num_q_heads, a.num_kv_heads, a.head_dim = 0, 4, 4, 128
    a.dtype, a.max_q_rows = binding.SV_BF16, 1
    assert binding.lib.spec_verify_attn(ctypes.byref(a), ws, 1 << 20, None) == binding.SV_OK
    s = binding.SampleArgs()
    s.batch, s.vocab, s.dtype, s.max_q_rows, s.num_rows = 0, 100, binding.SV_BF16, 1, 0
    s.temperature, s.top_p = 1.0, 1.0
    assert binding.lib.spec_reject_sample(ctypes.byref(s), ws, 1 << 20, None) == binding.SV_OK
    d = binding.DraftArgs()
    d.batch, d.vocab, d.dtype, d.temperature, d.top_p = 0, 100, binding.SV_BF16, 1.0, 1.0
    assert binding.lib.spec_draft_sample(ctypes.byref(d), ws, 1 << 20, None) == binding.SV_OK
    assert binding.lib.sv_draft_workspace_bytes(ctypes.byref(d)) > 0


def test_api_refuses_host_tensors():
    """The torch-facing calls take CUDA tensors only: there is no CPU path."""
    import torch
    from speculative_decoding_verify_09_gb300 import build
    build()
    from speculative_decoding_verify_09_gb300 import api
    x = torch.zeros(4, 2, 128, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="CUDA"):
        api.attn_args(x, x, x, x, x, torch.zeros(3, dtype=torch.int32),
                      torch.zeros(2, dtype=torch.int64), torch.zeros(2, dtype=torch.int32), x,
                      max_q_rows=2, kv_rows_bound=0)


@pytest.mark.parametrize("std,compiler,lang", [("c99", "gcc", "c"), ("c++17", "g++", "c++")])
def test_header_compiles_as_plain_c_and_cxx(tmp_path, std, compiler, lang):
    """include/spec_verify.h is a C ABI: it must compile as strict C99 (and as
    C++), with every argument struct usable from C."""
    src = tmp_path / "use_header.c"
    src.write_text('#include "spec_verify.h"\n'
                   "int main(void) {\n"
                   "  sv_attn_args a; sv_sample_args s; sv_draft_args d;\n"
                   "  sv_status (*step)(const sv_attn_args *, const sv_sample_args *,\n"
                   "                    const int32_t *, int32_t *, void *, size_t, void *)\n"
                   "      = spec_verify_step;\n"
                   "  (void)a; (void)s; (void)d; (void)step;\n"
                   "  return 0;\n"
                   "}\n")
    r = subprocess.run([compiler, f"-std={std}", "-Wall", "-Wextra", "-Werror", "-pedantic",
                        "-x", lang, "-fsyntax-only", "-I", os.path.join(ROOT, "include"),
                        str(src)], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr

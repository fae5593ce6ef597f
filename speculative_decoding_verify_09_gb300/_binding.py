"""ctypes binding of libspecverify.so (argument marshalling only).

Every step of the verify path runs in the library's CUDA kernels; this module
only turns torch CUDA tensors into pointers and the current torch stream into
the cudaStream_t the C ABI takes.  There is no fallback: if the library is
missing the import fails.
"""
import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_lib", "libspecverify.so")

SV_OK, SV_ERR_INVALID, SV_ERR_WORKSPACE, SV_ERR_CUDA, SV_ERR_UNSUPPORTED = range(5)
SV_F32, SV_BF16, SV_E4M3 = 0, 1, 2
DEV_CAPACITY, DEV_BAD_TOKEN, DEV_NONFINITE, DEV_EMPTY_RESIDUAL, DEV_BAD_LENGTH = 1, 2, 4, 8, 16
DEV_TIMEOUT, DEV_BAD_PARAM = 32, 64

_p = ctypes.c_void_p


class AttnArgs(ctypes.Structure):
    """Mirror of sv_attn_args."""
    _fields_ = [
        ("batch", ctypes.c_int32), ("num_q_heads", ctypes.c_int32),
        ("num_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
        ("dtype", ctypes.c_int32), ("max_q_rows", ctypes.c_int32),
        ("num_rows", ctypes.c_int64), ("kv_rows_bound", ctypes.c_int64),
        ("pool_rows", ctypes.c_int64), ("scale", ctypes.c_float),
        ("num_groups", ctypes.c_int32), ("prefix_rows_bound", ctypes.c_int64),
        ("cu_q", _p), ("q", _p), ("k_new", _p), ("v_new", _p), ("k_cache", _p),
        ("v_cache", _p), ("kv_start", _p), ("kv_len", _p), ("group", _p),
        ("prefix_start", _p), ("prefix_len", _p), ("out", _p), ("dev_status", _p),
        ("kv_dtype", ctypes.c_int32), ("k_scale", ctypes.c_float), ("v_scale", ctypes.c_float),
    ]


class SampleArgs(ctypes.Structure):
    """Mirror of sv_sample_args."""
    _fields_ = [
        ("batch", ctypes.c_int32), ("vocab", ctypes.c_int32), ("dtype", ctypes.c_int32),
        ("max_q_rows", ctypes.c_int32), ("num_rows", ctypes.c_int64),
        ("temperature", ctypes.c_float), ("top_p", ctypes.c_float), ("seed", ctypes.c_uint64),
        ("cu_q", _p), ("target_logits", _p), ("draft_logits", _p), ("draft_tokens", _p),
        ("kv_len", _p), ("seq_ids", _p), ("num_accepted", _p), ("out_tokens", _p),
        ("dev_status", _p), ("top_k", ctypes.c_int32), ("temperatures", _p), ("top_ps", _p),
        ("top_ks", _p),
    ]


class DraftArgs(ctypes.Structure):
    """Mirror of sv_draft_args."""
    _fields_ = [
        ("batch", ctypes.c_int32), ("vocab", ctypes.c_int32), ("dtype", ctypes.c_int32),
        ("top_k", ctypes.c_int32), ("temperature", ctypes.c_float), ("top_p", ctypes.c_float),
        ("seed", ctypes.c_uint64), ("draft_logits", _p), ("kv_len", _p), ("seq_ids", _p),
        ("temperatures", _p), ("top_ps", _p), ("top_ks", _p), ("draft_tokens", _p),
        ("dev_status", _p),
    ]


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"{LIB_PATH} is not built; run speculative_decoding_verify_09_gb300.build.build() "
            "(there is no non-CUDA fallback)")
    lib = ctypes.CDLL(LIB_PATH)
    P = ctypes.POINTER
    lib.sv_workspace_bytes.argtypes = [P(AttnArgs), P(SampleArgs)]
    lib.sv_workspace_bytes.restype = ctypes.c_size_t
    lib.sv_workspace_init.argtypes = [_p, ctypes.c_size_t, _p]
    lib.sv_workspace_init.restype = ctypes.c_int
    lib.spec_verify_attn.argtypes = [P(AttnArgs), _p, ctypes.c_size_t, _p]
    lib.spec_verify_attn.restype = ctypes.c_int
    lib.spec_verify_attn_static.argtypes = [P(AttnArgs), _p]
    lib.spec_verify_attn_static.restype = ctypes.c_int
    lib.sv_static_scratch_reset.argtypes = [_p]
    lib.sv_static_scratch_reset.restype = ctypes.c_int
    lib.sv_set_wait_limit.argtypes = [ctypes.c_uint32]
    lib.sv_set_wait_limit.restype = ctypes.c_int
    lib.spec_reject_sample.argtypes = [P(SampleArgs), _p, ctypes.c_size_t, _p]
    lib.spec_reject_sample.restype = ctypes.c_int
    lib.sv_draft_workspace_bytes.argtypes = [P(DraftArgs)]
    lib.sv_draft_workspace_bytes.restype = ctypes.c_size_t
    lib.spec_draft_sample.argtypes = [P(DraftArgs), _p, ctypes.c_size_t, _p]
    lib.spec_draft_sample.restype = ctypes.c_int
    lib.sv_draft_step_workspace_bytes.argtypes = [P(AttnArgs), P(DraftArgs)]
    lib.sv_draft_step_workspace_bytes.restype = ctypes.c_size_t
    lib.spec_draft_step.argtypes = [P(AttnArgs), P(DraftArgs), _p, _p, _p, ctypes.c_size_t, _p]
    lib.spec_draft_step.restype = ctypes.c_int
    lib.kv_append_ragged.argtypes = [ctypes.c_int32] * 5 + [ctypes.c_int64] + [_p] * 5 + \
        [ctypes.c_int64] + [_p] * 7
    lib.kv_append_ragged.restype = ctypes.c_int
    lib.spec_verify_step.argtypes = [P(AttnArgs), P(SampleArgs), _p, _p, _p, ctypes.c_size_t, _p]
    lib.spec_verify_step.restype = ctypes.c_int
    lib.sv_last_error.argtypes = []
    lib.sv_last_error.restype = ctypes.c_char_p
    lib.sv_abi_version.argtypes = []
    lib.sv_abi_version.restype = ctypes.c_int32
    lib.sv_struct_size.argtypes = [ctypes.c_int32]
    lib.sv_struct_size.restype = ctypes.c_size_t
    if lib.sv_struct_size(0) != ctypes.sizeof(AttnArgs) or \
            lib.sv_struct_size(1) != ctypes.sizeof(SampleArgs) or \
            lib.sv_struct_size(2) != ctypes.sizeof(DraftArgs):
        raise ImportError("libspecverify.so struct layout does not match this binding")
    return lib


lib = _load()


class SpecVerifyError(RuntimeError):
    def __init__(self, status, msg):
        super().__init__(f"status {status}: {msg}")
        self.status = status


def _check(st):
    if st != SV_OK:
        raise SpecVerifyError(st, lib.sv_last_error().decode())


def last_error():
    return lib.sv_last_error().decode()


def abi_version():
    return lib.sv_abi_version()

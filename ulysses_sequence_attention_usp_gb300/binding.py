"""ctypes binding of the USP C ABI (include/usp.h).

Argument marshalling only: every function here forwards to the entry point
of the same name in ``libusp.so``; tensors are passed as raw pointers
(``torch.Tensor.data_ptr()``), streams as ``cudaStream_t`` handles.  A
non-OK status raises :class:`UspError`.  If the library has not been built,
importing this module raises ImportError: there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
import re

_HERE = os.path.dirname(os.path.abspath(__file__))
# USP_DEBUG_BOUNDS=1 loads the build with index guards (build(debug=True))
DEBUG = os.environ.get("USP_DEBUG_BOUNDS") == "1"
LIB_PATH = os.path.join(_HERE, "_build_debug" if DEBUG else "_build", "libusp.so")
HEADER = os.path.join(os.path.dirname(_HERE), "include", "usp.h")

if not os.path.exists(LIB_PATH):
    raise ImportError(
        f"USP CUDA library not built ({LIB_PATH} missing); run "
        "`python -m ulysses_sequence_attention_usp_gb300.build" + (" -d`" if DEBUG else "`"))

_lib = ctypes.CDLL(LIB_PATH)

USP_OK = 0
STATUS_NAMES = {0: "USP_OK", 1: "USP_ERR_INVALID_ARG", 2: "USP_ERR_HEADS_NOT_DIVISIBLE",
                3: "USP_ERR_UNSUPPORTED", 4: "USP_ERR_CUDA", 5: "USP_ERR_TIMEOUT",
                6: "USP_ERR_OUT_OF_BOUNDS"}


class UspError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        msg = _lib.usp_status_string(status).decode()
        super().__init__(f"{where}: {STATUS_NAMES.get(status, status)} ({msg})")


class usp_dims(ctypes.Structure):
    _fields_ = [("S", ctypes.c_int64), ("P", ctypes.c_int32), ("Hq", ctypes.c_int32),
                ("Hkv", ctypes.c_int32), ("D", ctypes.c_int32),
                ("cu_seqlens", ctypes.c_void_p), ("cu_seqlens_host", ctypes.c_void_p),
                ("n_docs", ctypes.c_int32), ("causal", ctypes.c_int32),
                ("scale", ctypes.c_float), ("zigzag", ctypes.c_int32)]


_P = ctypes.c_void_p
_I32 = ctypes.c_int32
_I64 = ctypes.c_int64
_DIMS = ctypes.POINTER(usp_dims)

_SIGS = {
    "usp_pad_shard": [_DIMS, _P, _I32, _P, _P, _P, _P],
    "usp_seq_to_head_rope": [_DIMS, _P, _I32, _P, _P, _I64, _I32, _P, _P],
    "usp_attn_fwd": [_DIMS, _P, _P, _P, _P, _P, _P, _P],
    "usp_attn_fwd_window": [_DIMS, _P, _P, _P, _P, _I64, _I64, _P, _P, _P],
    "usp_lse_merge": [_DIMS, _P, _P, _P, _P, _I32, _P, _P],
    "usp_attn_bwd": [_DIMS, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, ctypes.c_size_t, _P],
    "usp_attn_bwd_noalloc": [_DIMS, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P],
    "usp_head_to_seq": [_DIMS, _P, _I32, _P, _P, _I64, _I32, _P, _P],
    "usp_rope_table": [_I64, _I32, ctypes.c_double, ctypes.c_double, _I32, _P],
    "usp_device_status": [_P],
    "usp_selftest_bounded_wait": [_I32, _P],
}
for _name, _args in _SIGS.items():
    _f = getattr(_lib, _name)
    _f.argtypes = _args
    _f.restype = ctypes.c_int
_lib.usp_attn_bwd_workspace.argtypes = [_DIMS]
_lib.usp_attn_bwd_workspace.restype = ctypes.c_size_t
_lib.usp_status_string.argtypes = [ctypes.c_int]
_lib.usp_status_string.restype = ctypes.c_char_p
_lib.usp_abi_version.argtypes = []
_lib.usp_abi_version.restype = ctypes.c_int
_lib.usp_debug_build.argtypes = []
_lib.usp_debug_build.restype = ctypes.c_int
_lib.usp_launch_count.argtypes = []
_lib.usp_launch_count.restype = ctypes.c_uint64


def header_entry_points() -> list:
    """Names of the functions include/usp.h declares."""
    with open(HEADER) as f:
        text = f.read()
    return sorted(set(re.findall(r"^\s*(?:usp_status|size_t|const char\*|int|uint64_t)\s+(usp_\w+)\s*\(",
                                 text, flags=re.M)))


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):
        return x.data_ptr()
    if hasattr(x, "ctypes"):          # numpy array (host)
        return x.ctypes.data
    raise TypeError(f"cannot pass {type(x)} as a pointer")


def _stream(s):
    if s is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(s, int):
        return s
    return s.cuda_stream


def _check(st, where):
    if st != USP_OK:
        raise UspError(st, where)


def make_dims(S, P, Hq, Hkv, D, cu_seqlens=None, cu_seqlens_host=None, scale=0.0,
              causal=True, zigzag=False):
    """Build a usp_dims.  ``cu_seqlens`` is a device int32 tensor (or None for
    one document); ``cu_seqlens_host`` an optional numpy int32 copy;
    ``causal=False`` selects bidirectional attention within each document;
    ``zigzag=True`` the zigzag shard layout of the sequence-sharded buffers.
    The returned struct keeps references to both arrays."""
    n_docs = 0
    if cu_seqlens is not None:
        n_docs = int(cu_seqlens.numel()) - 1
    d = usp_dims(int(S), int(P), int(Hq), int(Hkv), int(D), _ptr(cu_seqlens),
                 _ptr(cu_seqlens_host), n_docs, 1 if causal else 0, float(scale),
                 1 if zigzag else 0)
    d._keep = (cu_seqlens, cu_seqlens_host)
    return d


def usp_pad_shard(dims, x, H, x_seq, pos, doc, stream=None):
    _check(_lib.usp_pad_shard(ctypes.byref(dims), _ptr(x), H, _ptr(x_seq), _ptr(pos), _ptr(doc),
                              _stream(stream)), "usp_pad_shard")


def usp_seq_to_head_rope(dims, x_seq, H, pos, rope_cs, rope_len, rope_mode, x_head, stream=None):
    _check(_lib.usp_seq_to_head_rope(ctypes.byref(dims), _ptr(x_seq), H, _ptr(pos),
                                     _ptr(rope_cs), int(rope_len), int(rope_mode), _ptr(x_head),
                                     _stream(stream)), "usp_seq_to_head_rope")


def usp_attn_fwd(dims, q_h, k_h, v_h, doc, o_h, lse, stream=None):
    _check(_lib.usp_attn_fwd(ctypes.byref(dims), _ptr(q_h), _ptr(k_h), _ptr(v_h), _ptr(doc),
                             _ptr(o_h), _ptr(lse), _stream(stream)), "usp_attn_fwd")


def usp_attn_fwd_window(dims, q_h, k_h, v_h, doc, k_lo, k_hi, o_h, lse, stream=None):
    _check(_lib.usp_attn_fwd_window(ctypes.byref(dims), _ptr(q_h), _ptr(k_h), _ptr(v_h),
                                    _ptr(doc), int(k_lo), int(k_hi), _ptr(o_h), _ptr(lse),
                                    _stream(stream)), "usp_attn_fwd_window")


def usp_lse_merge(dims, o_acc, lse_acc, o_part, lse_part, first, o_out=None, stream=None):
    _check(_lib.usp_lse_merge(ctypes.byref(dims), _ptr(o_acc), _ptr(lse_acc), _ptr(o_part),
                              _ptr(lse_part), 1 if first else 0, _ptr(o_out), _stream(stream)),
           "usp_lse_merge")


def usp_attn_bwd_workspace(dims) -> int:
    return int(_lib.usp_attn_bwd_workspace(ctypes.byref(dims)))


def usp_attn_bwd(dims, q_h, k_h, v_h, o_h, lse, do_h, doc, dq_h, dk_h, dv_h, workspace,
                 ws_bytes, stream=None):
    _check(_lib.usp_attn_bwd(ctypes.byref(dims), _ptr(q_h), _ptr(k_h), _ptr(v_h), _ptr(o_h),
                             _ptr(lse), _ptr(do_h), _ptr(doc), _ptr(dq_h), _ptr(dk_h),
                             _ptr(dv_h), _ptr(workspace), int(ws_bytes), _stream(stream)),
           "usp_attn_bwd")


def usp_attn_bwd_noalloc(dims, q_h, k_h, v_h, o_h, lse, do_h, doc, dq_h, dk_h, dv_h,
                         stream=None):
    """usp_attn_bwd without a workspace argument (fixed scratch inside the
    library; see include/usp.h for the size limit and the sharing rules)."""
    _check(_lib.usp_attn_bwd_noalloc(ctypes.byref(dims), _ptr(q_h), _ptr(k_h), _ptr(v_h),
                                     _ptr(o_h), _ptr(lse), _ptr(do_h), _ptr(doc), _ptr(dq_h),
                                     _ptr(dk_h), _ptr(dv_h), _stream(stream)),
           "usp_attn_bwd_noalloc")


def usp_head_to_seq(dims, x_head, H, pos, rope_cs, rope_len, rope_mode, x_seq, stream=None):
    _check(_lib.usp_head_to_seq(ctypes.byref(dims), _ptr(x_head), H, _ptr(pos), _ptr(rope_cs),
                                int(rope_len), int(rope_mode), _ptr(x_seq), _stream(stream)),
           "usp_head_to_seq")


def usp_rope_table(n_pos, D, base, yarn_factor=1.0, yarn_orig_ctx=0):
    """Host fp32 table [n_pos][D/2][2] of (cos, sin) (numpy array)."""
    import numpy as np
    out = np.empty((int(n_pos), D // 2, 2), dtype=np.float32)
    _check(_lib.usp_rope_table(int(n_pos), int(D), float(base), float(yarn_factor),
                               int(yarn_orig_ctx), out.ctypes.data), "usp_rope_table")
    return out


def usp_device_status(stream=None):
    _check(_lib.usp_device_status(_stream(stream)), "usp_device_status")


def usp_selftest_bounded_wait(limit_us, stream=None):
    _check(_lib.usp_selftest_bounded_wait(int(limit_us), _stream(stream)),
           "usp_selftest_bounded_wait")


def usp_status_string(status: int) -> str:
    return _lib.usp_status_string(int(status)).decode()


def usp_abi_version() -> int:
    return int(_lib.usp_abi_version())


def usp_launch_count() -> int:
    return int(_lib.usp_launch_count())


def usp_debug_build() -> bool:
    return bool(_lib.usp_debug_build())


def raw_call(name, *args):
    """Call an entry point with already-marshalled ctypes arguments and return
    its raw status (used by the argument-validation tests)."""
    return getattr(_lib, name)(*args)

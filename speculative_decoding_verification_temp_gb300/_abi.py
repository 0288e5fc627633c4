"""ctypes view of the C ABI declared in include/specverify.h.

Loading fails loudly when libspecverify.so has not been built: there is no
other implementation of these operations in this package.
"""

import ctypes
import os

from . import build as _build

SPEC_OK = 0
SPEC_ERR_INVALID_ARG = 1
SPEC_ERR_CUDA = 2
SPEC_ERR_UNSUPPORTED = 3

SPEC_STATIC_SCRATCH_BYTES = 16 * 1024 * 1024

SPEC_F32 = 0
SPEC_BF16 = 1

FLAG_BAD_TOKEN = 1
FLAG_ZERO_Q = 2
FLAG_NONFINITE = 4
FLAG_DEGENERATE_RESIDUAL = 8
FLAG_DEPTH = 16
FLAG_TIMEOUT = 32
FLAG_BAD_TREE = 64

EXPORTS = (
    "spec_verify_chain_workspace_size",
    "spec_verify_chain",
    "spec_verify_chain_static",
    "spec_verify_tree_workspace_size",
    "spec_verify_tree",
    "spec_tree_mask",
    "spec_overlap",
    "spec_typical_workspace_size",
    "spec_typical_accept",
    "spec_tree_rerank",
    "spec_status_string",
    "spec_set_profile_events",
    "spec_set_wait_limit",
)


class spec_policy(ctypes.Structure):
    _fields_ = [("temperature", ctypes.c_void_p), ("top_k", ctypes.c_void_p),
                ("top_p", ctypes.c_void_p), ("min_p", ctypes.c_void_p)]


_p = ctypes.c_void_p
_i = ctypes.c_int
_i64 = ctypes.c_int64
_u64 = ctypes.c_uint64
_sz = ctypes.c_size_t

_lib = None


def library_path():
    return _build.LIB_PATH


def load():
    """The loaded shared library (raises if it was never built)."""
    global _lib
    if _lib is not None:
        return _lib
    path = library_path()
    if not os.path.exists(path):
        raise RuntimeError(
            f"{path} is missing: build it with "
            "`python -c 'import __graft_entry__ as g; g.build()'` (needs nvcc)")
    lib = ctypes.CDLL(path)
    lib.spec_verify_chain_workspace_size.argtypes = [_i, _i, _i, _i]
    lib.spec_verify_chain_workspace_size.restype = _sz
    lib.spec_verify_tree_workspace_size.argtypes = [_i, _i, _i, _i]
    lib.spec_verify_tree_workspace_size.restype = _sz
    lib.spec_verify_chain.argtypes = [
        _p, _i64, _p, _i64, _i, _i, _i, _i, _p, spec_policy, spec_policy, _u64, _p,
        _p, _p, _p, _p, _p, _sz, _p]
    lib.spec_verify_chain.restype = _i
    lib.spec_verify_chain_static.argtypes = [
        _p, _i64, _p, _i64, _i, _i, _i, _i, _p, spec_policy, spec_policy, _u64, _p,
        _p, _p, _p, _p, _p]
    lib.spec_verify_chain_static.restype = _i
    lib.spec_verify_tree.argtypes = [
        _p, _i64, _p, _i64, _i, _i, _i, _i, _i, _p, _p, spec_policy, spec_policy, _u64, _p,
        _p, _p, _p, _p, _p, _p, _sz, _p]
    lib.spec_verify_tree.restype = _i
    lib.spec_tree_mask.argtypes = [_p, _i, _i, _i, _p, _p, _p, _p]
    lib.spec_tree_mask.restype = _i
    lib.spec_overlap.argtypes = [_p, _i64, _p, _i64, _i, _i, _i, _i, spec_policy, spec_policy,
                                 _p, _p, _p]
    lib.spec_overlap.restype = _i
    lib.spec_typical_workspace_size.argtypes = [_i, _i, _i, _i]
    lib.spec_typical_workspace_size.restype = _sz
    lib.spec_typical_accept.argtypes = [_p, _i64, _i, _i, _i, _i, spec_policy, _p,
                                        ctypes.c_float, ctypes.c_float, _p, _p, _p, _p, _sz, _p]
    lib.spec_typical_accept.restype = _i
    lib.spec_tree_rerank.argtypes = [_p, _p, _i, _i, _i, _p, _p, _p, _p, _p, _p]
    lib.spec_tree_rerank.restype = _i
    lib.spec_status_string.argtypes = [_i]
    lib.spec_status_string.restype = ctypes.c_char_p
    lib.spec_set_profile_events.argtypes = [_p, _p]
    lib.spec_set_profile_events.restype = _i
    lib.spec_set_wait_limit.argtypes = [_i64]
    lib.spec_set_wait_limit.restype = _i
    _lib = lib
    return lib


def status_string(code):
    return load().spec_status_string(code).decode()

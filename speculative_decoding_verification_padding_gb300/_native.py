"""ctypes binding of libspecverify (argument marshalling only).

The structs mirror include/libspecverify.h.  Loading fails loudly when the
library has not been built: there is no fallback path.
"""

from __future__ import annotations

import ctypes
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libspecverify.so")

P = ctypes.c_void_p
I32 = ctypes.c_int32
F32 = ctypes.c_float
U64 = ctypes.c_uint64
SZ = ctypes.c_size_t

SV_OK = 0
SV_ERR_INVALID_ARGUMENT = 1
SV_ERR_UNSUPPORTED_SHAPE = 2
SV_ERR_WORKSPACE_TOO_SMALL = 3
SV_ERR_CUDA = 4

SV_DEV_BAD_BLOCK_ID = 1
SV_DEV_BAD_PARENT = 2
SV_DEV_POOL_OVERFLOW = 4
SV_DEV_BAD_WINDOW = 8
SV_DEV_TIMEOUT = 16
SV_DEV_BAD_TOKEN = 32
SV_DEV_UNSUPPORTED = 64
SV_DEV_BAD_LENGTH = 128

SV_ACCEPT_STATIC_SCRATCH_BYTES = 4 << 20


class SvPagedKV(ctypes.Structure):
    _fields_ = [("k_cache", P), ("v_cache", P), ("num_blocks", I32), ("block_size", I32),
                ("n_kv_heads", I32), ("head_dim", I32), ("block_tables", P),
                ("max_blocks_per_req", I32), ("cache_lens", P)]


class SvBatch(ctypes.Structure):
    _fields_ = [("n_req", I32), ("total_rows", I32), ("max_rows_per_req", I32),
                ("cu_rows", P), ("parent", P), ("tokens", P), ("row_begin", P),
                ("row_end", P), ("verify_len", P)]


class SvBlockPool(ctypes.Structure):
    _fields_ = [("free_list", P), ("free_count", P), ("capacity", I32)]


# name -> (restype, argtypes), exactly the functions declared in the header
PROTOTYPES = {
    "sv_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "sv_version": (ctypes.c_char_p, []),
    "sv_tree_attend_workspace": (SZ, [P, P, I32]),
    "sv_tree_attend": (ctypes.c_int, [P, P, P, I32, F32, P, P, SZ, P, P]),
    "sv_accept_workspace": (SZ, [P, I32]),
    "sv_accept": (ctypes.c_int, [P, P, P, I32, F32, U64, P, P, P, P, P, P, P, SZ, P, P]),
    "sv_accept_static": (ctypes.c_int, [P, P, P, I32, F32, U64, P, P, P, P, P, P, P, P]),
    "sv_commit_kv": (ctypes.c_int, [P, P, P, P, P, P, P]),
    "sv_accept_commit_workspace": (SZ, [P, I32]),
    "sv_accept_commit": (ctypes.c_int, [P, P, P, I32, F32, U64, P, P, P, P, P, P, P, P, P, SZ, P,
                                        P]),
    "sv_select_budget_workspace": (SZ, [I32, I32]),
    "sv_select_budget": (ctypes.c_int, [I32, I32, P, P, P, I32, P, P, P, P, SZ, P, P]),
    "sv_chunk_windows": (ctypes.c_int, [P, I32, I32, P, P, P, P]),
    "sv_verify_chunked_workspace": (SZ, [P, P, I32, I32]),
    "sv_verify_chunked": (ctypes.c_int, [P, P, P, I32, F32, P, P, P, I32, F32, U64, I32, P, P, P,
                                         P, P, P, SZ, P, P]),
    "sv_verify_chunked_commit": (ctypes.c_int, [P, P, P, I32, F32, P, P, P, I32, F32, U64, I32, P,
                                                P, P, P, P, P, P, SZ, P, P]),
    "sv_adapt_gamma": (ctypes.c_int, [I32, P, P, P, P, ctypes.c_double, ctypes.c_double, I32, I32,
                                      P, P]),
    "sv_select_chunk": (ctypes.c_int, [I32, P, P, P, ctypes.c_double, ctypes.c_double, U64, P, P,
                                       P, P, P]),
    "sv_selftest_bounded_wait": (ctypes.c_int, [I32, P, P]),
}

_lib = None


class SpecVerifyError(RuntimeError):
    pass


def lib():
    """Load libspecverify.so (built by build.py); raise if it is missing."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise SpecVerifyError(
                f"{LIB_PATH} is missing: build it with "
                "`python -m speculative_decoding_verification_padding_gb300.build`")
        handle = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in PROTOTYPES.items():
            fn = getattr(handle, name)
            fn.restype = res
            fn.argtypes = args
        _lib = handle
    return _lib


def check(status: int, what: str):
    if status != SV_OK:
        msg = lib().sv_status_string(status).decode()
        raise SpecVerifyError(f"{what}: {msg} ({status})")

"""The C-ABI library loads and exports every function include/libspecverify.h
declares, and the ctypes binding covers the same set (no GPU needed)."""

import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "libspecverify.h")


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"\b(sv_[a-z_]+)\s*\(", text)
    return sorted(set(names))


@pytest.fixture(scope="module")
def lib():
    from speculative_decoding_verification_padding_gb300 import build, _native
    build.build()
    return _native.lib()


def test_header_declares_the_boundary():
    names = _declared()
    for n in ("sv_tree_attend", "sv_accept", "sv_commit_kv", "sv_select_budget",
              "sv_verify_chunked", "sv_chunk_windows"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for name in _declared():
        assert hasattr(lib, name), name


def test_binding_covers_the_header():
    from speculative_decoding_verification_padding_gb300 import _native
    assert sorted(_native.PROTOTYPES) == _declared()


def test_host_side_validation_without_gpu(lib):
    # Argument errors are returned before anything is enqueued, so they can
    # be exercised without a device.
    from speculative_decoding_verification_padding_gb300 import _native as N
    assert lib.sv_status_string(N.SV_ERR_WORKSPACE_TOO_SMALL) == b"workspace too small"
    assert lib.sv_tree_attend(None, None, None, 8, 0.1, None, None, 0, None, None) == N.SV_ERR_INVALID_ARGUMENT
    assert lib.sv_select_budget(0, 4, None, None, None, 10, None, None, None, None, 0, None, None) == N.SV_ERR_INVALID_ARGUMENT
    assert lib.sv_select_budget(100, 100, 1, None, 1, 200, 1, 1, 1, None, 0, None, None) == N.SV_ERR_UNSUPPORTED_SHAPE
    import ctypes
    b = N.SvBatch(1, 2, 200, 1, 1, 1, None, None, None)
    assert lib.sv_accept(ctypes.byref(b), 1, None, 16, 0.0, 0, 1, 1, 1, 1, None, None, 1, 1 << 20,
                         None, None) == N.SV_ERR_UNSUPPORTED_SHAPE
    b = N.SvBatch(1, 2, 2, 1, 1, 1, None, None, None)
    assert lib.sv_accept(ctypes.byref(b), 1, None, 16, 1.0, 0, 1, 1, 1, 1, None, None, 256, 1 << 20,
                         None, None) == N.SV_ERR_INVALID_ARGUMENT  # T > 0 needs draft logits
    kv = N.SvPagedKV(256, 256, 10, 16, 2, 96, 1, 4, 1)
    assert lib.sv_tree_attend_workspace(ctypes.byref(b), ctypes.byref(kv), 8) == 0  # head_dim 96
    # draft-length controller: parameters out of range are refused on the host
    assert lib.sv_adapt_gamma(4, 1, 1, 1, 1, 0.7, 2.0, 3, 2, None, None) == N.SV_ERR_INVALID_ARGUMENT
    assert lib.sv_adapt_gamma(4, 1, 1, 1, 1, 0.0, 2.0, 1, 8, None, None) == N.SV_ERR_INVALID_ARGUMENT
    assert lib.sv_adapt_gamma(4, 1, 1, 1, 1, 0.7, -1.0, 1, 8, None, None) == N.SV_ERR_INVALID_ARGUMENT
    assert lib.sv_adapt_gamma(4, 1, 1, 1, 1, 0.7, 2.0, 1, 128, None, None) == N.SV_ERR_INVALID_ARGUMENT
    assert lib.sv_adapt_gamma(0, None, None, None, None, 0.7, 2.0, 1, 8, None, None) == N.SV_OK
    assert lib.sv_selftest_bounded_wait(0, 1, None) == N.SV_ERR_INVALID_ARGUMENT
    assert lib.sv_selftest_bounded_wait(1 << 21, 1, None) == N.SV_ERR_INVALID_ARGUMENT
    assert lib.sv_selftest_bounded_wait(100, None, None) == N.SV_ERR_INVALID_ARGUMENT
    kv = N.SvPagedKV(256, 256, 10, 16, 2, 64, 1, 4, 1)
    need = lib.sv_tree_attend_workspace(ctypes.byref(b), ctypes.byref(kv), 8)
    assert need > 0
    assert lib.sv_tree_attend(ctypes.byref(kv), ctypes.byref(b), 256, 8, 0.125, 256, 256, need - 1,
                              None, None) == N.SV_ERR_WORKSPACE_TOO_SMALL
    # chunked step with the fused commit: the pool is required, and the
    # commit's cache rules (16-token blocks, head_dim 64 / 128) hold
    pool = N.SvBlockPool(256, 256, 4)
    args = (256, 8, 0.125, 256, 256, None, 16, 0.0, 0, 2, 256, 256, 256, 256, 256)
    assert lib.sv_verify_chunked_commit(ctypes.byref(kv), ctypes.byref(b), *args, None, 256, 1 << 20,
                                        None, None) == N.SV_ERR_INVALID_ARGUMENT
    kv96 = N.SvPagedKV(256, 256, 10, 16, 2, 96, 1, 4, 1)
    assert lib.sv_verify_chunked_commit(ctypes.byref(kv96), ctypes.byref(b), *args,
                                        ctypes.byref(pool), 256, 1 << 20, None,
                                        None) == N.SV_ERR_UNSUPPORTED_SHAPE
    # chunk-size rule: sizes and pointers checked on the host
    assert lib.sv_select_chunk(-1, None, None, None, 4096.0, 1.0, 0, 256, 256, 256, None,
                               None) == N.SV_ERR_INVALID_ARGUMENT
    assert lib.sv_select_chunk(4, None, 256, 256, 4096.0, 1.0, 0, 256, 256, 256, None,
                               None) == N.SV_ERR_INVALID_ARGUMENT
    assert lib.sv_select_chunk(4, 256, 256, 256, -1.0, 1.0, 0, 256, 256, 256, None,
                               None) == N.SV_ERR_INVALID_ARGUMENT
    assert lib.sv_select_chunk(4, 256, 256, 256, 4096.0, 1.0, 0, 256, 256, None, None,
                               None) == N.SV_ERR_INVALID_ARGUMENT
    # its workspace is the chunked step's, which also holds the commit's ticket
    wsz = lib.sv_verify_chunked_workspace(ctypes.byref(b), ctypes.byref(kv), 8, 16)
    assert wsz > 0
    assert lib.sv_verify_chunked_commit(ctypes.byref(kv), ctypes.byref(b), *args,
                                        ctypes.byref(pool), 256, wsz - 1, None,
                                        None) == N.SV_ERR_WORKSPACE_TOO_SMALL


def test_static_scratch_holds_the_documented_batch(lib):
    # sv_accept_static promises that any batch of up to 40,000 packed rows fits
    # its fixed scratch array; sv_accept_workspace is a host function.
    import ctypes
    from speculative_decoding_verification_padding_gb300 import _native as N
    worst = 0
    for rows in (1, 100, 2432, 10000, 30000, 40000):
        for per in (1, 2, 5, 9, 128):
            R = max(1, rows // per)
            for maxr in {min(128, per), 128}:
                for V in (16, 1024, 128256, 151936, 262144):
                    b = N.SvBatch(R, rows, maxr, 1, 1, 1, None, None, None)
                    worst = max(worst, lib.sv_accept_workspace(ctypes.byref(b), V))
    assert worst <= N.SV_ACCEPT_STATIC_SCRATCH_BYTES


def test_bound_calls_check_their_arguments_once_when_bound(lib):
    # api.bind_* marshal a call's arguments when bound: host tensors and wrong
    # dtypes are refused there, before anything could be enqueued.
    import torch
    from speculative_decoding_verification_padding_gb300 import api, _native as N
    def i32(n):
        return torch.zeros(n, dtype=torch.int32)
    b = api.Batch(i32(2), torch.full((1,), -1, dtype=torch.int32), i32(1), 1)
    kv = api.PagedKV(torch.zeros((1, 1, 16, 64), dtype=torch.bfloat16),
                     torch.zeros((1, 1, 16, 64), dtype=torch.bfloat16), i32((1, 1)), i32(1))
    q = torch.zeros((1, 1, 64), dtype=torch.bfloat16)
    with pytest.raises(N.SpecVerifyError):
        api.bind_tree_attend(kv, b, q, 1, 0.125, q.clone(), torch.zeros(256, dtype=torch.uint8))
    with pytest.raises(N.SpecVerifyError):
        api.bind_tree_attend(kv, b, q.float(), 1, 0.125, q.clone(), torch.zeros(256, dtype=torch.uint8))
    with pytest.raises(N.SpecVerifyError):
        api.bind_select_budget(torch.zeros((1, 4)), None, torch.zeros(11), i32(1), i32(1),
                               torch.zeros(1, dtype=torch.float32))  # best_theta must be f64

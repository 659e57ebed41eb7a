"""sv_accept_static, the accept call that needs no caller workspace.

Some callers cannot allocate device memory (a plugin handed only its input
and output buffers, an engine that reserved all HBM for its cache pool, a
loop that cannot pay for cudaMalloc's synchronisation).  For them the library
offers sv_accept_static, whose scratch is a fixed array inside the library.
This file checks, through the C ABI, that it returns what sv_accept returns
on the same inputs, on two calls in a row (the array keeps the previous
call's contents, which must not leak into the next result), and that a
problem larger than the array is refused before any launch.  It is named so
that pytest collects it last.
"""

import ctypes

import numpy as np
import pytest
import torch

from speculative_decoding_verification_padding_gb300 import _native as N
from speculative_decoding_verification_padding_gb300 import api, build
from speculative_decoding_verification_padding_gb300 import workloads as wl
from speculative_decoding_verification_padding_gb300.step import DeviceStep

pytestmark = pytest.mark.gpu


def _outputs(w, dev="cuda"):
    R, rows = w.n_req, w.total_rows
    return {"accepted_len": torch.full((R,), -9, dtype=torch.int32, device=dev),
            "accepted_nodes": torch.full((R, w.max_rows), -9, dtype=torch.int32, device=dev),
            "next_token": torch.full((R,), -9, dtype=torch.int32, device=dev),
            "ambiguous": torch.full((R,), 7, dtype=torch.uint8, device=dev),
            "done": torch.full((R,), -9, dtype=torch.int32, device=dev),
            "row_stats": torch.full((rows, 4), float("nan"), dtype=torch.float32, device=dev),
            "dev_status": torch.zeros(1, dtype=torch.int32, device=dev)}


def _static_call(s, o):
    """sv_accept_static straight through the C ABI (ctypes)."""
    b = s.batch.c()
    st = N.lib().sv_accept_static(
        ctypes.byref(b), s.target.data_ptr(), None if s.draft is None else s.draft.data_ptr(),
        s.V, s.T, s.w.seed, o["accepted_len"].data_ptr(), o["accepted_nodes"].data_ptr(),
        o["next_token"].data_ptr(), o["ambiguous"].data_ptr(), o["done"].data_ptr(),
        o["row_stats"].data_ptr(), o["dev_status"].data_ptr(),
        torch.cuda.current_stream().cuda_stream)
    return st


@pytest.mark.parametrize("T", [0.7, 0.0])
def test_static_scratch_accept_matches_workspace_accept_twice(T):
    build.build()
    w = wl.make_workload(wl.config("batch64"), n_req=48, ctx_scale=0.01, vocab=8192,
                         temperature=T, draft_sigma=0.7)
    s = DeviceStep(w, mode="onepass")
    assert api.sv_accept_workspace(s.batch, s.V) <= N.SV_ACCEPT_STATIC_SCRATCH_BYTES
    ref = _outputs(w)
    api.sv_accept(s.batch, s.target, s.draft, s.V, s.T, w.seed, ref["accepted_len"],
                  ref["accepted_nodes"], ref["next_token"], ref["ambiguous"], ref["done"],
                  ref["row_stats"], s.ws, ref["dev_status"])
    torch.cuda.synchronize()
    assert ref["dev_status"].item() == 0
    for call in range(2):
        got = _outputs(w)
        assert _static_call(s, got) == N.SV_OK
        torch.cuda.synchronize()
        assert got["dev_status"].item() == 0, call
        for k in ("accepted_len", "accepted_nodes", "next_token", "ambiguous", "done"):
            assert torch.equal(got[k], ref[k]), (call, k)
        g, r = got["row_stats"].cpu().numpy(), ref["row_stats"].cpu().numpy()
        np.testing.assert_allclose(g, r, atol=1e-5, rtol=0, equal_nan=True)


def test_static_scratch_refuses_problems_larger_than_its_array():
    build.build()
    R, rows, V = 70000, 140000, 16  # needs more than 4 MiB of scratch
    cu = torch.arange(0, rows + 1, 2, dtype=torch.int32, device="cuda")
    b = api.Batch(cu, torch.zeros(rows, dtype=torch.int32, device="cuda"),
                  torch.zeros(rows, dtype=torch.int32, device="cuda"), 2)
    assert api.sv_accept_workspace(b, V) > N.SV_ACCEPT_STATIC_SCRATCH_BYTES
    z = torch.zeros(R, dtype=torch.int32, device="cuda")
    with pytest.raises(N.SpecVerifyError, match="workspace too small"):
        api.sv_accept_static(b, torch.zeros((rows, V), device="cuda"), None, V, 0.0, 1, z,
                             torch.zeros((R, 2), dtype=torch.int32, device="cuda"), z.clone(),
                             torch.zeros(R, dtype=torch.uint8, device="cuda"), None, None)

"""dq_reorder_static, the reordering entry point for callers that cannot
allocate device memory (for example an application that reserved all device
memory for its own pool, or a loop that forbids allocation while it runs).
It keeps its scratch inside the library, so the caller passes only the input
and the output.  Checked against dq_reorder (caller-supplied scratch) through
the C ABI on two calls in a row; the second call is smaller than the first,
so stale scratch contents from the first call must not leak into it.

This file runs last on purpose: it is an addition beside the hot path."""
import ctypes

import numpy as np
import pytest
import torch

from quantized_hop_gradient_gb300 import build, dq

pytestmark = pytest.mark.gpu


def test_reorder_static_matches_reorder_on_two_calls():
    build.build()
    L = dq.lib()
    stream = torch.cuda.current_stream().cuda_stream
    for trial, J in enumerate([1_000_003, 4_097]):
        rs = np.random.default_rng(100 + trial)
        b = torch.from_numpy(rs.choice([2, 4, 8], J, p=[0.25, 0.5, 0.25]).astype(np.uint8)).cuda()
        ref = torch.empty(J, dtype=torch.int32, device="cuda")
        ws = torch.empty(dq.dq_workspace_bytes(J), dtype=torch.uint8, device="cuda")
        dq.dq_reorder(b, J, ref, ws, ws.numel())
        got = torch.full((J,), -1, dtype=torch.int32, device="cuda")
        status = L.dq_reorder_static(ctypes.c_void_p(b.data_ptr()), J, ctypes.c_void_p(got.data_ptr()),
                                     ctypes.c_void_p(stream))
        assert status == dq.DQ_OK, dq.status_string(status)
        torch.cuda.synchronize()
        assert torch.equal(got, ref), f"call {trial}: {(got != ref).sum().item()} entries differ"


def test_reorder_static_at_its_maximum_size():
    """n_sg = DQ_REORDER_STATIC_MAX_SG uses the last tile slot of the fixed
    array; the result must still match dq_reorder."""
    L = dq.lib()
    J = dq.REORDER_STATIC_MAX_SG
    rs = np.random.default_rng(7)
    b = torch.from_numpy(rs.choice([2, 4, 8], J, p=[0.3, 0.4, 0.3]).astype(np.uint8)).cuda()
    ref = torch.empty(J, dtype=torch.int32, device="cuda")
    ws = torch.empty(dq.dq_workspace_bytes(J), dtype=torch.uint8, device="cuda")
    dq.dq_reorder(b, J, ref, ws, ws.numel())
    got = torch.full((J,), -1, dtype=torch.int32, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    status = L.dq_reorder_static(ctypes.c_void_p(b.data_ptr()), J, ctypes.c_void_p(got.data_ptr()),
                                 ctypes.c_void_p(stream))
    assert status == dq.DQ_OK, dq.status_string(status)
    torch.cuda.synchronize()
    assert torch.equal(got, ref)


def test_reorder_static_rejects_sizes_above_its_maximum():
    L = dq.lib()
    too_big = dq.REORDER_STATIC_MAX_SG + 1
    status = L.dq_reorder_static(ctypes.c_void_p(4096), too_big, ctypes.c_void_p(4096), None)
    assert status == dq.DQ_ERR_INVALID_ARG

"""Bounded waits of the per-call kernels: a wait that runs out is reported, not hidden.

The streaming output projection, the tcgen05 path of nt_ternary_gemm and the prefill GEMM wait
on copies in flight with a time limit. With the test hook nt_set_test_fault their producers
issue no copies, so the consumers' waits run out after a short limit (no GPU fault: every wait
gives up, the CTAs drain and free what they hold, the context stays usable). Checked: the
workspace's status header reports NT_ERR_TIMEOUT, the output projection writes -1 as the
arg-max, the error stays until the workspace is zero-filled, and the same workspace gives the
oracle's results afterwards.
"""
import numpy as np
import pytest
import torch

import oracle
from packed_weight_gemv_gb300 import nt
from synth import workloads as wl
from tests._gpu import DEV, assert_close, dev, host, tiled

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def fault_off():
    torch.cuda.set_device(DEV)
    nt.nt_device_check()
    yield
    nt.nt_set_test_fault(0)


def _head(seed, V=5003, K=4096):
    h = wl.head(V=V, K=K, B=1, seed=seed, workload=15)
    q, s = oracle.quantize(h.x)
    want_logits, want_am, _ = oracle.logits_argmax(h.T, h.s_T, V, K, q, s)
    return h, (dev(h.T), dev(h.s_T), dev(q), dev(s)), want_logits, want_am


def test_output_projection_timeout_is_reported_until_cleared():
    h, (T, s_T, q, s), want_logits, want_am = _head(31)
    V, K = h.V, h.K
    ws = torch.zeros(nt.nt_int8_logits_workspace_size(V, K, 1), dtype=torch.uint8, device=DEV)
    logits = torch.empty((1, V), device=DEV)
    am = torch.full((1,), 7, dtype=torch.int32, device=DEV)
    nt.nt_set_test_fault(1, 20.0)
    nt.nt_int8_logits_argmax(T, s_T, V, K, q, s, 1, logits, am, ws)
    torch.cuda.synchronize()
    nt.nt_set_test_fault(0)
    assert int(host(am)[0]) == -1
    assert nt.nt_workspace_status(ws) == nt.NT_ERR_TIMEOUT
    am.fill_(7)  # the error stays: the next call on this workspace does no work
    nt.nt_int8_logits_argmax(T, s_T, V, K, q, s, 1, logits, am, ws)
    torch.cuda.synchronize()
    assert int(host(am)[0]) == -1 and nt.nt_workspace_status(ws) == nt.NT_ERR_TIMEOUT
    ws.zero_()  # cleared, the same workspace serves correct calls again, twice in a row
    for _ in range(2):
        nt.nt_int8_logits_argmax(T, s_T, V, K, q, s, 1, logits, am, ws)
        torch.cuda.synchronize()
        assert_close(host(logits), want_logits, "logits after the workspace was cleared")
        assert np.array_equal(host(am), want_am)
        assert nt.nt_workspace_status(ws) == nt.NT_OK


def test_noalloc_timeout_shows_as_minus_one_then_recovers():
    h, (T, s_T, q, s), want_logits, want_am = _head(32)
    logits = torch.empty((1, h.V), device=DEV)
    am = torch.full((1,), 7, dtype=torch.int32, device=DEV)
    nt.nt_set_test_fault(1, 20.0)
    nt.nt_int8_logits_argmax_noalloc(T, s_T, h.V, h.K, q, s, 1, logits, am)
    torch.cuda.synchronize()
    nt.nt_set_test_fault(0)
    assert int(host(am)[0]) == -1
    nt.nt_int8_logits_argmax_noalloc(T, s_T, h.V, h.K, q, s, 1, logits, am)  # clears its own scratch
    torch.cuda.synchronize()
    assert_close(host(logits), want_logits, "no-alloc logits after a timeout")
    assert np.array_equal(host(am), want_am)


@pytest.mark.parametrize("fault,B", [(2, 8), (3, 128)])
def test_tensor_core_gemm_timeout_is_reported_until_cleared(fault, B):
    # fault 2: the tcgen05 path (2..16 vectors with a workspace); fault 3: the prefill GEMM
    N, K = 512, 2048
    p = wl.projection(16, 3, fault, N, K, B, seed=33)
    q, s = oracle.quantize(p.x)
    acc, y, _ = oracle.gemm(p.w_plain, p.s_w, N, K, q, s)
    w, s_w, qd, sd = tiled(p.w_plain, N, K), dev(p.s_w), dev(q), dev(s)
    ws = torch.zeros(nt.nt_ternary_gemm_workspace_size(N, K, B, nt.NT_LAYOUT_TILED), dtype=torch.uint8, device=DEV)
    assert ws.numel() > 0
    gy = torch.empty((B, N), device=DEV)
    gacc = torch.empty((B, N), dtype=torch.int32, device=DEV)
    nt.nt_set_test_fault(fault, 20.0)
    nt.nt_ternary_gemm(w, nt.NT_LAYOUT_TILED, s_w, N, K, qd, sd, B, gy, gacc, ws)
    torch.cuda.synchronize()
    nt.nt_set_test_fault(0)
    assert nt.nt_workspace_status(ws) == nt.NT_ERR_TIMEOUT
    ws.zero_()
    nt.nt_ternary_gemm(w, nt.NT_LAYOUT_TILED, s_w, N, K, qd, sd, B, gy, gacc, ws)
    torch.cuda.synchronize()
    assert nt.nt_workspace_status(ws) == nt.NT_OK
    assert np.array_equal(host(gacc), acc)
    assert_close(host(gy), y, "after the workspace was cleared")


def test_fault_hook_rejects_unknown_codes():
    with pytest.raises(nt.NtError) as e:
        nt.nt_set_test_fault(4, 1.0)
    assert e.value.status == nt.NT_ERR_INVALID_ARG

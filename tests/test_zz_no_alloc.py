"""The allocation-free output projection (nt_int8_logits_argmax_noalloc) against the regular
call with a caller workspace, through the C ABI, on two calls in a row.

That entry point is for callers that cannot allocate device memory (their host owns every
allocation, or they must not risk cudaMalloc's device synchronization); it keeps its scratch
in a fixed array of the library's device globals. Two consecutive calls on different inputs
check that the scratch left by the first call does not leak into the second. This file is
named to be collected last.
"""
import numpy as np
import pytest
import torch

from packed_weight_gemv_gb300 import nt
from synth import workloads as wl
from tests._gpu import DEV, assert_close, dev, host

pytestmark = pytest.mark.gpu


def _inputs(seed, V, K, B):
    h = wl.head(V=V, K=K, B=B, seed=seed, workload=14)
    q = torch.empty((B, K), dtype=torch.int8, device=DEV)
    s = torch.empty(B, dtype=torch.float32, device=DEV)
    nt.nt_quantize_act(dev(h.x), q, s)
    return dev(h.T), dev(h.s_T), q, s


def _with_workspace(T, s_T, V, K, q, s, B):
    logits = torch.empty((B, V), device=DEV)
    am = torch.empty(B, dtype=torch.int32, device=DEV)
    ws = torch.zeros(nt.nt_int8_logits_workspace_size(V, K, B), dtype=torch.uint8, device=DEV)
    nt.nt_int8_logits_argmax(T, s_T, V, K, q, s, B, logits, am, ws)
    return host(logits), host(am)


def test_noalloc_matches_workspace_call_twice():
    torch.cuda.set_device(DEV)
    V, K = 20011, 4096
    for call, (seed, B) in enumerate([(21, 3), (22, 1)]):
        T, s_T, q, s = _inputs(seed, V, K, B)
        want_logits, want_am = _with_workspace(T, s_T, V, K, q, s, B)
        logits = torch.full((B, V), float("nan"), device=DEV)
        am = torch.full((B,), -1, dtype=torch.int32, device=DEV)
        nt.nt_int8_logits_argmax_noalloc(T, s_T, V, K, q, s, B, logits, am)
        torch.cuda.synchronize()
        assert_close(host(logits), want_logits, f"no-alloc call {call + 1} logits")
        assert np.array_equal(host(am), want_am), f"no-alloc call {call + 1} arg-max"


def test_noalloc_rejects_batch_beyond_scratch():
    torch.cuda.set_device(DEV)
    V, K, B = 64, 64, 17
    T = torch.zeros((V, K), dtype=torch.int8, device=DEV)
    q = torch.zeros((B, K), dtype=torch.int8, device=DEV)
    with pytest.raises(nt.NtError) as e:
        nt.nt_int8_logits_argmax_noalloc(T, torch.ones(V, device=DEV), V, K, q,
                                         torch.ones(B, device=DEV), B, None,
                                         torch.empty(B, dtype=torch.int32, device=DEV))
    assert e.value.status == nt.NT_ERR_INVALID_ARG

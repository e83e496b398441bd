"""The allocation-free output projection (nt_int8_logits_argmax_noalloc) through the C ABI,
against the oracle and against the regular call with a caller workspace, over several calls in
a row.

That entry point is for callers that cannot allocate device memory (their host owns every
allocation, or they must not risk cudaMalloc's device synchronization); it keeps its scratch
in a fixed array of the library's device globals, sized for 16 vectors. The calls run the
largest batch the array serves twice, then one vector twice (the streaming kernel), then a
small batch, each on new inputs, so every kernel that uses the array runs on what the previous
call of the same kernel left there. This file is named to be collected last.
"""
import numpy as np
import pytest
import torch

import oracle
from packed_weight_gemv_gb300 import nt
from synth import workloads as wl
from tests._gpu import DEV, assert_close, dev, host

pytestmark = pytest.mark.gpu


def _with_workspace(T, s_T, V, K, q, s, B):
    logits = torch.empty((B, V), device=DEV)
    am = torch.empty(B, dtype=torch.int32, device=DEV)
    ws = torch.zeros(nt.nt_int8_logits_workspace_size(V, K, B), dtype=torch.uint8, device=DEV)
    nt.nt_int8_logits_argmax(T, s_T, V, K, q, s, B, logits, am, ws)
    return host(logits), host(am)


def test_noalloc_matches_oracle_over_calls_in_a_row():
    torch.cuda.set_device(DEV)
    V, K = 20011, 4096
    for call, (seed, B) in enumerate([(21, 16), (22, 16), (23, 1), (24, 1), (25, 3)]):
        h = wl.head(V=V, K=K, B=B, seed=seed, workload=14)
        q, s = oracle.quantize(h.x)
        want_logits, want_am, _ = oracle.logits_argmax(h.T, h.s_T, V, K, q, s)
        T, s_T, qd, sd = dev(h.T), dev(h.s_T), dev(q), dev(s)
        logits = torch.full((B, V), float("nan"), device=DEV)
        am = torch.full((B,), -2, dtype=torch.int32, device=DEV)
        nt.nt_int8_logits_argmax_noalloc(T, s_T, V, K, qd, sd, B, logits, am)
        torch.cuda.synchronize()
        what = f"no-alloc call {call + 1} (B={B})"
        assert_close(host(logits), want_logits, what + " logits")
        assert np.array_equal(host(am), want_am), what + " arg-max"
        ws_logits, ws_am = _with_workspace(T, s_T, V, K, qd, sd, B)
        assert np.array_equal(host(logits), ws_logits) and np.array_equal(host(am), ws_am), what


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

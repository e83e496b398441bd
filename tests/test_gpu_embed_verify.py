"""GPU parity of the input-table row gather and the verify-pass acceptance, standalone and
inside a decode plan, against the CPU oracle on the same seeded inputs. The gathered rows
and every arg-max / emitted token must match bit for bit."""
import numpy as np
import pytest
import torch

import oracle
from packed_weight_gemv_gb300 import nt
from synth import workloads as wl
from tests._gpu import DEV, assert_close, dev, host, plan_inputs

pytestmark = pytest.mark.gpu

SMALL = {"q": (512, 512), "k": (128, 512), "v": (128, 512), "o": (512, 512),
         "gate": (1536, 512), "up": (1536, 512), "down": (512, 1536)}


@pytest.fixture(scope="module", autouse=True)
def device():
    torch.cuda.set_device(DEV)
    nt.nt_device_check()


# ---- input-table row gather --------------------------------------------------------------

@pytest.mark.parametrize("V,K,B", [(5000, 512, 1), (3001, 4096, 7), (100, 16, 16), (2048, 1040, 33),
                                   (151936, 4096, 16)])
def test_embed_rows(V, K, B):
    e = wl.embedding(V, K, B, seed=2)
    x = torch.full((B, K), float("nan"), device=DEV)
    bad = torch.zeros(1, dtype=torch.int32, device=DEV)
    nt.nt_embed_rows(dev(e.T), dev(e.s_T), V, K, dev(e.tokens), B, x, bad)
    want, nbad = oracle.embed_rows(e.T, e.s_T, V, K, e.tokens)
    assert np.array_equal(host(x).view(np.uint32), want.view(np.uint32))
    assert int(bad.item()) == nbad == 0


def test_embed_rows_out_of_range_tokens_are_zero_and_counted():
    V, K = 777, 256
    e = wl.embedding(V, K, 6, seed=3)
    tok = e.tokens.copy()
    tok[[1, 3, 4]] = [-1, V, np.iinfo(np.int32).max]
    tok[5] = V - 1  # the last row is valid
    x = torch.full((6, K), float("nan"), device=DEV)
    bad = torch.full((1,), 5, dtype=torch.int32, device=DEV)  # the call adds to the counter
    nt.nt_embed_rows(dev(e.T), dev(e.s_T), V, K, dev(tok), 6, x, bad)
    want, nbad = oracle.embed_rows(e.T, e.s_T, V, K, tok)
    assert nbad == 3 and int(bad.item()) == 5 + 3
    assert np.array_equal(host(x).view(np.uint32), want.view(np.uint32))
    assert not host(x)[[1, 3, 4]].any()


def test_embed_rows_rejects_bad_arguments():
    T = torch.zeros((4, 24), dtype=torch.int8, device=DEV)
    s = torch.ones(4, device=DEV)
    tok = torch.zeros(1, dtype=torch.int32, device=DEV)
    x = torch.empty((1, 24), device=DEV)
    with pytest.raises(nt.NtError) as ei:
        nt.nt_embed_rows(T, s, 4, 24, tok, 1, x)  # K not a multiple of 16
    assert ei.value.status == nt.NT_ERR_INVALID_ARG
    xb = torch.empty(40, device=DEV)
    with pytest.raises(nt.NtError) as ei:
        nt.nt_embed_rows(T, s, 4, 16, tok, 1, xb[1:17])  # x 4 bytes past a 16-byte boundary
    assert ei.value.status == nt.NT_ERR_ALIGNMENT


# ---- verify-pass acceptance ------------------------------------------------------------

@pytest.mark.parametrize("B", [1, 2, 5, 16])
def test_verify_accept_every_prefix(B):
    greedy = (wl.embedding(1000, 16, B, seed=B).tokens + 1).astype(np.int32)
    for n_agree in range(B):
        draft = wl.draft_tokens(greedy, n_agree, 1000, seed=B)
        emit = torch.full((B,), -1, dtype=torch.int32, device=DEV)
        n = torch.zeros(1, dtype=torch.int32, device=DEV)
        nt.nt_verify_accept(dev(draft) if B > 1 else None, dev(greedy), B, emit, n)
        want = oracle.verify_accept(draft, greedy)
        assert int(n.item()) == want.size == n_agree + 1
        got = host(emit)
        assert np.array_equal(got[:want.size], want)
        assert (got[want.size:] == -1).all()  # nothing written past the emitted tokens


# ---- inside a decode plan ----------------------------------------------------------------

@pytest.mark.parametrize("launcher", [nt.NT_LAUNCH_PERSISTENT, nt.NT_LAUNCH_GRAPH, nt.NT_LAUNCH_STREAM])
@pytest.mark.parametrize("mode", [nt.NT_STEP_INDEPENDENT, nt.NT_STEP_ORDERED])
@pytest.mark.parametrize("B", [1, 3])
def test_decode_step_embed_feeds_first_layer(launcher, mode, B):
    # Layer 0's q, k and v quantize the gathered rows inside the same step.
    projs = wl.decoder_projections(2, SMALL, B=B, seed=9, workload=20)
    e = wl.embedding(4099, 512, B, seed=9)
    dp, _ = plan_inputs(projs, None, B=B)
    ex = torch.full((B, 512), float("nan"), device=DEV)
    for d in dp[:3]:
        d["x"] = ex
    emb = dict(T=dev(e.T), s=dev(e.s_T), V=e.V, K=e.K, tokens=dev(e.tokens), x=ex)
    plan = nt.DecodePlan(2, B, dp, None, mode, launcher, embed=emb)
    for _ in range(2):
        plan.nt_decode_step()
    torch.cuda.synchronize()
    assert plan.nt_decode_step_status() == nt.NT_OK
    xe, _ = oracle.embed_rows(e.T, e.s_T, e.V, e.K, e.tokens)
    assert np.array_equal(host(ex).view(np.uint32), xe.view(np.uint32))
    for i, (p, d) in enumerate(zip(projs, dp)):
        q, s = oracle.quantize(xe if i < 3 else p.x[:B])
        assert np.array_equal(host(d["q"]), q), p.name
        _, y, _ = oracle.gemm(p.w_plain, p.s_w, p.N, p.K, q, s)
        assert_close(host(d["y"]), y, p.name)
    plan.close()


@pytest.mark.parametrize("launcher", [nt.NT_LAUNCH_PERSISTENT, nt.NT_LAUNCH_GRAPH, nt.NT_LAUNCH_STREAM])
@pytest.mark.parametrize("B,n_agree", [(1, 0), (5, 0), (5, 2), (5, 4), (16, 9)])
def test_decode_step_verify_pass(launcher, B, n_agree):
    # One batched verify pass: the head scores B positions and the step keeps the longest
    # prefix of drafts that agrees with its arg-max.
    projs = wl.decoder_projections(1, SMALL, B=B, seed=10, workload=21)
    head = wl.head(V=2003, K=512, B=B, seed=10, workload=21)
    dp, hd = plan_inputs(projs, head, B=B)
    qh, sh = oracle.quantize(head.x[:B])
    _, greedy, _ = oracle.logits_argmax(head.T, head.s_T, head.V, head.K, qh, sh)
    greedy = np.asarray(greedy, dtype=np.int32)
    draft = wl.draft_tokens(greedy, n_agree, head.V, seed=10)
    emit = torch.full((B,), -1, dtype=torch.int32, device=DEV)
    n = torch.zeros(1, dtype=torch.int32, device=DEV)
    ver = dict(draft=dev(draft) if B > 1 else None, emit=emit, n=n)
    plan = nt.DecodePlan(1, B, dp, hd, nt.NT_STEP_INDEPENDENT, launcher, verify=ver)
    for _ in range(2):
        plan.nt_decode_step()
    torch.cuda.synchronize()
    assert plan.nt_decode_step_status() == nt.NT_OK
    assert np.array_equal(host(hd["argmax"]), greedy)
    want = oracle.verify_accept(draft, greedy)
    assert int(n.item()) == want.size == n_agree + 1
    assert np.array_equal(host(emit)[:want.size], want)
    plan.close()


def test_decode_plan_verify_needs_head():
    projs = wl.decoder_projections(1, SMALL, B=2, seed=11, workload=22)
    dp, _ = plan_inputs(projs, None, B=2)
    ver = dict(draft=torch.zeros(1, dtype=torch.int32, device=DEV),
               emit=torch.zeros(2, dtype=torch.int32, device=DEV), n=torch.zeros(1, dtype=torch.int32, device=DEV))
    with pytest.raises(nt.NtError) as ei:
        nt.DecodePlan(1, 2, dp, None, verify=ver)
    assert ei.value.status == nt.NT_ERR_INVALID_ARG

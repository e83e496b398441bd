"""GPU parity of chained decode steps (every stage quantizes the previous stages' outputs)
against the oracle's chained step on the same seeded inputs: every projection's int8 codes
and scale bit for bit, every output within 1e-6 relative, the output projection's arg-max
exactly -- on all three launchers, one and several vectors (several passes per stage on the
persistent kernel above 4 vectors), and with the first hidden state gathered from the input
table inside the step."""
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
LAUNCHERS = [nt.NT_LAUNCH_PERSISTENT, nt.NT_LAUNCH_GRAPH, nt.NT_LAUNCH_STREAM]


@pytest.fixture(scope="module", autouse=True)
def device():
    torch.cuda.set_device(DEV)
    nt.nt_device_check()


def oracle_layers(projs, n_layers):
    return [[(p.w_plain, p.s_w, p.N, p.K) for p in projs[7 * l:7 * l + 7]] for l in range(n_layers)]


def check_chain(projs, head, dp, hd, want):
    for i, (p, d) in enumerate(zip(projs, dp)):
        assert np.array_equal(host(d["q"]), want["q"][i]), p.name
        assert np.array_equal(host(d["s_x"]), want["s"][i]), p.name
        assert_close(host(d["y"]), want["y"][i], p.name)
    if head is not None:
        assert np.array_equal(host(hd["q"]), want["head_q"])
        assert np.array_equal(host(hd["sx"]), want["head_s"])
        assert_close(host(hd["logits"]), want["logits"], "head")
        assert np.array_equal(host(hd["argmax"]), want["argmax"])


@pytest.mark.parametrize("launcher", LAUNCHERS)
@pytest.mark.parametrize("B", [1, 3, 6])
def test_chained_step_small(launcher, B):
    L = 3
    projs = wl.decoder_projections(L, SMALL, B=B, seed=12, workload=30)
    head = wl.head(V=3001, K=512, B=B, seed=12, workload=30)
    dp, hd = plan_inputs(projs, head, B=B)
    plan = nt.DecodePlan(L, B, dp, hd, nt.NT_STEP_CHAINED, launcher)
    for _ in range(3):  # repeated steps: the residual stream starts from the input every step
        plan.nt_decode_step()
    torch.cuda.synchronize()
    assert plan.nt_decode_step_status() == nt.NT_OK
    want = oracle.decode_chained(oracle_layers(projs, L), projs[0].x[:B],
                                 (head.T, head.s_T, head.V, head.K))
    check_chain(projs, head, dp, hd, want)
    plan.close()


@pytest.mark.parametrize("launcher", LAUNCHERS)
def test_chained_step_without_head_and_ragged_shapes(launcher):
    # K, N not multiples of 512 (ragged tails inside the persistent kernel's activation
    # buffer), two query heads per key-value head of 64 dimensions
    shapes = {"q": (256, 320), "k": (128, 320), "v": (128, 320), "o": (320, 256),
              "gate": (784, 320), "up": (784, 320), "down": (320, 784)}
    L, B = 2, 2
    projs = wl.decoder_projections(L, shapes, B=B, seed=13, workload=31)
    dp, _ = plan_inputs(projs, None, B=B)
    plan = nt.DecodePlan(L, B, dp, None, nt.NT_STEP_CHAINED, launcher, head_dim=64)
    plan.nt_decode_step()
    torch.cuda.synchronize()
    assert plan.nt_decode_step_status() == nt.NT_OK
    want = oracle.decode_chained(oracle_layers(projs, L), projs[0].x[:B], None, head_dim=64)
    check_chain(projs, None, dp, None, want)
    plan.close()


@pytest.mark.parametrize("launcher", LAUNCHERS)
def test_chained_step_from_gathered_rows(launcher):
    L, B = 2, 3
    projs = wl.decoder_projections(L, SMALL, B=B, seed=14, workload=32)
    head = wl.head(V=1999, K=512, B=B, seed=14, workload=32)
    e = wl.embedding(4001, 512, B, seed=14)
    dp, hd = plan_inputs(projs, head, B=B)
    ex = torch.full((B, 512), float("nan"), device=DEV)
    dp[0]["x"] = ex
    emb = dict(T=dev(e.T), s=dev(e.s_T), V=e.V, K=e.K, tokens=dev(e.tokens), x=ex)
    plan = nt.DecodePlan(L, B, dp, hd, nt.NT_STEP_CHAINED, launcher, embed=emb)
    plan.nt_decode_step()
    torch.cuda.synchronize()
    assert plan.nt_decode_step_status() == nt.NT_OK
    x0, _ = oracle.embed_rows(e.T, e.s_T, e.V, e.K, e.tokens)
    want = oracle.decode_chained(oracle_layers(projs, L), x0, (head.T, head.s_T, head.V, head.K))
    check_chain(projs, head, dp, hd, want)
    plan.close()


def test_chained_step_8b_shapes_two_layers():
    # the 8B-shaped layer: 32 query heads, 8 key-value heads of 128 dimensions, K up to 12288
    L = 2
    projs = wl.decoder_projections(L, seed=15, workload=33)
    head = wl.head(V=20000, K=4096, seed=15, workload=33)
    dp, hd = plan_inputs(projs, head)
    plan = nt.DecodePlan(L, 1, dp, hd, nt.NT_STEP_CHAINED, nt.NT_LAUNCH_PERSISTENT)
    plan.nt_decode_step()
    torch.cuda.synchronize()
    assert plan.nt_decode_step_status() == nt.NT_OK
    want = oracle.decode_chained(oracle_layers(projs, L), projs[0].x[:1], (head.T, head.s_T, head.V, head.K))
    check_chain(projs, head, dp, hd, want)
    plan.close()


def test_chained_plan_rejects_mismatched_shapes():
    shapes = dict(SMALL, o=(512, 256))  # o.K != q.N
    projs = wl.decoder_projections(1, shapes, seed=16, workload=34)
    dp, _ = plan_inputs(projs, None)
    with pytest.raises(nt.NtError) as ei:
        nt.DecodePlan(1, 1, dp, None, nt.NT_STEP_CHAINED)
    assert ei.value.status == nt.NT_ERR_INVALID_ARG

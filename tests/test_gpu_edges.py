"""GPU parity at the full decode size and at the edges: the 8B-shaped step in the launch
configuration bench.py times (every output against the oracle), zero inputs, ragged rows in a
plan, long reductions, and the persistent launcher's size limit."""
import numpy as np
import pytest
import torch

import oracle
import synth
from packed_weight_gemv_gb300 import nt
from synth import workloads as wl
from tests._gpu import DEV, assert_close, dev, host, plan_inputs, tiled

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def device():
    torch.cuda.set_device(DEV)
    nt.nt_device_check()


def test_decode_step_8b_full_every_output():
    # 36 layers x 7 projections + the 151,936 x 4,096 table, persistent launcher, independent
    # mode, inputs quantized in the step: the configuration of the benchmark's timed steps.
    projs = wl.decoder_projections()
    head = wl.head()
    dp, hd = plan_inputs(projs, head)
    plan = nt.DecodePlan(36, 1, dp, hd, nt.NT_STEP_INDEPENDENT, nt.NT_LAUNCH_PERSISTENT)
    for _ in range(2):
        plan.nt_decode_step()
    torch.cuda.synchronize()
    assert plan.nt_decode_step_status() == nt.NT_OK
    for p, d in zip(projs, dp):
        q, s = oracle.quantize(p.x)
        assert np.array_equal(host(d["q"])[0], q[0]) and host(d["s_x"])[0] == s[0], p.name
        _, y, _ = oracle.gemv(p.w_plain, p.s_w, p.N, p.K, q[0], s)
        assert_close(host(d["y"])[0], y, p.name)
    q, s = oracle.quantize(head.x)
    logits, am, _ = oracle.logits_argmax(head.T, head.s_T, head.V, head.K, q, s)
    assert_close(host(hd["logits"]), logits, "head")
    assert int(host(hd["argmax"])[0]) == int(am[0])
    plan.close()


def test_decode_step_8b_full_ordered_every_output():
    # the same 36-layer step with a grid barrier before every stage (the ordered mode the
    # benchmark's breakdown times): every projection and the full table against the oracle
    projs = wl.decoder_projections()
    head = wl.head()
    dp, hd = plan_inputs(projs, head)
    plan = nt.DecodePlan(36, 1, dp, hd, nt.NT_STEP_ORDERED, nt.NT_LAUNCH_PERSISTENT)
    for _ in range(2):
        plan.nt_decode_step()
    torch.cuda.synchronize()
    assert plan.nt_decode_step_status() == nt.NT_OK
    for p, d in zip(projs, dp):
        q, s = oracle.quantize(p.x)
        assert np.array_equal(host(d["q"])[0], q[0]) and host(d["s_x"])[0] == s[0], p.name
        _, y, _ = oracle.gemv(p.w_plain, p.s_w, p.N, p.K, q[0], s)
        assert_close(host(d["y"])[0], y, p.name)
    q, s = oracle.quantize(head.x)
    logits, am, _ = oracle.logits_argmax(head.T, head.s_T, head.V, head.K, q, s)
    assert_close(host(hd["logits"]), logits, "head")
    assert int(host(hd["argmax"])[0]) == int(am[0])
    plan.close()


def test_decode_step_8b_full_chained_every_output():
    # 36 chained layers of the 8B shape and the full table: every stage quantizes what the
    # previous stages produced, so the whole trajectory is compared with the oracle's chained
    # step -- every stage's codes and scale bit for bit, every output within 1e-6
    L = wl.DECODER_8B_LAYERS
    projs = wl.decoder_projections()
    head = wl.head()
    # Without normalisation the gated product squares the hidden state's size every layer; an
    # input of about 1e-4 grows by ~1.3x per layer and stays finite through all 36 (the
    # quantizer is scale-free, so the codes still use the full int8 range at every stage)
    projs[0].x *= np.float32(1e-4)
    dp, hd = plan_inputs(projs, head)
    plan = nt.DecodePlan(L, 1, dp, hd, nt.NT_STEP_CHAINED, nt.NT_LAUNCH_PERSISTENT)
    for _ in range(2):  # the residual stream starts from the supplied input every step
        plan.nt_decode_step()
    torch.cuda.synchronize()
    assert plan.nt_decode_step_status() == nt.NT_OK
    layers = [[(p.w_plain, p.s_w, p.N, p.K) for p in projs[7 * l:7 * l + 7]] for l in range(L)]
    want = oracle.decode_chained(layers, projs[0].x[:1], (head.T, head.s_T, head.V, head.K))
    assert all(np.isfinite(h).all() and np.abs(h).max() < 1e6 for h in want["h"])
    assert all(np.abs(q).max() == 127 for q in want["q"])  # every stage uses the full code range
    for i, (p, d) in enumerate(zip(projs, dp)):
        assert np.array_equal(host(d["q"]), want["q"][i]), p.name
        assert np.array_equal(host(d["s_x"]), want["s"][i]), p.name
        assert_close(host(d["y"]), want["y"][i], p.name)
    assert np.array_equal(host(hd["q"]), want["head_q"])
    assert np.array_equal(host(hd["sx"]), want["head_s"])
    assert_close(host(hd["logits"]), want["logits"], "head")
    assert np.array_equal(host(hd["argmax"]), want["argmax"])
    plan.close()


def test_zero_inputs_give_positive_zero_and_argmax_zero():
    shapes = {"q": (64, 512), "k": (16, 512), "v": (16, 512), "o": (64, 512),
              "gate": (128, 512), "up": (128, 512), "down": (64, 1024)}
    projs = wl.decoder_projections(1, shapes, seed=3, workload=17)
    head = wl.head(V=777, K=512, seed=3, workload=17)
    for p in projs:
        p.x[:] = 0
    head.x[:] = 0
    dp, hd = plan_inputs(projs, head)
    plan = nt.DecodePlan(1, 1, dp, hd, nt.NT_STEP_ORDERED, nt.NT_LAUNCH_PERSISTENT)
    plan.nt_decode_step()
    torch.cuda.synchronize()
    for d in dp:
        y = host(d["y"])
        assert (y == 0).all() and not np.signbit(y).any()
        assert (host(d["s_x"]) == 0).all()
    assert (host(hd["logits"]) == 0).all() and int(host(hd["argmax"])[0]) == 0
    plan.close()


@pytest.mark.parametrize("launcher", [nt.NT_LAUNCH_PERSISTENT, nt.NT_LAUNCH_GRAPH])
def test_plan_with_ragged_rows_and_k(launcher):
    # N not a multiple of 4 (padded rows of the tiled layout), K not a multiple of 512.
    shapes = {"q": (130, 528), "k": (33, 528), "v": (7, 528), "o": (130, 1040),
              "gate": (257, 528), "up": (257, 528), "down": (130, 1552)}
    projs = wl.decoder_projections(2, shapes, seed=4, workload=18)
    head = wl.head(V=1001, K=528, seed=4, workload=18)
    dp, hd = plan_inputs(projs, head)
    plan = nt.DecodePlan(2, 1, dp, hd, nt.NT_STEP_ORDERED, launcher)
    plan.nt_decode_step()
    torch.cuda.synchronize()
    for p, d in zip(projs, dp):
        q, s = oracle.quantize(p.x)
        _, y, _ = oracle.gemv(p.w_plain, p.s_w, p.N, p.K, q[0], s)
        assert_close(host(d["y"])[0], y, p.name)
    q, s = oracle.quantize(head.x)
    _, am, _ = oracle.logits_argmax(head.T, head.s_T, head.V, head.K, q, s)
    assert int(host(hd["argmax"])[0]) == int(am[0])
    plan.close()


@pytest.mark.parametrize("K", [49152, 65536])
def test_long_reduction_per_call(K):
    N = 64
    p = wl.projection(19, 0, 0, N, K, 1, seed=5)
    q, s = oracle.quantize(p.x)
    acc, y, _ = oracle.gemv(p.w_plain, p.s_w, N, K, q[0], s)
    for layout in (nt.NT_LAYOUT_PLAIN, nt.NT_LAYOUT_TILED):
        w = dev(p.w_plain) if layout == nt.NT_LAYOUT_PLAIN else tiled(p.w_plain, N, K)
        gy = torch.empty(N, device=DEV)
        gacc = torch.empty(N, dtype=torch.int32, device=DEV)
        nt.nt_ternary_gemv(w, layout, dev(p.s_w), N, K, dev(q), dev(s), gy, gacc)
        assert np.array_equal(host(gacc), acc)
        assert_close(host(gy), y, f"K={K}")


def test_persistent_plan_rejects_activations_beyond_shared_memory():
    # K = 49152 still fits the persistent kernel (2 ring slots); K = 65536 does not.
    shapes = {n: (16, 512) for n in wl.PROJ_NAMES}
    shapes["down"] = (16, 65536)
    projs = wl.decoder_projections(1, shapes, seed=6, workload=20)
    dp, _ = plan_inputs(projs, None)
    with pytest.raises(nt.NtError) as e:
        nt.DecodePlan(1, 1, dp, None, nt.NT_STEP_INDEPENDENT, nt.NT_LAUNCH_PERSISTENT)
    assert e.value.status == nt.NT_ERR_INVALID_ARG
    plan = nt.DecodePlan(1, 1, dp, None, nt.NT_STEP_INDEPENDENT, nt.NT_LAUNCH_GRAPH)
    plan.nt_decode_step()
    torch.cuda.synchronize()
    p, d = projs[-1], dp[-1]
    q, s = oracle.quantize(p.x)
    _, y, _ = oracle.gemv(p.w_plain, p.s_w, p.N, p.K, q[0], s)
    assert_close(host(d["y"])[0], y, "down K=65536 (graph launcher)")
    plan.close()


def test_trace_timeline_is_ordered():
    projs = wl.decoder_projections(2, {"q": (256, 512), "k": (64, 512), "v": (64, 512),
                                       "o": (256, 512), "gate": (512, 512), "up": (512, 512),
                                       "down": (256, 1024)}, seed=7, workload=21)
    dp, _ = plan_inputs(projs, None)
    plan = nt.DecodePlan(2, 1, dp, None, nt.NT_STEP_ORDERED, nt.NT_LAUNCH_PERSISTENT)
    G, S = plan.nt_decode_plan_trace_layout()
    assert G > 0 and S == 1 + 4 * 2 - 1  # quantize barrier + 7 stage barriers
    tr = torch.zeros(G * (S + 1) * 4, dtype=torch.int64, device=DEV)
    plan.nt_decode_plan_set_trace(tr)
    plan.nt_decode_step()
    torch.cuda.synchronize()
    t = host(tr).reshape(G, S + 1, 4)
    for c in range(G):
        assert t[c, 0, 0] > 0 and t[c, 0, 1] >= t[c, 0, 0]
        for b in range(1, S + 1):
            assert t[c, 0, 0] <= t[c, b, 0] <= t[c, b, 1] <= t[c, b, 2] <= t[c, 0, 1]
    # every CTA leaves barrier b only after the last CTA reached it
    for b in range(1, S + 1):
        assert t[:, b, 1].min() >= t[:, b, 0].max()
    plan.close()

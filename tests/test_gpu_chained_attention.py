"""GPU parity of chained steps with the attention side (RMS norms, rotary embedding and
cache append, attention over the cache, SiLU gate) against the oracle's float64 layer on the
same seeded inputs, on the stream, graph and persistent launchers (the persistent launcher runs
one cooperative launch per segment of stages between two attention sides).

The kernels compute norms, rotations, attention and SiLU in fp32 where the oracle uses float64,
so a value that lies within a rounding step of an int8 boundary can quantize one code apart.
Checked: at most 0.2 % of any projection's codes differ and none by more than 1; scales and
outputs within 2e-3 of the projection's largest output; appended cache rows within one bf16
step (plus the upstream tolerance); the output projection's arg-max wherever the oracle's top two logits are more than 1e-2
(relative to the largest) apart."""
import numpy as np
import pytest
import torch

import oracle
import synth
from oracle import layer_ops as lo
from packed_weight_gemv_gb300 import nt
from synth import workloads as wl
from tests._gpu import DEV, dev, host, plan_inputs

pytestmark = pytest.mark.gpu

# 4 query heads and 2 key-value heads of 128 dimensions, hidden 512, feed-forward 1024
SHAPES = {"q": (512, 512), "k": (256, 512), "v": (256, 512), "o": (512, 512),
          "gate": (1024, 512), "up": (1024, 512), "down": (512, 1024)}


@pytest.fixture(scope="module", autouse=True)
def device():
    torch.cuda.set_device(DEV)
    nt.nt_device_check()


def close_codes(got, want, what):
    d = np.abs(got.astype(np.int32) - want.astype(np.int32))
    assert d.max() <= 1 and d.mean() <= 2e-3, f"{what}: {int((d > 0).sum())} codes differ"


def close(got, want, what, rel=2e-3):
    scale = max(float(np.abs(want).max()), 1e-30)
    err = float(np.abs(got.astype(np.float64) - want.astype(np.float64)).max())
    assert err <= rel * scale, f"{what}: max error {err:.3g} vs {rel * scale:.3g}"


@pytest.mark.parametrize("launcher", [nt.NT_LAUNCH_STREAM, nt.NT_LAUNCH_GRAPH, nt.NT_LAUNCH_PERSISTENT])
@pytest.mark.parametrize("B,pos,norms", [(1, 0, True), (1, 300, True), (3, 130, True), (2, 64, False)])
def test_chained_attention_step(launcher, B, pos, norms):
    L, Hkv, ts = 2, 2, 512
    projs = wl.decoder_projections(L, SHAPES, B=B, seed=40 + pos, workload=40)
    head = wl.head(V=2500, K=512, B=B, seed=40 + pos, workload=40)
    dp, hd = plan_inputs(projs, head, B=B)
    kb = [synth.bf16_normal(Hkv * ts * 128, pos, 10 + l).reshape(Hkv, ts, 128) for l in range(L)]
    vb = [synth.bf16_normal(Hkv * ts * 128, pos, 20 + l).reshape(Hkv, ts, 128) for l in range(L)]
    kc = [dev(k.view(np.int16)) for k in kb]
    vc = [dev(v.view(np.int16)) for v in vb]
    ga = [synth.scales(512, 1.0, pos, 30 + l) for l in range(L)]
    gf = [synth.scales(512, 1.0, pos, 40 + l) for l in range(L)]
    gz = synth.scales(512, 1.0, pos, 50)
    att = dict(k_cache=kc, v_cache=vc, t_stride=ts, pos=pos)
    if norms:
        att.update(norm_attn=[dev(g) for g in ga], norm_ffn=[dev(g) for g in gf], norm_final=dev(gz))
    plan = nt.DecodePlan(L, B, dp, hd, nt.NT_STEP_CHAINED, launcher, attention=att)
    plan.nt_decode_step()
    torch.cuda.synchronize()
    layers = [[(p.w_plain, p.s_w, p.N, p.K) for p in projs[7 * l:7 * l + 7]] for l in range(L)]
    kf = [lo.from_bf16_bits(k).copy() for k in kb]
    vf = [lo.from_bf16_bits(v).copy() for v in vb]
    want = oracle.decode_chained_attention(layers, projs[0].x[:B], (head.T, head.s_T, head.V, head.K), kf, vf, pos,
                                           ga if norms else None, gf if norms else None, gz if norms else None)
    for i, (p, d) in enumerate(zip(projs, dp)):
        close_codes(host(d["q"]), want["q"][i], p.name)
        close(host(d["s_x"]), want["s"][i], p.name + " scale")
        close(host(d["y"]), want["y"][i], p.name)
    close_codes(host(hd["q"]), want["head_q"], "head")
    close(host(hd["logits"]), want["logits"], "logits")
    lg = want["logits"].astype(np.float64)
    top2 = np.sort(lg, axis=1)[:, -2:]
    sure = (top2[:, 1] - top2[:, 0]) > 1e-2 * np.abs(lg).max(axis=1)
    assert np.array_equal(host(hd["argmax"])[sure], want["argmax"][sure])
    for l in range(L):  # appended rows: the rotated keys and the values, as bf16
        gk = lo.from_bf16_bits(host(kc[l]).view(np.uint16)[:, pos:pos + B]).astype(np.float64)
        wk = kf[l][:, pos:pos + B].astype(np.float64)
        assert np.all(np.abs(gk - wk) <= np.abs(wk) * 2.0 ** -7 * 1.01 + 2e-3 * np.abs(wk).max())
        gv = lo.from_bf16_bits(host(vc[l]).view(np.uint16)[:, pos:pos + B]).astype(np.float64)
        wv = vf[l][:, pos:pos + B].astype(np.float64)
        assert np.all(np.abs(gv - wv) <= np.abs(wv) * 2.0 ** -7 * 1.01 + 2e-3 * np.abs(wv).max())
    plan.close()


@pytest.mark.parametrize("launcher", [nt.NT_LAUNCH_GRAPH, nt.NT_LAUNCH_PERSISTENT])
def test_chained_attention_position_advances(launcher):
    L, B, Hkv, ts = 2, 1, 2, 256
    projs = wl.decoder_projections(L, SHAPES, B=B, seed=44, workload=41)
    dp, _ = plan_inputs(projs, None, B=B)
    kc = [torch.zeros((Hkv, ts, 128), dtype=torch.int16, device=DEV) for _ in range(L)]
    vc = [torch.zeros((Hkv, ts, 128), dtype=torch.int16, device=DEV) for _ in range(L)]
    att = dict(k_cache=kc, v_cache=vc, t_stride=ts, pos=0)
    plan = nt.DecodePlan(L, B, dp, None, nt.NT_STEP_CHAINED, launcher, attention=att)
    for p in range(3):  # three tokens: rows 0, 1, 2 of every layer's cache fill in order
        plan.nt_decode_plan_set_position(p)
        plan.nt_decode_step()
    torch.cuda.synchronize()
    for l in range(L):
        rows = host(kc[l]).view(np.uint16)
        assert rows[:, :3].any(axis=(0, 2)).all() and not rows[:, 3:].any()
    if launcher == nt.NT_LAUNCH_PERSISTENT:
        assert plan.nt_decode_step_status() == nt.NT_OK
    with pytest.raises(nt.NtError):
        plan.nt_decode_plan_set_position(ts)
    plan.close()

"""GPU parity of the attention-side operations against the float64 oracle on the same seeded
inputs. Tolerances follow from fp32 arithmetic: attention outputs within 3e-5 of max |v|
(128-term dot products and exp2 on scores of order 1-10, sums over <= 128 positions per chunk
plus the chunk merge), rotary outputs within 4 ulp of the largest element, RMS outputs within
4 ulp, cache entries equal to the oracle's bf16 rounding or one bf16 step away (the fp32
rotation may straddle a bf16 rounding boundary the float64 value does not)."""
import numpy as np
import pytest
import torch

import synth
from oracle import layer_ops as lo
from packed_weight_gemv_gb300 import nt
from tests._gpu import DEV, dev, host

pytestmark = pytest.mark.gpu
D = 128


@pytest.fixture(scope="module", autouse=True)
def device():
    torch.cuda.set_device(DEV)
    nt.nt_device_check()


def caches(Hkv, ts, seed):
    kb = synth.bf16_normal(Hkv * ts * D, seed, 1).reshape(Hkv, ts, D)
    vb = synth.bf16_normal(Hkv * ts * D, seed, 2).reshape(Hkv, ts, D)
    return kb, vb


def run_attention(q, kb, vb, B, Hq, Hkv, T, ts):
    out = torch.full((B, Hq, D), float("nan"), device=DEV)
    ws = torch.zeros(nt.nt_attention_workspace_size(B, Hq, Hkv, T), dtype=torch.uint8, device=DEV)
    nt.nt_attention_decode(dev(q), dev(kb.view(np.int16)), dev(vb.view(np.int16)), B, Hq, Hkv, D, T, ts, out, ws)
    return host(out)


@pytest.mark.parametrize("B,Hq,Hkv,T,ts,qscale", [
    (1, 32, 8, 1, 1, 1.0), (1, 32, 8, 127, 130, 1.0), (1, 32, 8, 128, 128, 1.0), (1, 32, 8, 129, 256, 1.0),
    (1, 32, 8, 4096, 4100, 1.0), (1, 32, 8, 3000, 3000, 4.0), (4, 32, 8, 300, 300, 1.0),
    (7, 16, 8, 1000, 1024, 2.0), (2, 8, 8, 200, 200, 1.0), (3, 8, 1, 260, 260, 1.0)])
def test_attention_decode(B, Hq, Hkv, T, ts, qscale):
    kb, vb = caches(Hkv, ts, T + B)
    q = (synth.normal(B * Hq * D, T, 3) * np.float32(qscale)).reshape(B, Hq, D)
    got = run_attention(q, kb, vb, B, Hq, Hkv, T, ts)
    want = lo.attention_decode(q, lo.from_bf16_bits(kb), lo.from_bf16_bits(vb), T)
    vmax = float(np.abs(lo.from_bf16_bits(vb[:, :T])).max())
    err = np.abs(got.astype(np.float64) - want)
    assert err.max() <= 3e-5 * vmax, f"max error {err.max()} vs bound {3e-5 * vmax}"


def test_attention_single_position_and_rejections():
    kb, vb = caches(8, 1, 99)
    q = synth.normal(32 * D, 99, 3).reshape(1, 32, D)
    got = run_attention(q, kb, vb, 1, 32, 8, 1, 1)
    for h in range(32):  # one position: the output is that position's value, exactly
        assert np.array_equal(got[0, h], lo.from_bf16_bits(vb[h // 4, 0]))
    ws = torch.empty(16, dtype=torch.uint8, device=DEV)
    out = torch.empty((1, 32, D), device=DEV)
    qd, kd, vd = dev(q), dev(kb.view(np.int16)), dev(vb.view(np.int16))
    with pytest.raises(nt.NtError) as ei:
        nt.nt_attention_decode(qd, kd, vd, 1, 32, 8, D, 1, 1, out, ws)
    assert ei.value.status == nt.NT_ERR_WORKSPACE
    ws = torch.zeros(nt.nt_attention_workspace_size(1, 32, 8, 1), dtype=torch.uint8, device=DEV)
    with pytest.raises(nt.NtError) as ei:
        nt.nt_attention_decode(qd, kd, vd, 1, 24, 8, D, 1, 1, out, ws)  # 3 query heads per group
    assert ei.value.status == nt.NT_ERR_UNSUPPORTED
    with pytest.raises(nt.NtError) as ei:
        nt.nt_attention_decode(qd, kd, vd, 1, 32, 8, 64, 1, 1, out, ws)
    assert ei.value.status == nt.NT_ERR_UNSUPPORTED


@pytest.mark.parametrize("B,pos0", [(1, 0), (3, 4093), (2, 16381), (8, 100000)])
def test_rope_append(B, pos0):
    Hq, Hkv, ts = 32, 8, pos0 + B + 3
    q = synth.normal(B * Hq * D, pos0, 4).reshape(B, Hq, D)
    k = synth.normal(B * Hkv * D, pos0, 5).reshape(B, Hkv, D)
    v = synth.normal(B * Hkv * D, pos0, 6).reshape(B, Hkv, D)
    sentinel = 0x7E7E
    kc = torch.full((Hkv, ts, D), sentinel, dtype=torch.int16, device=DEV)
    vc = torch.full((Hkv, ts, D), sentinel, dtype=torch.int16, device=DEV)
    qo = torch.empty((B, Hq, D), device=DEV)
    nt.nt_rope_append(dev(q), dev(k), dev(v), B, Hq, Hkv, D, pos0, 10000.0, qo, kc, vc, ts)
    pos = np.arange(pos0, pos0 + B)
    wq = lo.rope(q, pos)
    gq = host(qo).astype(np.float64)
    assert np.abs(gq - wq).max() <= 4 * 2.0 ** -24 * np.abs(wq).max() * 2
    kcu = host(kc).view(np.uint16)
    vcu = host(vc).view(np.uint16)
    wk = lo.rope(k, pos)  # [B, Hkv, D]
    gk = lo.from_bf16_bits(kcu[:, pos0:pos0 + B].transpose(1, 0, 2)).astype(np.float64)
    rk = lo.bf16_round(wk.astype(np.float32)).astype(np.float64)
    assert np.all(np.abs(gk - rk) <= np.abs(rk) * 2.0 ** -7 + 1e-38)  # at most one bf16 step
    assert np.mean(gk == rk) > 0.99
    assert np.array_equal(vcu[:, pos0:pos0 + B].transpose(1, 0, 2), lo.bf16_bits(lo.bf16_round(v)))
    other = np.ones(ts, bool)
    other[pos0:pos0 + B] = False
    assert np.all(kcu[:, other] == sentinel) and np.all(vcu[:, other] == sentinel)


@pytest.mark.parametrize("B,Dn", [(5, 4096), (2, 100), (1, 1), (3, 12288)])
def test_rmsnorm(B, Dn):
    x = synth.normal(B * Dn, Dn, 7).reshape(B, Dn) * np.float32(3.0)
    g = synth.scales(Dn, 1.0, Dn, 8)
    y = torch.empty((B, Dn), device=DEV)
    nt.nt_rmsnorm(dev(x), dev(g), B, Dn, 1e-6, y)
    want = lo.rmsnorm(x, g)
    got = host(y).astype(np.float64)
    assert np.all(np.abs(got - want) <= 4 * 2.0 ** -24 * np.abs(want) + 1e-30)

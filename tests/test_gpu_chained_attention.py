"""GPU parity of chained steps with the attention side (RMS norms, rotary embedding and cache
append, attention over the cache, SiLU gate), checked stage by stage on the step's own values.

A chained step quantizes, before every stage, a vector that the previous stages produced. One
rounding difference in a float operation (attention, norm, rotation, SiLU) early in the step
would otherwise travel through every later stage, so the comparison is teacher-forced: the plan
records every stage's fp32 input exactly as the step quantized it (nt_decode_plan_set_capture),
and each stage is checked against the oracle applied to the GPU's own inputs.

Exact (bit for bit, or within the 1e-6 relative bound the projections carry):
  * every stage's int8 codes and scale = the oracle's quantizer on the captured fp32 input;
  * every projection's output = the oracle's ternary GEMM on the GPU's codes and scale;
  * the residual stream: the next stage's un-normalised input is rebuilt from the GPU's outputs
    with one fp32 addition per term, as the pages' chain reads;
  * appended value rows = the bf16 rounding of the GPU's v outputs; rows before the step's
    positions untouched;
  * the output projection's logits and arg-max on the GPU's codes.

Derived tolerances, only for the float operations, each given the GPU's own inputs:
  * RMS norm (fl(fl(v*r)*gamma), r from fp32 sums of squares within a warp): a sum of m
    non-negative fp32 terms in any order is within (m-1)u of the exact sum (u = 2^-24), with m
    at most ceil(K/8) terms per warp (8 warps is the fewest any chained kernel uses); halved by
    the square root, plus r's own rounding and the two products: ((m-1)/2 + 2) u relative;
  * rotation: within 8 u of the largest element of its head, as the standalone rotation test
    bounds it; an appended key row within one bf16 rounding of the GPU's fp32 value beside it;
  * attention: 3e-5 max|v| (the standalone attention bound) plus the rotation error's effect:
    a score moves by at most delta = sum_i |dq_i||k_i| / sqrt(D), which moves the softmax
    weights by a factor within exp(+-2 delta);
  * SiLU-gated product: expf within 2 ulp, then an addition, a division and a product: within
    8 ulp (2^-23 relative each) of the float64 value.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from oracle import layer_ops as lo
from packed_weight_gemv_gb300 import nt
from synth import workloads as wl
from tests._gpu import DEV, assert_close, dev, host, plan_inputs

pytestmark = pytest.mark.gpu

U = 2.0 ** -24
D = 128

# 4 query heads and 2 key-value heads of 128 dimensions, hidden 512, feed-forward 1024
SHAPES = {"q": (512, 512), "k": (256, 512), "v": (256, 512), "o": (512, 512),
          "gate": (1024, 512), "up": (1024, 512), "down": (512, 1024)}


@pytest.fixture(scope="module", autouse=True)
def device():
    torch.cuda.set_device(DEV)
    nt.nt_device_check()


def rms_tol(want, K):
    m = -(-K // 8)
    return ((m - 1) / 2 + 2) * U * np.abs(want) + 1e-30


def check_quant(x, dq, ds, what):
    q, s = oracle.quantize(x)
    assert np.array_equal(host(dq), q), f"{what}: int8 codes differ from the quantizer on the captured input"
    assert np.array_equal(host(ds), s), f"{what}: scale differs"
    return q, s


def check_proj(p, d, q, s):
    _, y, _ = oracle.gemm(p.w_plain, p.s_w, p.N, p.K, q, s)
    got = host(d["y"])
    assert_close(got, y, p.name)
    return got


def check_float(got, want, tol, what):
    err = np.abs(got.astype(np.float64) - want)
    bad = err > tol
    assert not bad.any(), (f"{what}: {int(bad.sum())} values beyond the derived bound; worst "
                           f"{err.max():.3g} (bound there {np.broadcast_to(tol, err.shape).flat[err.argmax()]:.3g})")


def check_stagewise(projs, head, dp, hd, cap, x0, pos, kc_dev, vc_dev, k_before, v_before, ga, gf, gz):
    """Every stage of a chained step with attention against the oracle on the GPU's own inputs
    (module docstring). k_before / v_before: the caches' bf16 bits before the step."""
    L = len(projs) // 7
    B, d = x0.shape
    off = 0

    def take(K):
        nonlocal off
        a = cap[off:off + B * K].reshape(B, K)
        off += B * K
        return a

    def normed(v, gamma, what):  # the captured input of a normalised stage vs the float64 norm
        x = take(d)
        if gamma is None:
            assert np.array_equal(x, v), f"{what}: un-normalised stage input differs"
        else:
            want = lo.rmsnorm(v, gamma)
            check_float(x, want, rms_tol(want, d), what + " (RMS norm)")
        return x

    h = np.ascontiguousarray(x0, dtype=np.float32)
    posv = pos + np.arange(B)
    for l in range(L):
        P, Dl = projs[7 * l:7 * l + 7], dp[7 * l:7 * l + 7]
        xa = normed(h, None if ga is None else ga[l], f"layer {l} q/k/v input")
        q, s = check_quant(xa, Dl[0]["q"], Dl[0]["s_x"], f"layer {l} q/k/v")
        for j in (1, 2):
            assert np.array_equal(host(Dl[j]["q"]), q) and np.array_equal(host(Dl[j]["s_x"]), s)
        y_q, y_k, y_v = (check_proj(P[j], Dl[j], q, s) for j in range(3))
        Hq, Hkv = P[0].N // D, P[1].N // D
        kb = host(kc_dev[l]).view(np.uint16)
        vb = host(vc_dev[l]).view(np.uint16)
        assert np.array_equal(kb[:, :pos], k_before[l][:, :pos]) and np.array_equal(vb[:, :pos], v_before[l][:, :pos])
        new_v = vb[:, pos:pos + B].transpose(1, 0, 2)
        assert np.array_equal(new_v, lo.bf16_bits(lo.bf16_round(y_v.reshape(B, Hkv, D)))), f"layer {l} value rows"
        kr = lo.rope(y_k.reshape(B, Hkv, D), posv)
        rot_k = 8 * U * np.abs(kr).max(axis=2, keepdims=True)
        new_k = lo.from_bf16_bits(kb[:, pos:pos + B].transpose(1, 0, 2)).astype(np.float64)
        check_float(new_k, kr, rot_k + (np.abs(kr) + rot_k) * 2.0 ** -8, f"layer {l} key rows (rotation, bf16)")
        kf = lo.from_bf16_bits(kb)
        vf = lo.from_bf16_bits(vb)
        qr = lo.rope(y_q.reshape(B, Hq, D), posv)
        dq = 8 * U * np.abs(qr).max(axis=2)  # [B, Hq]: rotation bound per head
        T = pos + B
        ksum = np.abs(kf[:, :T].astype(np.float64)).sum(axis=2)  # [Hkv, T]
        delta = (dq[:, :, None] * ksum[np.arange(Hq) // (Hq // Hkv)][None]).max() / np.sqrt(D)
        vmax = float(np.abs(vf[:, :T]).max())
        u_want = lo.attention_decode(qr, kf, vf, T).reshape(B, Hq * D)
        xb = take(P[3].K)
        check_float(xb, u_want, 3e-5 * vmax + np.expm1(2 * delta) * vmax, f"layer {l} attention output")
        q, s = check_quant(xb, Dl[3]["q"], Dl[3]["s_x"], f"layer {l} o")
        y_o = check_proj(P[3], Dl[3], q, s)
        a = np.add(h, y_o, dtype=np.float32)
        xc = normed(a, None if gf is None else gf[l], f"layer {l} gate/up input")
        q, s = check_quant(xc, Dl[4]["q"], Dl[4]["s_x"], f"layer {l} gate/up")
        assert np.array_equal(host(Dl[5]["q"]), q) and np.array_equal(host(Dl[5]["s_x"]), s)
        y_gate, y_up = check_proj(P[4], Dl[4], q, s), check_proj(P[5], Dl[5], q, s)
        xd = take(P[6].K)
        g_want = lo.silu(y_gate) * y_up.astype(np.float64)
        check_float(xd, g_want, 8 * 2.0 ** -23 * np.abs(g_want) + 1e-37, f"layer {l} SiLU-gated product")
        q, s = check_quant(xd, Dl[6]["q"], Dl[6]["s_x"], f"layer {l} down")
        y_down = check_proj(P[6], Dl[6], q, s)
        h = np.add(a, y_down, dtype=np.float32)
    if head is not None:
        xh = normed(h, gz, "output projection input")
        q, s = check_quant(xh, hd["q"], hd["sx"], "output projection")
        logits, am, _ = oracle.logits_argmax(head.T, head.s_T, head.V, head.K, q, s)
        assert_close(host(hd["logits"]), logits, "logits")
        assert np.array_equal(host(hd["argmax"]), am)
    assert off == cap.size


def run_stagewise(L, B, pos, norms, launcher, shapes, head_V, Hkv, ts, seed, workload):
    d = shapes["q"][1]
    projs = wl.decoder_projections(L, shapes, B=B, seed=seed, workload=workload)
    head = wl.head(V=head_V, K=d, B=B, seed=seed, workload=workload)
    dp, hd = plan_inputs(projs, head, B=B)
    kb = [synth.bf16_normal(Hkv * ts * D, seed, 10 + l).reshape(Hkv, ts, D) for l in range(L)]
    vb = [synth.bf16_normal(Hkv * ts * D, seed, 20 + l).reshape(Hkv, ts, D) for l in range(L)]
    kc = [dev(k.view(np.int16)) for k in kb]
    vc = [dev(v.view(np.int16)) for v in vb]
    ga = [synth.scales(d, 1.0, seed, 30 + l) for l in range(L)] if norms else None
    gf = [synth.scales(d, 1.0, seed, 40 + l) for l in range(L)] if norms else None
    gz = synth.scales(d, 1.0, seed, 50) if norms else None
    att = dict(k_cache=kc, v_cache=vc, t_stride=ts, pos=pos)
    if norms:
        att.update(norm_attn=[dev(g) for g in ga], norm_ffn=[dev(g) for g in gf], norm_final=dev(gz))
    plan = nt.DecodePlan(L, B, dp, hd, nt.NT_STEP_CHAINED, launcher, attention=att)
    cap = torch.full((plan.nt_decode_plan_capture_size(),), float("nan"), device=DEV)
    plan.nt_decode_plan_set_capture(cap)
    plan.nt_decode_step()
    torch.cuda.synchronize()
    if launcher == nt.NT_LAUNCH_PERSISTENT:
        assert plan.nt_decode_step_status() == nt.NT_OK
    before_k = [k.view(np.uint16) for k in kb]
    before_v = [v.view(np.uint16) for v in vb]
    check_stagewise(projs, head, dp, hd, host(cap), projs[0].x[:B], pos, kc, vc, before_k, before_v, ga, gf, gz)
    plan.close()


@pytest.mark.parametrize("launcher", [nt.NT_LAUNCH_STREAM, nt.NT_LAUNCH_GRAPH, nt.NT_LAUNCH_PERSISTENT])
@pytest.mark.parametrize("B,pos,norms", [(1, 0, True), (1, 300, True), (3, 130, True), (2, 64, False), (5, 17, True)])
def test_chained_attention_stagewise(launcher, B, pos, norms):
    run_stagewise(2, B, pos, norms, launcher, SHAPES, 2500, 2, 512, 40 + pos, 40)


def test_chained_attention_8b_full_stagewise():
    # all 36 layers of the 8B shape (32 query / 8 key-value heads) with the full output table,
    # on the persistent launcher the decode path uses, 37 positions already cached
    run_stagewise(wl.DECODER_8B_LAYERS, 1, 37, True, nt.NT_LAUNCH_PERSISTENT, wl.DECODER_8B, wl.HEAD_V,
                  8, 64, 91, 42)


def test_capture_rejects_other_modes_and_misalignment():
    projs = wl.decoder_projections(1, SHAPES, seed=3, workload=43)
    dp, _ = plan_inputs(projs, None)
    plan = nt.DecodePlan(1, 1, dp, None, nt.NT_STEP_ORDERED, nt.NT_LAUNCH_PERSISTENT)
    with pytest.raises(nt.NtError) as e:
        plan.nt_decode_plan_capture_size()
    assert e.value.status == nt.NT_ERR_INVALID_ARG
    plan.close()
    plan = nt.DecodePlan(1, 1, dp, None, nt.NT_STEP_CHAINED, nt.NT_LAUNCH_GRAPH)
    n = plan.nt_decode_plan_capture_size()
    assert n == 512 + 512 + 512 + 1024
    buf = torch.empty(n + 4, device=DEV)
    with pytest.raises(nt.NtError) as e:
        plan.nt_decode_plan_set_capture(buf[1:])
    assert e.value.status == nt.NT_ERR_ALIGNMENT
    plan.nt_decode_plan_set_capture(None)
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


def test_chained_attention_step_refuses_graph_recording():
    # A persistent chained step with attention runs as several launches whose grid-barrier
    # counts live on the host; recording it into a CUDA graph is refused, not silently wrong.
    L, B, Hkv, ts = 1, 1, 2, 64
    projs = wl.decoder_projections(L, SHAPES, B=B, seed=45, workload=42)
    dp, _ = plan_inputs(projs, None, B=B)
    kc = [torch.zeros((Hkv, ts, 128), dtype=torch.int16, device=DEV) for _ in range(L)]
    vc = [torch.zeros((Hkv, ts, 128), dtype=torch.int16, device=DEV) for _ in range(L)]
    att = dict(k_cache=kc, v_cache=vc, t_stride=ts, pos=0)
    plan = nt.DecodePlan(L, B, dp, None, nt.NT_STEP_CHAINED, nt.NT_LAUNCH_PERSISTENT, attention=att)
    plan.nt_decode_step()
    torch.cuda.synchronize()
    graph, side = torch.cuda.CUDAGraph(), torch.cuda.Stream()
    with torch.cuda.stream(side):
        graph.capture_begin()
        try:
            with pytest.raises(nt.NtError) as e:
                plan.nt_decode_step()
        finally:
            graph.capture_end()
    assert e.value.status == nt.NT_ERR_UNSUPPORTED
    plan.nt_decode_step()  # still usable outside a recording
    torch.cuda.synchronize()
    assert plan.nt_decode_step_status() == nt.NT_OK
    del graph
    plan.close()

"""GPU parity: every C ABI call against the CPU oracle, element by element, on the same seeded
inputs. Integer results (int8 codes, int32 accumulators, arg-max indices, repacked bytes) must
match bit for bit; fp32 outputs within a relative error of 1e-6."""
import ctypes

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


# ---- quantization ---------------------------------------------------------------------

@pytest.mark.parametrize("B,K,kind", [(1, 512, "normal"), (3, 4096, "normal"), (2, 12288, "normal"),
                                      (1, 17, "normal"), (5, 1, "normal"), (2, 64, "zero"),
                                      (2, 256, "constant"), (1, 4096, "tiny"), (4, 1000, "heavy")])
def test_quantize(B, K, kind):
    x = synth.normal(B * K, 3, 100 + K).reshape(B, K)
    if kind == "zero":
        x[:] = 0
    elif kind == "constant":
        x[:] = -2.5
    elif kind == "tiny":
        x *= np.float32(1e-30)
    elif kind == "heavy":
        x = (x ** 3).astype(np.float32)
    q = torch.empty((B, K), dtype=torch.int8, device=DEV)
    s = torch.empty(B, dtype=torch.float32, device=DEV)
    nt.nt_quantize_act(dev(x), q, s)
    oq, os_ = oracle.quantize(x)
    assert np.array_equal(host(q), oq)
    assert np.array_equal(host(s), os_)


def half_integer_quotients(m: float) -> np.ndarray:
    """A vector of absmax m whose quotients x / s (s = fl(m / 127)) sit on and beside every
    half-integer k + 0.5: the products fl((k + 0.5) s) and their neighbours up to 3 ulps away,
    padded to a multiple of 16 with m."""
    m = np.float32(m)
    s = m / np.float32(127)
    vals = [m, -m]
    for k in range(-127, 127):
        x = np.float32(np.float32(k + 0.5) * s)
        if abs(x) > m:
            continue
        vals.append(x)
        up, down = x, x
        for _ in range(3):
            up, down = np.nextafter(up, np.float32(np.inf)), np.nextafter(down, np.float32(-np.inf))
            vals += [v for v in (up, down) if abs(v) <= m]
    vals += [m] * (-len(vals) % 16)
    return np.array(vals, dtype=np.float32)


@pytest.mark.parametrize("m", [100.0, 3.7, 1e-3, 55.55, 127.0, 0.1])
def test_quantize_half_integer_quotients(m):
    # The kernels form the quotient as x * fl(1/s) and fall back to the IEEE division near a
    # half-integer; these inputs sit exactly there. Per call and in a decode step's first phase.
    x = half_integer_quotients(m)
    oq, os_ = oracle.quantize(x)
    q = torch.empty(x.size, dtype=torch.int8, device=DEV)
    s = torch.empty(1, dtype=torch.float32, device=DEV)
    nt.nt_quantize_act(dev(x), q, s)
    assert np.array_equal(host(q), oq.reshape(-1)) and host(s)[0] == os_[0]
    K = x.size
    shapes = {n: (64, K) for n in wl.PROJ_NAMES}
    projs = wl.decoder_projections(1, shapes, seed=8, workload=44)
    for p in projs:
        p.x[0] = x
    dp, _ = plan_inputs(projs, None)
    plan = nt.DecodePlan(1, 1, dp, None, nt.NT_STEP_INDEPENDENT, nt.NT_LAUNCH_PERSISTENT)
    plan.nt_decode_step()
    torch.cuda.synchronize()
    for d in dp:
        assert np.array_equal(host(d["q"])[0], oq.reshape(-1)) and host(d["s_x"])[0] == os_[0]
    plan.close()


# ---- load-time repack ------------------------------------------------------------------

@pytest.mark.parametrize("N,K", [(1536, 512), (5, 48), (7, 528), (13, 1040), (1024, 4096), (4, 12288)])
def test_repack(N, K):
    w = synth.ternary_plain(N, K, 4, N + K)
    got = host(tiled(w, N, K))
    assert np.array_equal(got, oracle.repack_tiled(w, N, K))


def test_repack_counts_invalid_fields():
    N, K = 9, 64
    w = synth.ternary_plain(N, K, 5, 1)
    w[0, 0] = (w[0, 0] & ~np.uint32(0x3)) | np.uint32(0x2)        # field 0 of row 0 -> 10
    w[8, 3] = (w[8, 3] & ~np.uint32(0xC0000000)) | np.uint32(0x80000000)  # field 15
    cnt = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = torch.empty(nt.nt_repack_size(N, K), dtype=torch.uint8, device=DEV)
    nt.nt_repack_ternary(dev(w), N, K, out, cnt)
    assert int(cnt.item()) == oracle.count_invalid(w) == 2


@pytest.mark.parametrize("N,K,n_bad", [(9, 64, 0), (9, 64, 2), (1536, 512, 1), (4096, 4096, 977)])
def test_validate_ternary(N, K, n_bad):
    w = synth.ternary_plain(N, K, 6, N + K + n_bad)
    rng = np.random.default_rng(N + n_bad)
    flat = w.reshape(-1)
    for i in rng.choice(flat.size * 16, size=n_bad, replace=False):  # distinct fields -> 10
        word, f = divmod(int(i), 16)
        flat[word] = (flat[word] & ~np.uint32(3 << (2 * f))) | np.uint32(2 << (2 * f))
    assert oracle.count_invalid(w) == n_bad
    wd = dev(w)
    assert nt.nt_validate_ternary(wd, N, K) == n_bad
    n = ctypes.c_uint64(7)
    st = nt.load_library().nt_validate_ternary(ctypes.c_void_p(wd.data_ptr()), N, K, ctypes.byref(n), None)
    assert st == (nt.NT_ERR_INVALID_CODE if n_bad else nt.NT_OK) and n.value == n_bad


# ---- ternary projection ----------------------------------------------------------------

SHAPES = [(1536, 512), (5, 48), (7, 528), (33, 1040), (4096, 4096), (1024, 12288), (1, 16)]


@pytest.mark.parametrize("layout", [nt.NT_LAYOUT_PLAIN, nt.NT_LAYOUT_TILED])
@pytest.mark.parametrize("N,K", SHAPES)
def test_gemv(layout, N, K):
    p = wl.projection(8, 0, 0, N, K, 1, seed=1)
    q, s = oracle.quantize(p.x)
    acc, y, _ = oracle.gemv(p.w_plain, p.s_w, N, K, q[0], s)
    w = dev(p.w_plain) if layout == nt.NT_LAYOUT_PLAIN else tiled(p.w_plain, N, K)
    gy = torch.full((N,), float("nan"), device=DEV)
    gacc = torch.empty(N, dtype=torch.int32, device=DEV)
    nt.nt_ternary_gemv(w, layout, dev(p.s_w), N, K, dev(q), dev(s), gy, gacc)
    assert np.array_equal(host(gacc), acc)
    assert_close(host(gy), y, f"gemv {N}x{K}")


def test_single_gemv_workload():
    # The single ternary GEMV: W 1536 x 512, seed 0, batch 1, through both layouts.
    p = wl.single_gemv()
    q, s = oracle.quantize(p.x)
    acc, y, _ = oracle.gemv(p.w_plain, p.s_w, p.N, p.K, q[0], s)
    for layout in (nt.NT_LAYOUT_PLAIN, nt.NT_LAYOUT_TILED):
        w = dev(p.w_plain) if layout == nt.NT_LAYOUT_PLAIN else tiled(p.w_plain, p.N, p.K)
        gq = torch.empty((1, p.K), dtype=torch.int8, device=DEV)
        gs = torch.empty(1, dtype=torch.float32, device=DEV)
        nt.nt_quantize_act(dev(p.x), gq, gs)
        gy = torch.empty(p.N, device=DEV)
        gacc = torch.empty(p.N, dtype=torch.int32, device=DEV)
        nt.nt_ternary_gemv(w, layout, dev(p.s_w), p.N, p.K, gq, gs, gy, gacc)
        assert np.array_equal(host(gacc), acc)
        assert np.array_equal(host(gy), y)  # the fp32 epilogue order is fixed, so bit-equal


def test_gemv_closed_forms():
    N, K = 8, 512
    q = synth.int8_uniform(K, 9, 9)
    sq = int(q.astype(np.int64).sum())
    for word, expect in [(0, 0), (0x55555555, sq), (0xFFFFFFFF, -sq)]:
        w = np.full((N, K // 16), word, dtype=np.uint32)
        for layout in (nt.NT_LAYOUT_PLAIN, nt.NT_LAYOUT_TILED):
            ww = dev(w) if layout == nt.NT_LAYOUT_PLAIN else tiled(w, N, K)
            gy = torch.empty(N, device=DEV)
            gacc = torch.empty(N, dtype=torch.int32, device=DEV)
            nt.nt_ternary_gemv(ww, layout, dev(np.ones(N, np.float32)), N, K, dev(q),
                               dev(np.ones(1, np.float32)), gy, gacc)
            assert (host(gacc) == expect).all()


@pytest.mark.parametrize("layout", [nt.NT_LAYOUT_PLAIN, nt.NT_LAYOUT_TILED])
@pytest.mark.parametrize("B", [2, 3, 16, 17])
def test_gemm(layout, B):
    N, K = 260, 1024
    p = wl.projection(8, 1, B, N, K, B, seed=2)
    q, s = oracle.quantize(p.x)
    acc, y, _ = oracle.gemm(p.w_plain, p.s_w, N, K, q, s)
    w = dev(p.w_plain) if layout == nt.NT_LAYOUT_PLAIN else tiled(p.w_plain, N, K)
    gy = torch.empty((B, N), device=DEV)
    gacc = torch.empty((B, N), dtype=torch.int32, device=DEV)
    nt.nt_ternary_gemm(w, layout, dev(p.s_w), N, K, dev(q), dev(s), B, gy, gacc)
    assert np.array_equal(host(gacc), acc)
    assert_close(host(gy), y, f"gemm B={B}")


@pytest.mark.parametrize("B,N,K", [(2, 260, 1024), (3, 33, 1040), (8, 4096, 4096), (9, 1024, 12288),
                                   (16, 70001, 512), (5, 4, 16), (4, 128, 16), (7, 131, 208), (12, 300, 131072)])
def test_gemm_small_batch_tensor_cores(B, N, K):
    # Tiled weights, 2..16 vectors and a workspace: one pass on the tensor cores (tcgen05 with
    # the decoded weights in tensor memory from 128 rows on, mma.sync below); K parts meet in
    # the workspace, a wide matrix runs K unsplit; K of 16 / 208 (partial K-blocks) and
    # 131,072. Bit-exact sums.
    p = wl.projection(8, 2, B, N, K, B, seed=21)
    nbytes = nt.nt_ternary_gemm_workspace_size(N, K, B, nt.NT_LAYOUT_TILED)
    assert nbytes > 0
    ws = torch.zeros(nbytes, dtype=torch.uint8, device=DEV)
    w = tiled(p.w_plain, N, K)
    for x in (p.x, -0.5 * p.x[::-1].copy()):  # the second call reuses the workspace as the first left it
        q, s = oracle.quantize(x)
        q[0, :min(K, 64)] = 127  # extreme codes: digits (7, 15)
        q[-1, :min(K, 64)] = -127  # digits (-8, 1)
        acc, y, _ = oracle.gemm(p.w_plain, p.s_w, N, K, q, s)
        gy = torch.full((B, N), float("nan"), device=DEV)
        gacc = torch.empty((B, N), dtype=torch.int32, device=DEV)
        nt.nt_ternary_gemm(w, nt.NT_LAYOUT_TILED, dev(p.s_w), N, K, dev(q), dev(s), B, gy, gacc, ws)
        assert np.array_equal(host(gacc), acc)
        assert_close(host(gy), y, f"gemm B={B}")


# ---- int8 output projection ------------------------------------------------------------

def _head_call(T, s_T, V, K, q, s, B, ws=None):
    logits = torch.full((B, V), float("nan"), device=DEV)
    am = torch.full((B,), -1, dtype=torch.int32, device=DEV)
    if ws is None:
        ws = torch.zeros(nt.nt_int8_logits_workspace_size(V, K, B), dtype=torch.uint8, device=DEV)
    nt.nt_int8_logits_argmax(dev(T), dev(s_T), V, K, dev(q), dev(s), B, logits, am, ws)
    return host(logits), host(am), ws


@pytest.mark.parametrize("B", [1, 2, 3, 8, 16, 17])
def test_head_small(B):
    h = wl.head(V=5000, K=4096, B=B, seed=3)
    q, s = oracle.quantize(h.x)
    logits, am, _ = oracle.logits_argmax(h.T, h.s_T, h.V, h.K, q, s)
    gl, ga, ws = _head_call(h.T, h.s_T, h.V, h.K, q, s, B)
    assert_close(gl, logits, "head logits")
    assert np.array_equal(ga, am)
    gl2, ga2, _ = _head_call(h.T, h.s_T, h.V, h.K, q, s, B, ws)  # workspace reused as left
    assert np.array_equal(ga2, am) and np.array_equal(gl2, gl)


@pytest.mark.parametrize("plant", [0, 4999, 511, 512, 2048, 2049])
def test_head_planted_max_and_ties(plant):
    V, K = 5000, 256
    T = (synth.int8_uniform(V * K, 6, 7).reshape(V, K) // 4).astype(np.int8)
    T[plant] = 127
    tie = (plant * 7 + 13) % V
    T[tie] = 127
    q = np.full(K, 1, dtype=np.int8)
    s_T = np.ones(V, dtype=np.float32)
    s = np.ones(1, dtype=np.float32)
    logits, am, _ = oracle.logits_argmax(T, s_T, V, K, q, s)
    assert am[0] == min(plant, tie)
    _, ga, _ = _head_call(T, s_T, V, K, q, s, 1)
    assert ga[0] == am[0]


@pytest.mark.parametrize("B,K", [(2, 4144), (9, 1040), (16, 48)])
def test_head_batched_ragged_k_and_extremes(B, K):
    # 2..16 vectors take the tensor-core pass: K not a multiple of 64 (a partial last span and
    # chunk), rows of -128 / 127 against activations of +-127 (the largest chunk sums), and
    # planted ties between rows for every vector.
    V = 3001
    T = synth.int8_uniform(V * K, 11, B).reshape(V, K).copy()
    T[7] = -128
    T[8] = 127
    T[2990] = 127
    h = wl.head(V=V, K=K, B=B, seed=12)
    q, s = oracle.quantize(h.x)
    q[0] = 127
    q[-1] = -127
    s_T = np.ones(V, dtype=np.float32)
    s_T[::3] = 0.5
    logits, am, _ = oracle.logits_argmax(T, s_T, V, K, q, s)
    gl, ga, ws = _head_call(T, s_T, V, K, q, s, B)
    assert_close(gl, logits, "head logits")
    assert np.array_equal(ga, am)
    gl2, ga2, _ = _head_call(T, s_T, V, K, q, s, B, ws)
    assert np.array_equal(ga2, am) and np.array_equal(gl2, gl)


def test_head_full_table_batched():
    # The full table for 8 vectors in one tensor-core pass.
    h = wl.head(B=8)
    q, s = oracle.quantize(h.x)
    logits, am, _ = oracle.logits_argmax(h.T, h.s_T, h.V, h.K, q, s)
    gl, ga, _ = _head_call(h.T, h.s_T, h.V, h.K, q, s, 8)
    assert_close(gl, logits, "head full batched")
    assert np.array_equal(ga, am)


def test_head_full_table():
    # The int8 output projection at its full size: 151,936 x 4,096, batch 1.
    h = wl.head()
    q, s = oracle.quantize(h.x)
    logits, am, _ = oracle.logits_argmax(h.T, h.s_T, h.V, h.K, q, s)
    gl, ga, _ = _head_call(h.T, h.s_T, h.V, h.K, q, s, 1)
    assert_close(gl, logits, "head full")
    assert ga[0] == am[0]


# ---- decode step -----------------------------------------------------------------------

SMALL = {"q": (512, 512), "k": (128, 512), "v": (128, 512), "o": (512, 512),
         "gate": (1536, 512), "up": (1536, 512), "down": (512, 1536)}


def _check_step(projs, head, dp, hd, B=1):
    for p, d in zip(projs, dp):
        q, s = oracle.quantize(p.x[:B])
        assert np.array_equal(host(d["q"]), q), p.name
        assert np.array_equal(host(d["s_x"]), s), p.name
        _, y, _ = oracle.gemm(p.w_plain, p.s_w, p.N, p.K, q, s)
        assert_close(host(d["y"]), y, p.name)
    if head is not None:
        q, s = oracle.quantize(head.x[:B])
        logits, am, _ = oracle.logits_argmax(head.T, head.s_T, head.V, head.K, q, s)
        assert_close(host(hd["logits"]), logits, "head")
        assert np.array_equal(host(hd["argmax"]), am)


@pytest.mark.parametrize("launcher", [nt.NT_LAUNCH_PERSISTENT, nt.NT_LAUNCH_GRAPH, nt.NT_LAUNCH_STREAM])
@pytest.mark.parametrize("mode", [nt.NT_STEP_INDEPENDENT, nt.NT_STEP_ORDERED])
def test_decode_step_small(launcher, mode):
    projs = wl.decoder_projections(2, SMALL, seed=4, workload=10)
    head = wl.head(V=3001, K=512, seed=4, workload=10)
    dp, hd = plan_inputs(projs, head)
    plan = nt.DecodePlan(2, 1, dp, hd, mode, launcher)
    for _ in range(3):  # repeated steps reuse the plan's counters and workspace
        plan.nt_decode_step()
    torch.cuda.synchronize()
    assert plan.nt_decode_step_status() == nt.NT_OK
    _check_step(projs, head, dp, hd)
    plan.close()


@pytest.mark.parametrize("launcher", [nt.NT_LAUNCH_PERSISTENT, nt.NT_LAUNCH_GRAPH])
@pytest.mark.parametrize("mode", [nt.NT_STEP_INDEPENDENT, nt.NT_STEP_ORDERED])
@pytest.mark.parametrize("B", [2, 5, 16])
def test_decode_step_batched(launcher, mode, B):
    # Batches above 4 vectors take several passes in the persistent kernel (4 + 1, 4 x 4).
    projs = wl.decoder_projections(1, SMALL, B=B, seed=5, workload=11)
    head = wl.head(V=2000, K=512, B=B, seed=5, workload=11)
    dp, hd = plan_inputs(projs, head, B=B)
    plan = nt.DecodePlan(1, B, dp, hd, mode, launcher)
    for _ in range(2):
        plan.nt_decode_step()
    torch.cuda.synchronize()
    assert plan.nt_decode_step_status() == nt.NT_OK
    _check_step(projs, head, dp, hd, B=B)
    plan.close()


def test_decode_step_batched_8b_down_projection_shape():
    # K = 12288 activations for 4 vectors fill the shared-memory budget of one pass.
    shapes = dict(SMALL, down=(512, 12288), gate=(12288, 512), up=(12288, 512))
    projs = wl.decoder_projections(1, shapes, B=4, seed=8, workload=15)
    dp, _ = plan_inputs(projs, None, B=4)
    plan = nt.DecodePlan(1, 4, dp, None, nt.NT_STEP_ORDERED, nt.NT_LAUNCH_PERSISTENT)
    plan.nt_decode_step()
    torch.cuda.synchronize()
    assert plan.nt_decode_step_status() == nt.NT_OK
    _check_step(projs, None, dp, None, B=4)
    plan.close()


@pytest.mark.parametrize("launcher", [nt.NT_LAUNCH_GRAPH, nt.NT_LAUNCH_STREAM])
@pytest.mark.parametrize("B", [3, 11])
def test_decode_step_batched_wide_stage(launcher, B):
    # A stage with enough rows for four CTAs per SM takes K unsplit on the tensor-core batched
    # path: the sums go from registers straight to y (the split path meets in a workspace).
    shapes = dict(SMALL, gate=(81920, 1024), up=(81917, 1024))
    projs = wl.decoder_projections(1, shapes, B=B, seed=9, workload=16)
    dp, _ = plan_inputs(projs, None, B=B)
    plan = nt.DecodePlan(1, B, dp, None, nt.NT_STEP_INDEPENDENT, launcher)
    for _ in range(2):
        plan.nt_decode_step()
    torch.cuda.synchronize()
    _check_step(projs, None, dp, None, B=B)
    plan.close()


@pytest.mark.parametrize("B", [1, 3])
def test_decode_step_persistent_quantize_paths(B):
    # The persistent step's first phase keeps vectors of up to 12,288 values in registers when
    # they are 16-byte aligned; wider (14,336) or only 4-byte aligned inputs take the two-pass
    # path. Every other projection's input (and the table's) is offset by one float here, and
    # the codes and scales must be the oracle's either way.
    shapes = dict(SMALL, down=(512, 14336), gate=(14336, 512), up=(14336, 512))
    projs = wl.decoder_projections(1, shapes, B=B, seed=19, workload=19)
    head = wl.head(V=1999, K=512, B=B, seed=19, workload=19)
    dp, hd = plan_inputs(projs, head, B=B)

    def offset(x):
        buf = torch.empty(x.numel() + 1, dtype=torch.float32, device=DEV)
        v = buf[1:].view(x.shape)
        v.copy_(x)
        assert v.data_ptr() % 16 == 4
        return v

    for i, d in enumerate(dp):
        if i % 2 == 0:
            d["x"] = offset(d["x"])
    hd["x"] = offset(hd["x"])
    plan = nt.DecodePlan(1, B, dp, hd, nt.NT_STEP_INDEPENDENT, nt.NT_LAUNCH_PERSISTENT)
    for _ in range(2):
        plan.nt_decode_step()
    torch.cuda.synchronize()
    assert plan.nt_decode_step_status() == nt.NT_OK
    _check_step(projs, head, dp, hd, B=B)
    plan.close()


@pytest.mark.parametrize("launcher", [nt.NT_LAUNCH_PERSISTENT, nt.NT_LAUNCH_GRAPH])
def test_decode_step_inputs_in_pinned_host_memory(launcher):
    # The step reads its fp32 inputs straight from pinned host memory (no copy call): codes,
    # scales, outputs and the arg-max are the oracle's, over repeated steps.
    projs = wl.decoder_projections(1, SMALL, B=2, seed=21, workload=21)
    head = wl.head(V=2003, K=512, B=2, seed=21, workload=21)
    dp, hd = plan_inputs(projs, head, B=2)
    for d in dp:
        d["x"] = d["x"].cpu().pin_memory()
    hd["x"] = hd["x"].cpu().pin_memory()
    plan = nt.DecodePlan(1, 2, dp, hd, nt.NT_STEP_INDEPENDENT, launcher)
    for _ in range(3):
        plan.nt_decode_step()
    torch.cuda.synchronize()
    assert plan.nt_decode_step_status() == nt.NT_OK
    _check_step(projs, head, dp, hd, B=2)
    plan.close()


@pytest.mark.parametrize("mode", [nt.NT_STEP_INDEPENDENT, nt.NT_STEP_ORDERED, nt.NT_STEP_CHAINED])
@pytest.mark.parametrize("with_head", [True, False])
def test_persistent_step_replayed_from_cuda_graph(mode, with_head):
    # One persistent step recorded into a CUDA graph by stream capture, replayed with new
    # inputs written in place before each replay: every replay matches the oracle (the grid
    # barriers' counter is reset on the device, so the recorded parameters stay valid).
    L = 2
    projs = wl.decoder_projections(L, SMALL, seed=22, workload=22)
    head = wl.head(V=3001, K=512, seed=22, workload=22) if with_head else None
    dp, hd = plan_inputs(projs, head)
    plan = nt.DecodePlan(L, 1, dp, hd, mode, nt.NT_LAUNCH_PERSISTENT)
    plan.nt_decode_step()
    torch.cuda.synchronize()
    graph, side = torch.cuda.CUDAGraph(), torch.cuda.Stream()
    with torch.cuda.graph(graph, stream=side):
        plan.nt_decode_step()
    x0 = [p.x.copy() for p in projs]
    hx0 = head.x.copy() if with_head else None
    for rep in range(3):
        scale = np.float32(1.0 + 0.37 * rep)
        for p, d, x in zip(projs, dp, x0):
            p.x = (x * scale).astype(np.float32)
            d["x"].copy_(dev(p.x[:1]))
        if with_head:
            head.x = (hx0 * scale).astype(np.float32)
            hd["x"].copy_(dev(head.x[:1]))
        graph.replay()
        torch.cuda.synchronize()
        assert plan.nt_decode_step_status() == nt.NT_OK
        if mode != nt.NT_STEP_CHAINED:
            _check_step(projs, head, dp, hd)
        else:
            layers = [[(p.w_plain, p.s_w, p.N, p.K) for p in projs[7 * l:7 * l + 7]] for l in range(L)]
            want = oracle.decode_chained(layers, projs[0].x[:1],
                                         (head.T, head.s_T, head.V, head.K) if with_head else None)
            for i, (p, d) in enumerate(zip(projs, dp)):
                assert np.array_equal(host(d["q"]), want["q"][i]), p.name
                assert_close(host(d["y"]), want["y"][i], p.name)
            if with_head:
                assert np.array_equal(host(hd["argmax"]), want["argmax"])
    del graph
    plan.close()


def test_decode_step_prequantized_inputs():
    projs = wl.decoder_projections(1, SMALL, seed=6, workload=12)
    dp, _ = plan_inputs(projs, None, quantize_in_step=False)
    for p, d in zip(projs, dp):
        q, s = oracle.quantize(p.x)
        d["q"].copy_(dev(q))
        d["s_x"].copy_(dev(s))
    plan = nt.DecodePlan(1, 1, dp, None, nt.NT_STEP_INDEPENDENT, nt.NT_LAUNCH_PERSISTENT)
    plan.nt_decode_step()
    torch.cuda.synchronize()
    _check_step(projs, None, dp, None)
    plan.close()


def test_persistent_timeout_is_reported_and_recoverable():
    # A grid barrier that waits for one arrival more than the grid makes runs out after
    # timeout_ms; the step reports NT_ERR_TIMEOUT and the context stays usable.
    projs = wl.decoder_projections(1, SMALL, seed=7, workload=13)
    dp, _ = plan_inputs(projs, None)
    plan = nt.DecodePlan(1, 1, dp, None, nt.NT_STEP_ORDERED, nt.NT_LAUNCH_PERSISTENT,
                         timeout_ms=20.0, test_fault=1)
    plan.nt_decode_step()
    torch.cuda.synchronize()
    assert plan.nt_decode_step_status() == nt.NT_ERR_TIMEOUT
    plan.close()
    good = nt.DecodePlan(1, 1, dp, None, nt.NT_STEP_ORDERED, nt.NT_LAUNCH_PERSISTENT)
    good.nt_decode_step()
    torch.cuda.synchronize()
    assert good.nt_decode_step_status() == nt.NT_OK
    _check_step(projs, None, dp, None)
    good.close()


@pytest.mark.parametrize("launcher", [nt.NT_LAUNCH_GRAPH, nt.NT_LAUNCH_STREAM])
def test_tcgen05_batched_timeout_is_reported_and_recoverable(launcher):
    # The tcgen05 batched kernel with producers that issue no copies: every consumer's wait runs
    # out after timeout_ms, the CTAs free their tensor memory and report NT_ERR_TIMEOUT; the
    # context stays usable and a plan without the fault is correct.
    B = 3
    projs = wl.decoder_projections(1, SMALL, B=B, seed=17, workload=18)
    dp, _ = plan_inputs(projs, None, B=B)
    plan = nt.DecodePlan(1, B, dp, None, nt.NT_STEP_INDEPENDENT, launcher, timeout_ms=20.0, test_fault=2)
    plan.nt_decode_step()
    torch.cuda.synchronize()
    assert plan.nt_decode_step_status() == nt.NT_ERR_TIMEOUT
    plan.close()
    good = nt.DecodePlan(1, B, dp, None, nt.NT_STEP_INDEPENDENT, launcher)
    good.nt_decode_step()
    torch.cuda.synchronize()
    assert good.nt_decode_step_status() == nt.NT_OK
    _check_step(projs, None, dp, None, B=B)
    good.close()


# ---- prefill-shaped batches on the tensor cores -----------------------------------------

TC_SHAPES = [(128, 256, 512), (200, 260, 1024), (64, 20, 528), (256, 3072, 1024),
             (2048, 1024, 3072), (130, 1024, 2048), (8192, 640, 2048), (97, 4100, 1040)]


@pytest.mark.parametrize("M,N,K", TC_SHAPES)
def test_gemm_tensor_cores(M, N, K):
    p = wl.projection(16, M % 7, N % 5, N, K, M, seed=9)
    q, s = oracle.quantize(p.x)
    acc, y, _ = oracle.gemm(p.w_plain, p.s_w, N, K, q, s)
    gy = torch.full((M, N), float("nan"), device=DEV)
    gacc = torch.empty((M, N), dtype=torch.int32, device=DEV)
    ws = torch.empty(nt.nt_ternary_gemm_workspace_size(N, K, M, nt.NT_LAYOUT_TILED), dtype=torch.uint8,
                     device=DEV)
    assert ws.numel() > 0
    nt.nt_ternary_gemm(tiled(p.w_plain, N, K), nt.NT_LAYOUT_TILED, dev(p.s_w), N, K, dev(q), dev(s),
                       M, gy, gacc, ws)
    assert np.array_equal(host(gacc), acc)
    assert_close(host(gy), y, f"tensor-core gemm {M}x{N}x{K}")


def test_gemm_tensor_cores_cancellation():
    # Rows of alternating +1/-1 against constant activations cancel to exactly 0; all-+1 rows
    # against 127 reach 127 * K. A tensor-core accumulator that rounded would miss either.
    M, N, K = 128, 256, 16384
    w = np.empty((N, K // 16), dtype=np.uint32)
    w[0::2] = 0xDDDDDDDD
    w[1::2] = 0x55555555
    q = np.full((M, K), 127, dtype=np.int8)
    q[1::2] = -127
    s_w = np.ones(N, dtype=np.float32)
    s = np.ones(M, dtype=np.float32)
    acc, _, _ = oracle.gemm(w, s_w, N, K, q, s)
    assert (acc[:, 0::2] == 0).all() and (np.abs(acc[:, 1::2]) == 127 * K).all()
    gy = torch.empty((M, N), device=DEV)
    gacc = torch.empty((M, N), dtype=torch.int32, device=DEV)
    ws = torch.empty(nt.nt_ternary_gemm_workspace_size(N, K, M, nt.NT_LAYOUT_TILED), dtype=torch.uint8,
                     device=DEV)
    nt.nt_ternary_gemm(tiled(w, N, K), nt.NT_LAYOUT_TILED, dev(s_w), N, K, dev(q), dev(s), M, gy, gacc, ws)
    assert np.array_equal(host(gacc), acc)


@pytest.mark.parametrize("M,Ns,K", [(300, (200, 128, 389), 1040), (2048, (2048, 1024, 1024), 1024),
                                    (64, (3072, 3072), 1024), (40, (100, 36, 64), 512)])
def test_gemm_multi_shared_activations(M, Ns, K):
    # several matrices of one input in one call: every output exact, whatever the row counts
    # (tiles of one matrix never mix rows of another), on the tensor-core path (M >= 64) and
    # the per-matrix path below it
    ps = [wl.projection(17, i, len(Ns), N, K, M, seed=10) for i, N in enumerate(Ns)]
    x = ps[0].x
    q, s = oracle.quantize(x)
    ws = torch.empty(max(1, nt.nt_ternary_gemm_multi_workspace_size(list(Ns), K, M)), dtype=torch.uint8, device=DEV)
    ys = [torch.full((M, N), float("nan"), device=DEV) for N in Ns]
    accs = [torch.empty((M, N), dtype=torch.int32, device=DEV) for N in Ns]
    nt.nt_ternary_gemm_multi([tiled(p.w_plain, p.N, K) for p in ps], [dev(p.s_w) for p in ps], list(Ns), K, dev(q),
                             dev(s), M, ys, accs, ws)
    for p, gy, ga in zip(ps, ys, accs):
        acc, y, _ = oracle.gemm(p.w_plain, p.s_w, p.N, K, q, s)
        assert np.array_equal(host(ga), acc)
        assert_close(host(gy), y, f"multi {p.N}")

"""The C ABI library loads and exports every symbol include/nt.h declares; host-side argument
validation of every call and of the decode-plan descriptor answers without a GPU (no compute
call is made): each malformed argument gets the status the header states, and well-formed ones
get as far as the device check."""
import ctypes
import os
import re

import pytest

from packed_weight_gemv_gb300 import build as nt_build
from packed_weight_gemv_gb300 import nt

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    nt_build.build()
    return nt.load_library()


def declared_functions():
    src = open(os.path.join(ROOT, "include", "nt.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(nt_[a-z0-9_]+)\s*\(", src)))


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert len(names) >= 16
    for name in names:
        assert hasattr(lib, name), name
    assert set(names) == set(nt.EXPORTS)


def test_abi_version_and_status_strings(lib):
    assert lib.nt_abi_version() == 1
    for s in range(8):
        assert lib.nt_status_string(s)
    assert b"unknown" in lib.nt_status_string(99)


def test_size_queries(lib):
    assert nt.nt_repack_size(1536, 512) == 1536 * 512 // 4
    assert nt.nt_repack_size(5, 16) == 8 * 512 // 4
    assert nt.nt_repack_size(4096, 12288) == 4096 * 12288 // 4
    assert nt.nt_int8_logits_workspace_size(151936, 4096, 1) > 0
    with pytest.raises(nt.NtError) as e:
        nt.nt_repack_size(4, 15)
    assert e.value.status == nt.NT_ERR_INVALID_ARG


def _gemv(lib, w, layout, N, K, q, y, B=1):
    vp = ctypes.c_void_p
    return lib.nt_ternary_gemm(vp(w), layout, vp(0x1000), N, K, vp(q), vp(0x2000), B, vp(y),
                               None, None, 0, None)


def test_argument_errors_without_gpu(lib):
    # Validation happens before any device call, so these answer on a machine with no GPU.
    assert _gemv(lib, 0x10000, 1, 16, 15, 0x20000, 0x30000) == nt.NT_ERR_INVALID_ARG
    assert _gemv(lib, 0x10000, 1, 0, 16, 0x20000, 0x30000) == nt.NT_ERR_INVALID_ARG
    assert _gemv(lib, 0x10000, 7, 16, 16, 0x20000, 0x30000) == nt.NT_ERR_INVALID_ARG
    assert _gemv(lib, 0x10008, 1, 16, 16, 0x20000, 0x30000) == nt.NT_ERR_ALIGNMENT
    assert _gemv(lib, 0x10000, 1, 16, 16, 0x20004, 0x30000) == nt.NT_ERR_ALIGNMENT
    assert _gemv(lib, 0, 1, 16, 16, 0x20000, 0x30000) == nt.NT_ERR_INVALID_ARG
    # the tensor-core path (tiled, B >= 64) needs a workspace: refused before any device call
    assert _gemv(lib, 0x10000, 1, 256, 512, 0x20000, 0x30000, B=64) == nt.NT_ERR_WORKSPACE
    # every workspace starts with the 256-byte status header (16 bytes used, the rest keeps the
    # data's alignment)
    H = 256
    # prefill: the status header and an f16 copy of the activations (the weights stay packed)
    assert nt.nt_ternary_gemm_workspace_size(256, 512, 64, nt.NT_LAYOUT_TILED) == H + 64 * 512 * 2
    # 2..16 vectors, from 128 rows: an optional workspace of e4m3 digit rows (16 for B <= 8,
    # else 32, K rounded up to 128), int32 partial sums [B][N] and one counter per 128-row
    # tile, rounded up to 16 bytes; below 128 rows sums and one counter per 256 rows; none for
    # one vector or above 16
    r16 = lambda b: (b + 15) // 16 * 16  # noqa: E731
    assert nt.nt_ternary_gemm_workspace_size(256, 512, 16, nt.NT_LAYOUT_TILED) == H + r16(32 * 512 + 16 * 256 * 4 + 2 * 4)
    assert nt.nt_ternary_gemm_workspace_size(1000, 512, 3, nt.NT_LAYOUT_TILED) == H + r16(16 * 512 + 3 * 1000 * 4 + 8 * 4)
    assert nt.nt_ternary_gemm_workspace_size(1000, 208, 3, nt.NT_LAYOUT_TILED) == H + r16(16 * 256 + 3 * 1000 * 4 + 8 * 4)
    assert nt.nt_ternary_gemm_workspace_size(100, 512, 3, nt.NT_LAYOUT_TILED) == H + (3 * 100 * 4 + 4 + 15) // 16 * 16
    assert nt.nt_ternary_gemm_workspace_size(256, 512, 1, nt.NT_LAYOUT_TILED) == 0
    assert nt.nt_ternary_gemm_workspace_size(256, 512, 17, nt.NT_LAYOUT_TILED) == 0
    assert nt.nt_ternary_gemm_workspace_size(256, 512, 16, nt.NT_LAYOUT_PLAIN) == 0
    assert b"multiple of 16" in lib.nt_last_error_string() or True
    vp = ctypes.c_void_p
    assert lib.nt_quantize_act(None, 1, 16, vp(0x100), vp(0x200), None) == nt.NT_ERR_INVALID_ARG
    assert lib.nt_quantize_act(vp(0x102), 1, 16, vp(0x100), vp(0x200), None) == nt.NT_ERR_ALIGNMENT
    r = lib.nt_int8_logits_argmax(vp(0x1000), vp(0x2000), 10, 16, vp(0x3000), vp(0x4000), 1,
                                  None, vp(0x5000), None, 0, None)
    assert r == nt.NT_ERR_WORKSPACE
    r = lib.nt_int8_logits_argmax(vp(0x1008), vp(0x2000), 10, 16, vp(0x3000), vp(0x4000), 1,
                                  None, vp(0x5000), vp(0x6000), 1 << 20, None)
    assert r == nt.NT_ERR_ALIGNMENT


def test_validate_argument_errors_without_gpu(lib):
    vp, n = ctypes.c_void_p, ctypes.c_uint64(0)
    assert lib.nt_validate_ternary(None, 4, 16, ctypes.byref(n), None) == nt.NT_ERR_INVALID_ARG
    assert lib.nt_validate_ternary(vp(0x1000), 4, 15, ctypes.byref(n), None) == nt.NT_ERR_INVALID_ARG
    assert lib.nt_validate_ternary(vp(0x1000), 0, 16, ctypes.byref(n), None) == nt.NT_ERR_INVALID_ARG
    assert lib.nt_validate_ternary(vp(0x1002), 4, 16, ctypes.byref(n), None) == nt.NT_ERR_ALIGNMENT
    assert b"10" in lib.nt_status_string(nt.NT_ERR_INVALID_CODE)


def test_status_and_fault_hook_without_gpu(lib):
    st = ctypes.c_int(-1)
    assert lib.nt_workspace_status(None, ctypes.byref(st)) == nt.NT_ERR_INVALID_ARG
    assert lib.nt_workspace_status(ctypes.c_void_p(0x1000), None) == nt.NT_ERR_INVALID_ARG
    assert lib.nt_set_test_fault(4, 1.0) == nt.NT_ERR_INVALID_ARG
    assert lib.nt_set_test_fault(-1, 1.0) == nt.NT_ERR_INVALID_ARG
    assert lib.nt_set_test_fault(0, 0.0) == nt.NT_OK
    assert lib.nt_decode_plan_capture_size(None, ctypes.byref(ctypes.c_size_t(0))) == nt.NT_ERR_INVALID_ARG
    assert lib.nt_decode_plan_set_capture(None, None) == nt.NT_ERR_INVALID_ARG


def test_plan_descriptor_errors_without_gpu(lib):
    d = nt.nt_decode_desc()
    h = ctypes.c_void_p(None)
    assert lib.nt_decode_plan_create(ctypes.byref(d), ctypes.byref(h)) == nt.NT_ERR_INVALID_ARG
    arr = (nt.nt_proj * 7)()
    for i in range(7):
        arr[i] = nt.nt_proj(64, 48, 0x10000, 0x20000, None, 0x30000, 0x40000, 0x50000)
    d.n_layers, d.batch, d.proj = 1, 17, ctypes.cast(arr, ctypes.POINTER(nt.nt_proj))
    assert lib.nt_decode_plan_create(ctypes.byref(d), ctypes.byref(h)) == nt.NT_ERR_INVALID_ARG
    d.batch, d.mode = 1, 5
    assert lib.nt_decode_plan_create(ctypes.byref(d), ctypes.byref(h)) == nt.NT_ERR_INVALID_ARG
    d.mode = 0
    arr[3] = nt.nt_proj(64, 40, 0x10000, 0x20000, None, 0x30000, 0x40000, 0x50000)
    assert lib.nt_decode_plan_create(ctypes.byref(d), ctypes.byref(h)) == nt.NT_ERR_INVALID_ARG
    arr[3] = nt.nt_proj(64, 48, 0x10004, 0x20000, None, 0x30000, 0x40000, 0x50000)
    assert lib.nt_decode_plan_create(ctypes.byref(d), ctypes.byref(h)) == nt.NT_ERR_ALIGNMENT
    assert not h.value


# Past validation a call checks the device; with no GPU that check answers NT_ERR_CUDA (no
# device) or NT_ERR_UNSUPPORTED (not a GB300). Either way the arguments were accepted.
REACHED_DEVICE = (nt.NT_ERR_CUDA, nt.NT_ERR_UNSUPPORTED)
INT_MAX = 2**31 - 1


def test_gather_and_acceptance_argument_errors(lib):
    vp = ctypes.c_void_p

    def embed(T=0x1000, s=0x2000, V=10, K=16, tok=0x3000, B=2, x=0x4000, nbad=None):
        return lib.nt_embed_rows(vp(T), vp(s), V, K, vp(tok), B, vp(x), vp(nbad) if nbad else None, None)

    assert embed() in REACHED_DEVICE
    assert embed(T=0) == nt.NT_ERR_INVALID_ARG
    assert embed(tok=0) == nt.NT_ERR_INVALID_ARG
    assert embed(V=0) == nt.NT_ERR_INVALID_ARG
    assert embed(K=24) == nt.NT_ERR_INVALID_ARG
    assert embed(B=0) == nt.NT_ERR_INVALID_ARG
    assert embed(B=65536) == nt.NT_ERR_INVALID_ARG
    assert embed(T=0x1008) == nt.NT_ERR_ALIGNMENT
    assert embed(x=0x4004) == nt.NT_ERR_ALIGNMENT
    assert embed(tok=0x3002) == nt.NT_ERR_ALIGNMENT
    assert embed(nbad=0x5001) == nt.NT_ERR_ALIGNMENT
    assert embed(nbad=0x5000) in REACHED_DEVICE  # the counter is optional

    def accept(draft=0x1000, am=0x2000, B=3, emit=0x3000, n=0x4000):
        return lib.nt_verify_accept(vp(draft) if draft else None, vp(am), B, vp(emit), vp(n), None)

    assert accept() in REACHED_DEVICE
    assert accept(draft=0, B=1) in REACHED_DEVICE  # one position has no drafts
    assert accept(draft=0, B=2) == nt.NT_ERR_INVALID_ARG
    assert accept(B=0) == nt.NT_ERR_INVALID_ARG
    assert accept(emit=0x3002) == nt.NT_ERR_ALIGNMENT
    assert accept(draft=0x1001) == nt.NT_ERR_ALIGNMENT


def test_attention_side_argument_errors(lib):
    vp, sz = ctypes.c_void_p, ctypes.c_size_t(0)
    assert lib.nt_attention_workspace_size(2, 32, 8, 4096, ctypes.byref(sz)) == nt.NT_OK and sz.value > 0
    big = sz.value

    def attend(q=0x1000, kc=0x2000, vc=0x3000, B=2, Hq=32, Hkv=8, D=128, T=4096, ts=4096, out=0x4000,
               ws=0x5000, ws_bytes=big):
        return lib.nt_attention_decode(vp(q), vp(kc), vp(vc), B, Hq, Hkv, D, T, ts, vp(out), vp(ws), ws_bytes, None)

    assert attend() in REACHED_DEVICE
    assert attend(q=0) == nt.NT_ERR_INVALID_ARG
    assert attend(D=64) == nt.NT_ERR_UNSUPPORTED
    assert attend(Hq=12, Hkv=8) == nt.NT_ERR_INVALID_ARG
    assert attend(Hq=24, Hkv=8) == nt.NT_ERR_UNSUPPORTED  # 3 query heads per key-value head
    assert attend(B=65) == nt.NT_ERR_INVALID_ARG
    assert attend(T=1) == nt.NT_ERR_INVALID_ARG  # fewer cached rows than new positions
    assert attend(ts=4095) == nt.NT_ERR_INVALID_ARG
    assert attend(kc=0x2008) == nt.NT_ERR_ALIGNMENT
    assert attend(ws_bytes=big - 1) == nt.NT_ERR_WORKSPACE

    def rope(q=0x1000, k=0x2000, v=0x3000, B=2, Hq=32, Hkv=8, D=128, pos0=10, base=10000.0, qo=0x4000,
             kc=0x5000, vc=0x6000, ts=4096):
        return lib.nt_rope_append(vp(q), vp(k), vp(v), B, Hq, Hkv, D, pos0, ctypes.c_float(base), vp(qo), vp(kc),
                                  vp(vc), ts, None)

    assert rope() in REACHED_DEVICE
    assert rope(kc=0) == nt.NT_ERR_INVALID_ARG
    assert rope(D=256) == nt.NT_ERR_UNSUPPORTED
    assert rope(pos0=-1) == nt.NT_ERR_INVALID_ARG
    assert rope(pos0=4095) == nt.NT_ERR_INVALID_ARG  # the last new position would be row 4096
    assert rope(pos0=4094) in REACHED_DEVICE
    assert rope(pos0=INT_MAX) == nt.NT_ERR_INVALID_ARG  # no overflow in the range check
    assert rope(base=1.0) == nt.NT_ERR_INVALID_ARG
    assert rope(base=float("nan")) == nt.NT_ERR_INVALID_ARG
    assert rope(kc=0x5001) == nt.NT_ERR_ALIGNMENT
    assert rope(q=0x1002) == nt.NT_ERR_ALIGNMENT

    def norm(x=0x1000, g=0x2000, B=2, D=4096, eps=1e-6, y=0x3000):
        return lib.nt_rmsnorm(vp(x), vp(g), B, D, ctypes.c_float(eps), vp(y), None)

    assert norm() in REACHED_DEVICE
    assert norm(eps=0.0) in REACHED_DEVICE
    assert norm(g=0) == nt.NT_ERR_INVALID_ARG
    assert norm(D=0) == nt.NT_ERR_INVALID_ARG
    assert norm(eps=-1e-6) == nt.NT_ERR_INVALID_ARG
    assert norm(eps=float("nan")) == nt.NT_ERR_INVALID_ARG
    assert norm(y=0x3002) == nt.NT_ERR_ALIGNMENT


def test_multi_matrix_and_noalloc_argument_errors(lib):
    vp = ctypes.c_void_p
    P = ctypes.c_void_p * 2
    Ns = (ctypes.c_int * 2)(256, 512)
    w, s_w, y = P(0x10000, 0x20000), P(0x30000, 0x30100), P(0x40000, 0x50000)

    def multi(n=2, w=w, N=Ns, K=512, q=0x60000, B=8, ws=None, ws_bytes=0):
        return lib.nt_ternary_gemm_multi(n, w, s_w, N, K, vp(q), vp(0x70000), B, y, None,
                                         vp(ws) if ws else None, ws_bytes, None)

    assert multi() in REACHED_DEVICE
    assert multi(n=0) == nt.NT_ERR_INVALID_ARG
    assert multi(n=9) == nt.NT_ERR_INVALID_ARG
    assert multi(w=None) == nt.NT_ERR_INVALID_ARG
    assert multi(N=(ctypes.c_int * 2)(256, 0)) == nt.NT_ERR_INVALID_ARG
    assert multi(K=500) == nt.NT_ERR_INVALID_ARG
    assert multi(w=P(0x10000, 0x20008)) == nt.NT_ERR_ALIGNMENT
    assert multi(B=64) == nt.NT_ERR_WORKSPACE  # the tensor-core path needs its workspace
    sz = ctypes.c_size_t(0)
    assert lib.nt_ternary_gemm_multi_workspace_size(2, Ns, 512, 64, ctypes.byref(sz)) == nt.NT_OK
    assert multi(B=64, ws=0x80000, ws_bytes=sz.value) in REACHED_DEVICE
    assert multi(B=64, ws=0x80000, ws_bytes=sz.value - 1) == nt.NT_ERR_WORKSPACE
    assert lib.nt_ternary_gemm_multi_workspace_size(9, Ns, 512, 64, ctypes.byref(sz)) == nt.NT_ERR_INVALID_ARG

    def noalloc(T=0x1000, B=1, q=0x3000, logits=0x5000):
        return lib.nt_int8_logits_argmax_noalloc(vp(T), vp(0x2000), 100, 64, vp(q), vp(0x4000), B,
                                                 vp(logits) if logits else None, vp(0x6000), None)

    assert noalloc() in REACHED_DEVICE
    assert noalloc(B=16, logits=None) in REACHED_DEVICE
    assert noalloc(B=17) == nt.NT_ERR_INVALID_ARG  # its fixed scratch serves 16 vectors
    assert noalloc(T=0) == nt.NT_ERR_INVALID_ARG
    assert noalloc(q=0x3004) == nt.NT_ERR_ALIGNMENT
    assert noalloc(logits=0x5002) == nt.NT_ERR_ALIGNMENT


def test_plan_calls_refuse_a_null_plan(lib):
    i, u = ctypes.c_int(0), ctypes.c_int(0)
    st, n = ctypes.c_int(0), ctypes.c_size_t(0)
    assert lib.nt_decode_step(None, None) == nt.NT_ERR_INVALID_ARG
    assert lib.nt_decode_step_status(None, ctypes.byref(st)) == nt.NT_ERR_INVALID_ARG
    assert lib.nt_decode_plan_reset(None) == nt.NT_ERR_INVALID_ARG
    assert lib.nt_decode_plan_set_position(None, 0, None) == nt.NT_ERR_INVALID_ARG
    assert lib.nt_decode_plan_trace_layout(None, ctypes.byref(i), ctypes.byref(u)) == nt.NT_ERR_INVALID_ARG
    assert lib.nt_decode_plan_set_trace(None, None) == nt.NT_ERR_INVALID_ARG
    assert lib.nt_decode_plan_capture_size(None, ctypes.byref(n)) == nt.NT_ERR_INVALID_ARG
    lib.nt_decode_plan_destroy(None)  # a no-op
    assert lib.nt_decode_plan_create(None, None) == nt.NT_ERR_INVALID_ARG


def _chained_desc(n_layers=1, dm=256, q=256, kv=128, ffn=384):
    """A consistent chained descriptor with fake (aligned, never dereferenced) device addresses."""
    shapes = [(q, dm), (kv, dm), (kv, dm), (dm, q), (ffn, dm), (ffn, dm), (dm, ffn)]
    arr = (nt.nt_proj * (7 * n_layers))()
    for l in range(n_layers):
        for i, (N, K) in enumerate(shapes):
            base = 0x100000 * (1 + 7 * l + i)
            arr[7 * l + i] = nt.nt_proj(N, K, base, base + 0x10000, base + 0x20000 if l == 0 and i == 0 else None,
                                        base + 0x30000, base + 0x40000, base + 0x50000)
    d = nt.nt_decode_desc()
    d.n_layers, d.batch, d.proj = n_layers, 2, ctypes.cast(arr, ctypes.POINTER(nt.nt_proj))
    d.mode, d.launcher = nt.NT_STEP_CHAINED, nt.NT_LAUNCH_PERSISTENT
    return d, arr


def test_chained_plan_descriptor_errors_without_gpu(lib):
    h = ctypes.c_void_p(None)
    create = lambda d: lib.nt_decode_plan_create(ctypes.byref(d), ctypes.byref(h))  # noqa: E731
    d, arr = _chained_desc()
    assert create(d) in REACHED_DEVICE
    d.head_dim = 6
    assert create(d) == nt.NT_ERR_INVALID_ARG  # head_dim must be a multiple of 4
    d.head_dim = 0
    arr[3] = nt.nt_proj(256, 128, 0x400000, 0x410000, None, 0x430000, 0x440000, 0x450000)  # o.K != q.N
    assert create(d) == nt.NT_ERR_INVALID_ARG
    d, arr = _chained_desc()
    arr[5] = nt.nt_proj(384, 256, 0x600000, 0x610000, None, 0x630000, 0x640000, 0x650008)  # y not 16-aligned
    assert create(d) == nt.NT_ERR_ALIGNMENT
    d, arr = _chained_desc()
    arr[0] = nt.nt_proj(256, 256, 0x100000, 0x110000, None, 0x130000, 0x140000, 0x150000)  # no first input
    assert create(d) == nt.NT_ERR_INVALID_ARG
    # the attention side: head counts, grouping, cache range
    d, arr = _chained_desc()
    caches = (ctypes.c_void_p * 1)(0x9000000)
    d.attn_k_cache = d.attn_v_cache = ctypes.cast(caches, ctypes.POINTER(ctypes.c_void_p))
    d.attn_t_stride, d.attn_pos = 64, 10
    assert create(d) in REACHED_DEVICE
    d.attn_pos = 63  # position 63 + batch 2 passes the cache's end
    assert create(d) == nt.NT_ERR_INVALID_ARG
    d.attn_pos = INT_MAX  # no overflow in the range check
    assert create(d) == nt.NT_ERR_INVALID_ARG
    d.attn_pos = 0
    d.head_dim = 64
    assert create(d) == nt.NT_ERR_UNSUPPORTED  # attention needs 128-dimension heads
    d.head_dim = 0
    d3, _ = _chained_desc(q=384, kv=128)  # 3 query heads per key-value head
    d3.attn_k_cache = d3.attn_v_cache = d.attn_k_cache
    d3.attn_t_stride = 64
    assert create(d3) == nt.NT_ERR_UNSUPPORTED
    assert not h.value


def test_step_extras_descriptor_errors_without_gpu(lib):
    h = ctypes.c_void_p(None)
    create = lambda d: lib.nt_decode_plan_create(ctypes.byref(d), ctypes.byref(h))  # noqa: E731
    arr = (nt.nt_proj * 7)()
    for i in range(7):
        arr[i] = nt.nt_proj(64, 48, 0x10000, 0x20000, None, 0x30000, 0x40000, 0x50000)
    d = nt.nt_decode_desc()
    d.n_layers, d.batch, d.proj = 1, 2, ctypes.cast(arr, ctypes.POINTER(nt.nt_proj))
    assert create(d) in REACHED_DEVICE
    d.launcher = 7
    assert create(d) == nt.NT_ERR_INVALID_ARG
    d.launcher = nt.NT_LAUNCH_GRAPH
    d.verify_emit, d.verify_n, d.verify_draft = 0x70000, 0x71000, 0x72000
    assert create(d) == nt.NT_ERR_INVALID_ARG  # acceptance needs the output projection
    d.head_T, d.head_s, d.head_V, d.head_K = 0x80000, 0x81000, 100, 64
    d.head_q, d.head_sx, d.head_argmax = 0x82000, 0x83000, 0x84000
    assert create(d) in REACHED_DEVICE
    d.verify_draft = None
    assert create(d) == nt.NT_ERR_INVALID_ARG  # two positions need a draft
    d.verify_draft = 0x72000
    d.head_K = 40
    assert create(d) == nt.NT_ERR_INVALID_ARG
    d.head_K = 64
    d.embed_T, d.embed_s, d.embed_V, d.embed_K, d.tokens, d.embed_x = 0x90000, 0x91000, 50, 48, 0x92000, 0x93008
    assert create(d) == nt.NT_ERR_ALIGNMENT  # the gathered rows must be 16-byte aligned
    d.embed_x = 0x93000
    assert create(d) in REACHED_DEVICE
    d.tokens = None
    assert create(d) == nt.NT_ERR_INVALID_ARG
    assert not h.value

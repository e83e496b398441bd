"""Thin ctypes binding of the C ABI in include/nt.h (libnt.so), with the same call names.

Argument marshalling only: every call passes device pointers of torch tensors (and the
current torch CUDA stream unless one is given) to the library, and raises :class:`NtError`
when the library returns a non-zero status. There is no fallback of any kind: if
``libnt.so`` has not been built, importing a call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional, Sequence

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_lib", "libnt.so")

NT_OK = 0
NT_ERR_INVALID_ARG = 1
NT_ERR_ALIGNMENT = 2
NT_ERR_UNSUPPORTED = 3
NT_ERR_CUDA = 4
NT_ERR_TIMEOUT = 5
NT_ERR_WORKSPACE = 6
NT_ERR_INVALID_CODE = 7

NT_LAYOUT_PLAIN = 0
NT_LAYOUT_TILED = 1
NT_STEP_INDEPENDENT = 0
NT_STEP_ORDERED = 1
NT_STEP_CHAINED = 2
NT_LAUNCH_PERSISTENT = 0
NT_LAUNCH_GRAPH = 1
NT_LAUNCH_STREAM = 2

# Every symbol include/nt.h declares.
EXPORTS = (
    "nt_abi_version", "nt_status_string", "nt_last_error_string", "nt_workspace_status",
    "nt_set_test_fault", "nt_device_check",
    "nt_quantize_act", "nt_repack_size", "nt_validate_ternary", "nt_repack_ternary", "nt_ternary_gemv",
    "nt_ternary_gemm_workspace_size", "nt_ternary_gemm", "nt_ternary_gemm_multi_workspace_size",
    "nt_ternary_gemm_multi", "nt_int8_logits_workspace_size", "nt_int8_logits_argmax",
    "nt_int8_logits_argmax_noalloc", "nt_embed_rows", "nt_verify_accept",
    "nt_attention_workspace_size", "nt_attention_decode", "nt_rope_append", "nt_rmsnorm",
    "nt_decode_plan_create", "nt_decode_step", "nt_decode_step_status", "nt_decode_plan_reset",
    "nt_decode_plan_set_position",
    "nt_decode_plan_trace_layout", "nt_decode_plan_set_trace", "nt_decode_plan_capture_size",
    "nt_decode_plan_set_capture", "nt_decode_plan_destroy",
)


class NtError(RuntimeError):
    def __init__(self, status: int, call: str, detail: str):
        self.status = status
        super().__init__(f"{call}: status {status} ({detail})")


class nt_proj(ctypes.Structure):
    _fields_ = [("N", ctypes.c_int), ("K", ctypes.c_int), ("w", ctypes.c_void_p),
                ("s_w", ctypes.c_void_p), ("x", ctypes.c_void_p), ("q", ctypes.c_void_p),
                ("s_x", ctypes.c_void_p), ("y", ctypes.c_void_p)]


class nt_decode_desc(ctypes.Structure):
    _fields_ = [("n_layers", ctypes.c_int), ("batch", ctypes.c_int),
                ("proj", ctypes.POINTER(nt_proj)),
                ("head_T", ctypes.c_void_p), ("head_s", ctypes.c_void_p),
                ("head_V", ctypes.c_int), ("head_K", ctypes.c_int),
                ("head_x", ctypes.c_void_p), ("head_q", ctypes.c_void_p),
                ("head_sx", ctypes.c_void_p), ("head_logits", ctypes.c_void_p),
                ("head_argmax", ctypes.c_void_p), ("mode", ctypes.c_int),
                ("launcher", ctypes.c_int), ("timeout_ms", ctypes.c_double),
                ("test_fault", ctypes.c_int),
                ("embed_T", ctypes.c_void_p), ("embed_s", ctypes.c_void_p),
                ("embed_V", ctypes.c_int), ("embed_K", ctypes.c_int),
                ("tokens", ctypes.c_void_p), ("embed_x", ctypes.c_void_p),
                ("verify_draft", ctypes.c_void_p), ("verify_emit", ctypes.c_void_p),
                ("verify_n", ctypes.c_void_p), ("head_dim", ctypes.c_int),
                ("attn_k_cache", ctypes.POINTER(ctypes.c_void_p)), ("attn_v_cache", ctypes.POINTER(ctypes.c_void_p)),
                ("attn_t_stride", ctypes.c_int), ("attn_pos", ctypes.c_int),
                ("rope_base", ctypes.c_float), ("norm_eps", ctypes.c_float),
                ("norm_attn", ctypes.POINTER(ctypes.c_void_p)), ("norm_ffn", ctypes.POINTER(ctypes.c_void_p)),
                ("norm_final", ctypes.c_void_p)]


_lock = threading.Lock()
_lib = None


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Loads libnt.so (once). Raises if it is missing: there is no other implementation."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is missing: build it with "
                               "`python -c 'import __graft_entry__ as g; g.build()'`")
        lib = ctypes.CDLL(path)
        i, vp, sz = ctypes.c_int, ctypes.c_void_p, ctypes.c_size_t
        sig = {
            "nt_abi_version": ([], i),
            "nt_status_string": ([i], ctypes.c_char_p),
            "nt_last_error_string": ([], ctypes.c_char_p),
            "nt_device_check": ([ctypes.POINTER(i)], i),
            "nt_workspace_status": ([vp, ctypes.POINTER(i)], i),
            "nt_set_test_fault": ([i, ctypes.c_double], i),
            "nt_quantize_act": ([vp, i, i, vp, vp, vp], i),
            "nt_repack_size": ([i, i, ctypes.POINTER(sz)], i),
            "nt_repack_ternary": ([vp, i, i, vp, vp, vp], i),
            "nt_validate_ternary": ([vp, i, i, ctypes.POINTER(ctypes.c_uint64), vp], i),
            "nt_ternary_gemv": ([vp, i, vp, i, i, vp, vp, vp, vp, vp], i),
            "nt_ternary_gemm_workspace_size": ([i, i, i, i, ctypes.POINTER(sz)], i),
            "nt_ternary_gemm": ([vp, i, vp, i, i, vp, vp, i, vp, vp, vp, sz, vp], i),
            "nt_ternary_gemm_multi_workspace_size": ([i, ctypes.POINTER(i), i, i, ctypes.POINTER(sz)], i),
            "nt_ternary_gemm_multi": ([i, ctypes.POINTER(vp), ctypes.POINTER(vp), ctypes.POINTER(i), i, vp, vp, i,
                                       ctypes.POINTER(vp), ctypes.POINTER(vp), vp, sz, vp], i),
            "nt_int8_logits_workspace_size": ([i, i, i, ctypes.POINTER(sz)], i),
            "nt_int8_logits_argmax": ([vp, vp, i, i, vp, vp, i, vp, vp, vp, sz, vp], i),
            "nt_int8_logits_argmax_noalloc": ([vp, vp, i, i, vp, vp, i, vp, vp, vp], i),
            "nt_embed_rows": ([vp, vp, i, i, vp, i, vp, vp, vp], i),
            "nt_verify_accept": ([vp, vp, i, vp, vp, vp], i),
            "nt_attention_workspace_size": ([i, i, i, i, ctypes.POINTER(sz)], i),
            "nt_attention_decode": ([vp, vp, vp, i, i, i, i, i, i, vp, vp, sz, vp], i),
            "nt_rope_append": ([vp, vp, vp, i, i, i, i, i, ctypes.c_float, vp, vp, vp, i, vp], i),
            "nt_rmsnorm": ([vp, vp, i, i, ctypes.c_float, vp, vp], i),
            "nt_decode_plan_create": ([ctypes.POINTER(nt_decode_desc), ctypes.POINTER(vp)], i),
            "nt_decode_step": ([vp, vp], i),
            "nt_decode_step_status": ([vp, ctypes.POINTER(i)], i),
            "nt_decode_plan_reset": ([vp], i),
            "nt_decode_plan_set_position": ([vp, i, vp], i),
            "nt_decode_plan_trace_layout": ([vp, ctypes.POINTER(i), ctypes.POINTER(i)], i),
            "nt_decode_plan_set_trace": ([vp, vp], i),
            "nt_decode_plan_capture_size": ([vp, ctypes.POINTER(sz)], i),
            "nt_decode_plan_set_capture": ([vp, vp], i),
            "nt_decode_plan_destroy": ([vp], None),
        }
        for name, (args, res) in sig.items():
            f = getattr(lib, name)
            f.argtypes = args
            f.restype = res
        _lib = lib
        return lib


def _check(status: int, call: str):
    if status != NT_OK:
        lib = load_library()
        detail = lib.nt_last_error_string().decode() or lib.nt_status_string(status).decode()
        raise NtError(status, call, detail)


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def nt_abi_version() -> int:
    return load_library().nt_abi_version()


def nt_workspace_status(ws: torch.Tensor) -> int:
    """NT_OK or NT_ERR_TIMEOUT from a workspace's status header (synchronous)."""
    st = ctypes.c_int(0)
    _check(load_library().nt_workspace_status(_ptr(ws), ctypes.byref(st)), "nt_workspace_status")
    return st.value


def nt_set_test_fault(fault: int, timeout_ms: float = 0.0):
    """Test hook of the per-call timeout paths (0 = off)."""
    _check(load_library().nt_set_test_fault(fault, timeout_ms), "nt_set_test_fault")


def nt_device_check() -> int:
    n = ctypes.c_int(0)
    _check(load_library().nt_device_check(ctypes.byref(n)), "nt_device_check")
    return n.value


def nt_quantize_act(x: torch.Tensor, q: torch.Tensor, s_x: torch.Tensor, stream=None):
    B, K = (1, x.numel()) if x.dim() == 1 else x.shape
    _check(load_library().nt_quantize_act(_ptr(x), B, K, _ptr(q), _ptr(s_x), _stream(stream)),
           "nt_quantize_act")


def nt_repack_size(N: int, K: int) -> int:
    n = ctypes.c_size_t(0)
    _check(load_library().nt_repack_size(N, K, ctypes.byref(n)), "nt_repack_size")
    return n.value


def nt_validate_ternary(w_plain: torch.Tensor, N: int, K: int, stream=None) -> int:
    """Number of invalid 10 fields in a plain matrix (0 when valid); synchronous."""
    n = ctypes.c_uint64(0)
    st = load_library().nt_validate_ternary(_ptr(w_plain), N, K, ctypes.byref(n), _stream(stream))
    if st not in (NT_OK, NT_ERR_INVALID_CODE):
        _check(st, "nt_validate_ternary")
    return n.value


def nt_repack_ternary(w_plain: torch.Tensor, N: int, K: int, w_tiled: torch.Tensor,
                      n_invalid: Optional[torch.Tensor] = None, stream=None):
    _check(load_library().nt_repack_ternary(_ptr(w_plain), N, K, _ptr(w_tiled), _ptr(n_invalid),
                                            _stream(stream)), "nt_repack_ternary")


def nt_ternary_gemv(w: torch.Tensor, layout: int, s_w: torch.Tensor, N: int, K: int,
                    q: torch.Tensor, s_x: torch.Tensor, y: torch.Tensor,
                    acc: Optional[torch.Tensor] = None, stream=None):
    _check(load_library().nt_ternary_gemv(_ptr(w), layout, _ptr(s_w), N, K, _ptr(q), _ptr(s_x),
                                          _ptr(y), _ptr(acc), _stream(stream)), "nt_ternary_gemv")


def nt_ternary_gemm_workspace_size(N: int, K: int, B: int, layout: int) -> int:
    n = ctypes.c_size_t(0)
    _check(load_library().nt_ternary_gemm_workspace_size(N, K, B, layout, ctypes.byref(n)),
           "nt_ternary_gemm_workspace_size")
    return n.value


def nt_ternary_gemm(w: torch.Tensor, layout: int, s_w: torch.Tensor, N: int, K: int,
                    q: torch.Tensor, s_x: torch.Tensor, B: int, y: torch.Tensor,
                    acc: Optional[torch.Tensor] = None, ws: Optional[torch.Tensor] = None,
                    stream=None):
    ws_bytes = 0 if ws is None else ws.numel() * ws.element_size()
    _check(load_library().nt_ternary_gemm(_ptr(w), layout, _ptr(s_w), N, K, _ptr(q), _ptr(s_x), B,
                                          _ptr(y), _ptr(acc), _ptr(ws), ws_bytes, _stream(stream)),
           "nt_ternary_gemm")


def nt_ternary_gemm_multi_workspace_size(N: Sequence[int], K: int, B: int) -> int:
    n = ctypes.c_size_t(0)
    arr = (ctypes.c_int * len(N))(*N)
    _check(load_library().nt_ternary_gemm_multi_workspace_size(len(N), arr, K, B, ctypes.byref(n)),
           "nt_ternary_gemm_multi_workspace_size")
    return n.value


def nt_ternary_gemm_multi(w: Sequence[torch.Tensor], s_w: Sequence[torch.Tensor], N: Sequence[int], K: int,
                          q: torch.Tensor, s_x: torch.Tensor, B: int, y: Sequence[torch.Tensor],
                          acc: Optional[Sequence[Optional[torch.Tensor]]] = None,
                          ws: Optional[torch.Tensor] = None, stream=None):
    n = len(w)
    vp = ctypes.c_void_p
    wa = (vp * n)(*[t.data_ptr() for t in w])
    sa = (vp * n)(*[t.data_ptr() for t in s_w])
    na = (ctypes.c_int * n)(*N)
    ya = (vp * n)(*[t.data_ptr() for t in y])
    aa = None if acc is None else (vp * n)(*[None if t is None else t.data_ptr() for t in acc])
    ws_bytes = 0 if ws is None else ws.numel() * ws.element_size()
    _check(load_library().nt_ternary_gemm_multi(n, wa, sa, na, K, _ptr(q), _ptr(s_x), B, ya, aa, _ptr(ws),
                                                ws_bytes, _stream(stream)), "nt_ternary_gemm_multi")


def nt_int8_logits_workspace_size(V: int, K: int, B: int) -> int:
    n = ctypes.c_size_t(0)
    _check(load_library().nt_int8_logits_workspace_size(V, K, B, ctypes.byref(n)),
           "nt_int8_logits_workspace_size")
    return n.value


def nt_int8_logits_argmax(T: torch.Tensor, s_T: torch.Tensor, V: int, K: int, q: torch.Tensor,
                          s_x: torch.Tensor, B: int, logits: Optional[torch.Tensor],
                          argmax: torch.Tensor, ws: torch.Tensor, stream=None):
    _check(load_library().nt_int8_logits_argmax(
        _ptr(T), _ptr(s_T), V, K, _ptr(q), _ptr(s_x), B, _ptr(logits), _ptr(argmax), _ptr(ws),
        ws.numel() * ws.element_size(), _stream(stream)), "nt_int8_logits_argmax")


def nt_int8_logits_argmax_noalloc(T: torch.Tensor, s_T: torch.Tensor, V: int, K: int,
                                  q: torch.Tensor, s_x: torch.Tensor, B: int,
                                  logits: Optional[torch.Tensor], argmax: torch.Tensor,
                                  stream=None):
    """nt_int8_logits_argmax without a workspace, for callers that cannot allocate device
    memory; B <= 16, and calls on one device must not overlap (they share fixed scratch)."""
    _check(load_library().nt_int8_logits_argmax_noalloc(
        _ptr(T), _ptr(s_T), V, K, _ptr(q), _ptr(s_x), B, _ptr(logits), _ptr(argmax),
        _stream(stream)), "nt_int8_logits_argmax_noalloc")


def nt_embed_rows(T: torch.Tensor, s_T: torch.Tensor, V: int, K: int, tokens: torch.Tensor,
                  B: int, x: torch.Tensor, n_bad: Optional[torch.Tensor] = None, stream=None):
    _check(load_library().nt_embed_rows(_ptr(T), _ptr(s_T), V, K, _ptr(tokens), B, _ptr(x),
                                        _ptr(n_bad), _stream(stream)), "nt_embed_rows")


def nt_verify_accept(draft: Optional[torch.Tensor], argmax: torch.Tensor, B: int,
                     emit: torch.Tensor, n_emit: torch.Tensor, stream=None):
    _check(load_library().nt_verify_accept(_ptr(draft), _ptr(argmax), B, _ptr(emit), _ptr(n_emit),
                                           _stream(stream)), "nt_verify_accept")


def nt_attention_workspace_size(B: int, Hq: int, Hkv: int, T: int) -> int:
    n = ctypes.c_size_t(0)
    _check(load_library().nt_attention_workspace_size(B, Hq, Hkv, T, ctypes.byref(n)), "nt_attention_workspace_size")
    return n.value


def nt_attention_decode(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor, B: int, Hq: int,
                        Hkv: int, D: int, T: int, t_stride: int, out: torch.Tensor, ws: torch.Tensor,
                        stream=None):
    _check(load_library().nt_attention_decode(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), B, Hq, Hkv, D, T, t_stride, _ptr(out), _ptr(ws),
        ws.numel() * ws.element_size(), _stream(stream)), "nt_attention_decode")


def nt_rope_append(q: torch.Tensor, k_new: torch.Tensor, v_new: torch.Tensor, B: int, Hq: int, Hkv: int,
                   D: int, pos0: int, base: float, q_out: torch.Tensor, k_cache: torch.Tensor,
                   v_cache: torch.Tensor, t_stride: int, stream=None):
    _check(load_library().nt_rope_append(
        _ptr(q), _ptr(k_new), _ptr(v_new), B, Hq, Hkv, D, pos0, base, _ptr(q_out), _ptr(k_cache),
        _ptr(v_cache), t_stride, _stream(stream)), "nt_rope_append")


def nt_rmsnorm(x: torch.Tensor, gamma: torch.Tensor, B: int, D: int, eps: float, y: torch.Tensor,
               stream=None):
    _check(load_library().nt_rmsnorm(_ptr(x), _ptr(gamma), B, D, eps, _ptr(y), _stream(stream)), "nt_rmsnorm")


class DecodePlan:
    """Owns an nt_decode_plan and keeps every tensor it names alive.

    ``projs`` is a sequence of dicts with keys N, K, w, s_w, q, s_x, y and optionally x
    (torch tensors on the current device), n_layers * 7 of them in q, k, v, o, gate, up, down
    order per layer. ``head`` is None or a dict with T, s, V, K, q, sx, argmax and optionally
    x and logits. ``embed`` is None or a dict with T, s, V, K, tokens, x (the input-table
    gather that runs first; projection inputs may be views of its x). ``verify`` is None or a
    dict with emit, n and (for batch > 1) draft, applied to the head's arg-max.
    """

    def __init__(self, n_layers: int, batch: int, projs: Sequence[dict], head: Optional[dict],
                 mode: int = NT_STEP_INDEPENDENT, launcher: int = NT_LAUNCH_PERSISTENT,
                 timeout_ms: float = 0.0, test_fault: int = 0, embed: Optional[dict] = None,
                 verify: Optional[dict] = None, head_dim: int = 0, attention: Optional[dict] = None):
        lib = load_library()
        self._keep = [projs, head, embed, verify, attention]
        arr = (nt_proj * len(projs))()
        for i, p in enumerate(projs):
            arr[i] = nt_proj(p["N"], p["K"], p["w"].data_ptr(), p["s_w"].data_ptr(),
                             p["x"].data_ptr() if p.get("x") is not None else None,
                             p["q"].data_ptr(), p["s_x"].data_ptr(), p["y"].data_ptr())
        d = nt_decode_desc()
        d.n_layers, d.batch, d.proj = n_layers, batch, ctypes.cast(arr, ctypes.POINTER(nt_proj))
        if head is not None:
            d.head_T, d.head_s = head["T"].data_ptr(), head["s"].data_ptr()
            d.head_V, d.head_K = head["V"], head["K"]
            d.head_x = head["x"].data_ptr() if head.get("x") is not None else None
            d.head_q, d.head_sx = head["q"].data_ptr(), head["sx"].data_ptr()
            d.head_logits = head["logits"].data_ptr() if head.get("logits") is not None else None
            d.head_argmax = head["argmax"].data_ptr()
        d.mode, d.launcher, d.timeout_ms, d.test_fault = mode, launcher, timeout_ms, test_fault
        d.head_dim = head_dim
        if attention is not None:
            # dict: k_cache, v_cache (lists of device tensors per layer), t_stride, pos, and
            # optionally rope_base, eps, norm_attn / norm_ffn (lists), norm_final
            L = n_layers
            ptrs = lambda ts: (ctypes.c_void_p * L)(*[t.data_ptr() for t in ts])
            self._kc, self._vc = ptrs(attention["k_cache"]), ptrs(attention["v_cache"])
            d.attn_k_cache = ctypes.cast(self._kc, ctypes.POINTER(ctypes.c_void_p))
            d.attn_v_cache = ctypes.cast(self._vc, ctypes.POINTER(ctypes.c_void_p))
            d.attn_t_stride, d.attn_pos = attention["t_stride"], attention["pos"]
            d.rope_base = attention.get("rope_base", 0.0)
            d.norm_eps = attention.get("eps", 0.0)
            if attention.get("norm_attn") is not None:
                self._na = ptrs(attention["norm_attn"])
                d.norm_attn = ctypes.cast(self._na, ctypes.POINTER(ctypes.c_void_p))
            if attention.get("norm_ffn") is not None:
                self._nf = ptrs(attention["norm_ffn"])
                d.norm_ffn = ctypes.cast(self._nf, ctypes.POINTER(ctypes.c_void_p))
            if attention.get("norm_final") is not None:
                d.norm_final = attention["norm_final"].data_ptr()
        if embed is not None:
            d.embed_T, d.embed_s = embed["T"].data_ptr(), embed["s"].data_ptr()
            d.embed_V, d.embed_K = embed["V"], embed["K"]
            d.tokens, d.embed_x = embed["tokens"].data_ptr(), embed["x"].data_ptr()
        if verify is not None:
            d.verify_draft = verify["draft"].data_ptr() if verify.get("draft") is not None else None
            d.verify_emit, d.verify_n = verify["emit"].data_ptr(), verify["n"].data_ptr()
        self._arr = arr
        handle = ctypes.c_void_p(None)
        _check(lib.nt_decode_plan_create(ctypes.byref(d), ctypes.byref(handle)),
               "nt_decode_plan_create")
        self._h = handle

    def nt_decode_step(self, stream=None):
        _check(load_library().nt_decode_step(self._h, _stream(stream)), "nt_decode_step")

    def nt_decode_plan_set_position(self, pos: int, stream=None):
        _check(load_library().nt_decode_plan_set_position(self._h, pos, _stream(stream)),
               "nt_decode_plan_set_position")

    def nt_decode_step_status(self) -> int:
        s = ctypes.c_int(0)
        _check(load_library().nt_decode_step_status(self._h, ctypes.byref(s)),
               "nt_decode_step_status")
        return s.value

    def nt_decode_plan_reset(self):
        _check(load_library().nt_decode_plan_reset(self._h), "nt_decode_plan_reset")

    def nt_decode_plan_trace_layout(self):
        """(grid, barriers per step) of the persistent launcher's timeline."""
        g, b = ctypes.c_int(0), ctypes.c_int(0)
        _check(load_library().nt_decode_plan_trace_layout(self._h, ctypes.byref(g), ctypes.byref(b)),
               "nt_decode_plan_trace_layout")
        return g.value, b.value

    def nt_decode_plan_set_trace(self, trace: Optional[torch.Tensor]):
        """Installs a device int64 tensor of grid * (barriers + 1) * 4 values (or None)."""
        self._trace = trace
        _check(load_library().nt_decode_plan_set_trace(self._h, _ptr(trace)), "nt_decode_plan_set_trace")

    def nt_decode_plan_capture_size(self) -> int:
        """Floats of the stage-input capture buffer of a chained plan."""
        n = ctypes.c_size_t(0)
        _check(load_library().nt_decode_plan_capture_size(self._h, ctypes.byref(n)), "nt_decode_plan_capture_size")
        return n.value

    def nt_decode_plan_set_capture(self, buf: Optional[torch.Tensor]):
        """Installs a device fp32 tensor of nt_decode_plan_capture_size() values (or None)."""
        self._capture = buf
        _check(load_library().nt_decode_plan_set_capture(self._h, _ptr(buf)), "nt_decode_plan_set_capture")

    def close(self):
        if getattr(self, "_h", None) and self._h.value:
            load_library().nt_decode_plan_destroy(self._h)
            self._h = ctypes.c_void_p(None)

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

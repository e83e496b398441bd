"""Helpers for the GPU parity tests: move seeded inputs to the device and build plans."""
import numpy as np
import torch

from packed_weight_gemv_gb300 import nt

DEV = torch.device("cuda:0")
RTOL = 1e-6  # fp32 outputs: relative error bound against the oracle


def dev(a: np.ndarray) -> torch.Tensor:
    if a.dtype == np.uint32:
        a = a.view(np.int32)
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


def host(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().numpy()


def tiled(w_plain: np.ndarray, N: int, K: int) -> torch.Tensor:
    w = torch.empty(nt.nt_repack_size(N, K), dtype=torch.uint8, device=DEV)
    nt.nt_repack_ternary(dev(w_plain), N, K, w)
    return w


def assert_close(got: np.ndarray, want: np.ndarray, what: str = ""):
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    err = np.abs(got - want)
    bad = err > RTOL * np.abs(want)
    assert not bad.any(), (f"{what}: {int(bad.sum())} of {bad.size} outputs beyond rel {RTOL}; "
                           f"first at {np.argwhere(bad)[0]} got {got[bad][0]} want {want[bad][0]}")


def plan_inputs(projs, head, B=1, quantize_in_step=True):
    """Device tensors for a decode plan from synth.workloads projections / head."""
    dp = []
    for p in projs:
        d = dict(N=p.N, K=p.K, w=tiled(p.w_plain, p.N, p.K), s_w=dev(p.s_w),
                 q=torch.empty((B, p.K), dtype=torch.int8, device=DEV),
                 s_x=torch.empty(B, dtype=torch.float32, device=DEV),
                 y=torch.full((B, p.N), float("nan"), dtype=torch.float32, device=DEV))
        if quantize_in_step:
            d["x"] = dev(p.x[:B])
        dp.append(d)
    hd = None
    if head is not None:
        hd = dict(T=dev(head.T), s=dev(head.s_T), V=head.V, K=head.K,
                  q=torch.empty((B, head.K), dtype=torch.int8, device=DEV),
                  sx=torch.empty(B, dtype=torch.float32, device=DEV),
                  logits=torch.full((B, head.V), float("nan"), dtype=torch.float32, device=DEV),
                  argmax=torch.full((B,), -1, dtype=torch.int32, device=DEV))
        if quantize_in_step:
            hd["x"] = dev(head.x[:B])
    return dp, hd

"""Helpers shared by the GPU parity tests: run the library and the oracle on the same inputs."""
from __future__ import annotations

import ctypes

import numpy as np
import torch

import chunked_ssd_scan_gb300 as pkg
import oracle
from chunked_ssd_scan_gb300 import workloads as wl

# Element-wise gates: |got - ref| <= tol * (1 + |ref|) on y and on the final state.
TOL = {"f32": 1e-4, "bf16": 2e-2}


def to_np(t):
    return None if t is None else t.detach().to("cpu", torch.float64).numpy()


GUARD_BYTES = 4096
GUARD_FILL = 0xFF   # every guard byte: 0xFFFF is a bf16 NaN, 0xFFFFFFFF an fp32 NaN


class Guarded:
    """A device buffer of `nbytes` carved out of a larger one with GUARD_BYTES of NaN pattern on
    each side; check() asserts that nothing wrote into either guard band."""

    def __init__(self, nbytes: int, dev: str, fill_inner: int = 0):
        self.base = torch.full((GUARD_BYTES + nbytes + GUARD_BYTES,), GUARD_FILL,
                               dtype=torch.uint8, device=dev)
        self.inner = self.base[GUARD_BYTES:GUARD_BYTES + nbytes]
        self.inner.fill_(fill_inner)

    def view(self, dtype, shape):
        return self.inner.view(dtype).view(shape)

    def check(self, what: str):
        lo = self.base[:GUARD_BYTES]
        hi = self.base[-GUARD_BYTES:]
        for name, band in (("before", lo), ("after", hi)):
            bad = int((band != GUARD_FILL).sum().item())
            assert bad == 0, f"{what}: {bad} bytes of the guard band {name} the buffer were written"


def gpu_ssd(inp: dict, chunk_len: int, dev: str = "cuda", final: bool = True,
            guard: bool = False, tf32: bool = False, valid_len=None):
    """One forward through the C ABI (ssd_chunked_forward_tf32 with tf32=True; valid lengths per
    sequence if given); the device-side error word of its workspace must be clean (a bounded
    wait that gave up would otherwise only show as wrong numbers).  With guard=True,
    y, the final state and the workspace sit between NaN-pattern guard bands that must be intact
    after the call (an out-of-bounds store that element-wise parity cannot see would show)."""
    d = {k: (v.to(dev) if v is not None else None) for k, v in inp.items()}
    kw = {}
    bands = []
    if guard:
        x, B = d["x"], d["B"]
        b, T, R, H, P = x.shape
        N = B.shape[4]
        gy = Guarded(x.numel() * x.element_size(), dev, fill_inner=GUARD_FILL)
        kw["y"] = gy.view(x.dtype, x.shape)
        bands.append((gy, "y"))
        if final:
            gf = Guarded(b * H * P * N * 4, dev, fill_inner=GUARD_FILL)
            kw["final_state"] = gf.view(torch.float32, (b, H, P, N))
            bands.append((gf, "final_state"))
        shape = pkg.shape_of(x, B, chunk_len, d["theta"] is not None)
        nws = int(pkg.load_library().ssd_chunked_workspace_bytes(ctypes.byref(shape)))
        gw = Guarded(nws, dev, fill_inner=0)   # a workspace starts with a zeroed header
        kw["workspace"] = gw.inner
        bands.append((gw, "workspace"))
    if valid_len is not None:
        kw["valid_len"] = torch.as_tensor(valid_len, dtype=torch.int64, device=dev)
    plan = pkg.SSDForwardPlan(d["x"], d["dA"], d["B"], d["C"], chunk_len=chunk_len,
                              theta=d["theta"], init_state=d["init_state"],
                              return_final_state=final, tf32=tf32, **kw)
    y, fin = plan()
    assert pkg.workspace_status(plan.workspace) == ("SSD_OK", 0)
    torch.cuda.synchronize()
    for g, what in bands:
        g.check(what)
    return to_np(y), to_np(fin)


def oracle_ssd(inp: dict):
    return oracle.ssd(to_np(inp["x"]), to_np(inp["dA"]), to_np(inp["B"]), to_np(inp["C"]),
                      to_np(inp["theta"]), to_np(inp["init_state"]))


def check_close(got, ref, tol, what):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, f"{what}: shape {got.shape} != {ref.shape}"
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    err = np.abs(got - ref)
    bound = tol * (1.0 + np.abs(ref))
    bad = err > bound
    if np.any(bad):
        idx = np.unravel_index(np.argmax(err - bound), err.shape)
        raise AssertionError(
            f"{what}: {int(bad.sum())} of {bad.size} elements outside tol {tol}: worst at {idx} "
            f"got {got[idx]:.6g} ref {ref[idx]:.6g} (max abs err {err.max():.3e})")
    nrel = float(np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-300))
    return float(err.max()), nrel


def check_close_inner(got, ref, tol, what, axis=1):
    """Gate for a gradient that is an inner product of two state-sized matrices per element
    (ddA_t = exp(dA_t) <dL/dh_t, h_{t-1}>): its fp32 rounding scales with the size of the
    summed terms, which is the size of the values along the time axis, not with |ref| of one
    element (the inner product crosses zero).  |got - ref| <= tol (1 + |ref|) + tol / 10 * the
    RMS of ref along `axis` (the same (batch, head) sequence)."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, f"{what}: shape {got.shape} != {ref.shape}"
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    rms = np.sqrt(np.mean(ref * ref, axis=axis, keepdims=True))
    err = np.abs(got - ref)
    bound = tol * (1.0 + np.abs(ref)) + 0.1 * tol * rms
    bad = err > bound
    if np.any(bad):
        idx = np.unravel_index(np.argmax(err - bound), err.shape)
        raise AssertionError(
            f"{what}: {int(bad.sum())} of {bad.size} elements outside the gate: worst at {idx} "
            f"got {got[idx]:.6g} ref {ref[idx]:.6g} bound {bound[idx]:.3g}")
    return float(err.max())


def slice_heads(inp: dict, cfg: wl.SSDConfig, b: int, h: int) -> dict:
    """The independent (batch b, head h) sub-problem, as a batch-1, one-head, one-group problem."""
    g = h // (cfg.nheads // cfg.ngroups)
    return {
        "x": inp["x"][b:b + 1, :, :, h:h + 1].contiguous(),
        "dA": inp["dA"][b:b + 1, :, h:h + 1].contiguous(),
        "B": inp["B"][b:b + 1, :, :, g:g + 1].contiguous(),
        "C": inp["C"][b:b + 1, :, :, g:g + 1].contiguous(),
        "theta": None if inp["theta"] is None else inp["theta"][b:b + 1, :, h:h + 1].contiguous(),
        "init_state": (None if inp["init_state"] is None
                       else inp["init_state"][b:b + 1, h:h + 1].contiguous()),
    }


def gpu_trap(inp: dict, chunk_len: int, dev: str = "cuda"):
    """One trapezoidal forward through the C ABI, workspace error word checked."""
    d = {k: (v.to(dev) if v is not None else None) for k, v in inp.items()}
    plan = pkg.SSDTrapezoidalPlan(d["x"], d["dA"], d["B"], d["C"], d["gamma"], d["beta"],
                                  chunk_len=chunk_len, theta=d["theta"], prev_x=d["prev_x"],
                                  prev_B=d["prev_B"], init_state=d["init_state"])
    y, fin = plan()
    assert pkg.workspace_status(plan.workspace) == ("SSD_OK", 0)
    torch.cuda.synchronize()
    return to_np(y), to_np(fin)


def oracle_trap(inp: dict):
    return oracle.ssd_trapezoidal(to_np(inp["x"]), to_np(inp["dA"]), to_np(inp["B"]),
                                  to_np(inp["C"]), to_np(inp["gamma"]), to_np(inp["beta"]),
                                  to_np(inp["theta"]), to_np(inp["init_state"]),
                                  to_np(inp["prev_x"]), to_np(inp["prev_B"]))

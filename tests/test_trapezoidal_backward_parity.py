"""Backward of the trapezoidal Mamba-3 forward through the C ABI vs the fp64 oracle's reverse
mode of the trapezoidal recurrence, element by element (GPU)."""
import pytest
import torch

import chunked_ssd_scan_gb300 as pkg
from chunked_ssd_scan_gb300 import workloads as wl
from tests.parity_util import TOL, check_close, check_close_inner, to_np
import oracle

pytestmark = pytest.mark.gpu

T = dict(trapezoidal=True)
CASES = [
    # SISO, three heads in three groups, ragged T (64-row chunks of the 2-channel expansion)
    wl.SSDConfig("tbwd_siso_f32", 2, 200, 3, 16, 16, 64, 1, 3, "f32", **T),
    # MIMO R = 2 with the rotation (4 write channels, B^ per head), two heads per group
    wl.SSDConfig("tbwd_mimo_rot_f32", 1, 256, 4, 16, 32, 64, 2, 2, "f32", theta=True, **T),
    # bf16 inputs, rotation, P = N = 64
    wl.SSDConfig("tbwd_rot_bf16", 1, 130, 2, 64, 64, 64, 1, 1, "bf16", theta=True, **T),
    # R = 4 (8 write channels), groups shared by two heads, no rotation
    wl.SSDConfig("tbwd_rank4_f32", 1, 70, 4, 32, 32, 64, 4, 2, "f32", **T),
]


def _draw(cfg, seed, variant):
    kw = dict(slow_decay=True, init_state=True) if variant == "slow_decay_init_prev" else {}
    inp = wl.make_trap_inputs(cfg, seed=seed, prev=variant != "no_prev", **kw)
    g = torch.Generator().manual_seed(seed + 5)
    b, Tn, R, H, P, N = cfg.batch, cfg.seqlen, cfg.mimo_rank, cfg.nheads, cfg.headdim, cfg.dstate
    inp["dy"] = torch.randn((b, Tn, R, H, P), generator=g)
    inp["dfinal"] = torch.randn((b, H, P, N), generator=g) if variant != "no_prev" else None
    return inp


def _gpu(inp):
    d = {k: (v.cuda() if v is not None else None) for k, v in inp.items()}
    out = pkg.ssd_trapezoidal_backward(d["x"], d["dA"], d["B"], d["C"], d["gamma"], d["beta"],
                                       d["dy"], theta=d["theta"], prev_x=d["prev_x"],
                                       prev_B=d["prev_B"], init_state=d["init_state"],
                                       dfinal=d["dfinal"])
    assert pkg.workspace_status(out.pop("workspace")) == ("SSD_OK", 0)
    torch.cuda.synchronize()
    return {k: to_np(v) for k, v in out.items() if v is not None}


def _oracle(inp):
    f = to_np
    return oracle.ssd_trap_backward(f(inp["x"]), f(inp["dA"]), f(inp["B"]), f(inp["C"]),
                                    f(inp["gamma"]), f(inp["beta"]), f(inp["dy"]),
                                    theta=f(inp["theta"]), init_state=f(inp["init_state"]),
                                    prev_x=f(inp["prev_x"]), prev_B=f(inp["prev_B"]),
                                    dfinal=f(inp["dfinal"]))


@pytest.mark.parametrize("cfg", CASES, ids=lambda c: c.name)
@pytest.mark.parametrize("variant", ["stated", "slow_decay_init_prev", "no_prev"])
def test_trapezoidal_backward_parity(cfg, variant):
    inp = _draw(cfg, 51, variant)
    got, ref = _gpu(inp), _oracle(inp)
    assert set(got) == set(ref), (sorted(got), sorted(ref))
    for k in sorted(ref):
        if k in ("ddA", "dtheta", "dgamma", "dbeta"):   # inner products of state-sized terms
            check_close_inner(got[k], ref[k], TOL["f32"], f"{cfg.name}/{variant} {k}")
        else:
            check_close(got[k], ref[k], TOL["f32"], f"{cfg.name}/{variant} {k}")


def test_trapezoidal_backward_rejections():
    lib = pkg.load_library()
    import ctypes
    ok = pkg.make_shape(1, 64, 2, 16, 16, 1, 2, 64, "f32", False)
    assert lib.ssd_trapezoidal_backward_workspace_bytes(ctypes.byref(ok)) > 0
    too_wide = pkg.make_shape(1, 64, 2, 16, 16, 1, 64, 64, "f32", False)   # 2R = 128 channels
    assert lib.ssd_trapezoidal_backward_workspace_bytes(ctypes.byref(too_wide)) == 0
    st = lib.ssd_trapezoidal_backward(ctypes.byref(too_wide), *([None] * 23), ctypes.c_size_t(0),
                                      None)
    assert pkg.STATUS[st] == "SSD_ERR_UNSUPPORTED"


def test_trapezoidal_backward_full_size_sampled():
    """The measured trapezoidal backward shape (T = 16384, 16 heads, P = N = 64, R = 2, one B/C
    group per head, rotation, f32) through the launch the bench times; the oracle recomputes
    heads 0 and 15 (each its own group, so every gradient of those heads is checked)."""
    cfg = wl.TRAP_BWD_F32
    inp = wl.make_trap_bwd_inputs(cfg, seed=0)   # the bench's inputs
    got = _gpu(inp)
    for h in (0, 15):
        hs = slice(h, h + 1)
        sub = {"x": inp["x"][:, :, :, hs], "dA": inp["dA"][:, :, hs],
               "B": inp["B"][:, :, :, hs], "C": inp["C"][:, :, :, hs],
               "gamma": inp["gamma"][:, :, hs], "beta": inp["beta"][:, :, hs],
               "theta": inp["theta"][:, :, hs], "dy": inp["dy"][:, :, :, hs],
               "init_state": inp["init_state"][:, hs], "dfinal": inp["dfinal"][:, hs],
               "prev_x": inp["prev_x"][:, :, hs], "prev_B": inp["prev_B"][:, :, hs]}
        ref = _oracle(sub)
        view = {"dx": got["dx"][:, :, :, hs], "ddA": got["ddA"][:, :, hs],
                "dB": got["dB"][:, :, :, hs], "dC": got["dC"][:, :, :, hs],
                "dgamma": got["dgamma"][:, :, hs], "dbeta": got["dbeta"][:, :, hs],
                "dtheta": got["dtheta"][:, :, hs], "dinit": got["dinit"][:, hs],
                "dprev_x": got["dprev_x"][:, :, hs], "dprev_B": got["dprev_B"][:, :, hs]}
        for k in sorted(ref):
            if k in ("ddA", "dtheta", "dgamma", "dbeta"):
                check_close_inner(view[k], ref[k], TOL["f32"], f"{k} head {h}")
            else:
                check_close(view[k], ref[k], TOL["f32"], f"{k} head {h}")


def test_trapezoidal_backward_reduces_to_the_plain_backward():
    """gamma = 1, beta = 0, no previous write: ssd_trapezoidal_backward equals
    ssd_chunked_backward on the same data (rotated), through two different GPU paths."""
    cfg = wl.SSDConfig("tbwd_plain", 1, 150, 4, 16, 32, 64, 2, 2, "f32", theta=True, **T)
    inp = _draw(cfg, 53, "slow_decay_init_prev")
    inp["gamma"] = torch.ones_like(inp["gamma"])
    inp["beta"] = torch.zeros_like(inp["beta"])
    inp["prev_x"] = inp["prev_B"] = None
    got = _gpu(inp)
    d = {k: (v.cuda() if v is not None else None) for k, v in inp.items()}
    plain = pkg.ssd_chunked_backward(d["x"], d["dA"], d["B"], d["C"], d["dy"], theta=d["theta"],
                                     init_state=d["init_state"], dfinal=d["dfinal"])
    torch.cuda.synchronize()
    # each path is within TOL of the oracle, so the two are within twice that of each other
    for k in ("dx", "ddA", "dB", "dC", "dtheta", "dinit"):
        gate = check_close_inner if k in ("ddA", "dtheta") else check_close
        gate(got[k], to_np(plain[k]), 2 * TOL["f32"], f"trapezoid(beta=0) vs plain {k}")

"""Backward of the unrotated SSD forward through the C ABI vs the fp64 oracle's reverse mode,
element by element (GPU)."""
import ctypes

import pytest
import torch

import chunked_ssd_scan_gb300 as pkg
from chunked_ssd_scan_gb300 import workloads as wl
from tests.parity_util import TOL, check_close, check_close_inner, to_np
import oracle

pytestmark = pytest.mark.gpu

CASES = [
    # SISO, two groups, ragged T (150 = 64 + 64 + 22 steps per 64-row chunk)
    wl.SSDConfig("bwd_siso_f32", 2, 150, 4, 16, 16, 64, 1, 2, "f32"),
    # MIMO R = 2 (32 steps per chunk), all heads in one group, ragged T
    wl.SSDConfig("bwd_mimo2_f32", 1, 100, 4, 32, 32, 64, 2, 1, "f32"),
    # P = N = 64, several chunks
    wl.SSDConfig("bwd_p64n64_f32", 1, 256, 2, 64, 64, 64, 1, 1, "f32"),
    # N = 128, MIMO R = 4, bf16 inputs
    wl.SSDConfig("bwd_n128_mimo4_bf16", 1, 70, 2, 64, 128, 64, 4, 1, "bf16"),
    # R = 3: 21 steps = 63 fused rows per chunk
    wl.SSDConfig("bwd_mimo3_f32", 1, 50, 2, 16, 32, 64, 3, 2, "f32"),
    # one step
    wl.SSDConfig("bwd_one_step_f32", 1, 1, 2, 16, 16, 64, 2, 1, "f32"),
    # R = 5 (12 steps = 60 rows per chunk), P = 48, N = 96: partial row and column tiles
    wl.SSDConfig("bwd_mimo5_p48_n96_f32", 1, 40, 2, 48, 96, 64, 5, 1, "f32"),
    # P = N = 20: two-wide column runs, odd tile edges, bf16
    wl.SSDConfig("bwd_p20_n20_bf16", 1, 70, 4, 20, 20, 64, 1, 2, "bf16"),
    # rotated: two heads per B/C group (dB, dC summed over differently turned heads), ragged T
    wl.SSDConfig("bwd_rot_siso_f32", 2, 150, 4, 16, 16, 64, 1, 2, "f32", theta=True),
    # rotated MIMO R = 2, bf16 inputs, one group
    wl.SSDConfig("bwd_rot_mimo2_bf16", 1, 100, 4, 32, 32, 64, 2, 1, "bf16", theta=True),
    # rotated P = N = 64 over four chunks
    wl.SSDConfig("bwd_rot_p64n64_f32", 1, 256, 2, 64, 64, 64, 1, 1, "f32", theta=True),
]

KEYS = ("dx", "ddA", "dB", "dC", "dinit")


def _keys(inp):
    return KEYS + (("dtheta",) if inp.get("theta") is not None else ())


def _check(got, ref, k, what):
    if k in ("ddA", "dtheta"):   # inner products of two state-sized matrices per element
        check_close_inner(got, ref, TOL["f32"], what)
    else:
        check_close(got, ref, TOL["f32"], what)


def _draw(cfg, seed, with_state):
    inp = wl.make_ssd_inputs(cfg, seed=seed, init_state=with_state)
    g = torch.Generator().manual_seed(seed + 1)
    b, T, R, H, P, N = cfg.batch, cfg.seqlen, cfg.mimo_rank, cfg.nheads, cfg.headdim, cfg.dstate
    inp["dy"] = torch.randn((b, T, R, H, P), generator=g)
    inp["dfinal"] = torch.randn((b, H, P, N), generator=g) if with_state else None
    return inp


def _gpu(inp):
    d = {k: (v.cuda() if v is not None else None) for k, v in inp.items()}
    shape = pkg.shape_of(d["x"], d["B"], 64, d.get("theta") is not None)
    ws = torch.zeros(pkg.ssd_backward_workspace_bytes(shape), dtype=torch.uint8, device="cuda")
    out = pkg.ssd_chunked_backward(d["x"], d["dA"], d["B"], d["C"], d["dy"],
                                   theta=d.get("theta"), init_state=d["init_state"],
                                   dfinal=d["dfinal"], workspace=ws)
    assert pkg.workspace_status(ws) == ("SSD_OK", 0)
    torch.cuda.synchronize()
    return {k: to_np(v) for k, v in out.items() if v is not None}


def _oracle(inp):
    return oracle.ssd_backward(to_np(inp["x"]), to_np(inp["dA"]), to_np(inp["B"]),
                               to_np(inp["C"]), to_np(inp["dy"]),
                               init_state=to_np(inp["init_state"]), dfinal=to_np(inp["dfinal"]),
                               theta=to_np(inp.get("theta")))


@pytest.mark.parametrize("cfg", CASES, ids=lambda c: c.name)
@pytest.mark.parametrize("with_state", [False, True], ids=["zero_state", "init_and_dfinal"])
def test_backward_parity(cfg, with_state):
    inp = _draw(cfg, 41, with_state)
    got, ref = _gpu(inp), _oracle(inp)
    for k in _keys(inp):
        _check(got[k], ref[k], k, f"{cfg.name} {k}")


def test_backward_slow_decay_long():
    """Slow decay over 1000 steps: gradients reach far back and grow large, so the relative
    gate tests the fp64 log-decay sums and the chunk-to-chunk carry."""
    cfg = wl.SSDConfig("bwd_slow_f32", 1, 1000, 2, 32, 32, 64, 1, 1, "f32")
    inp = wl.make_ssd_inputs(cfg, seed=43, slow_decay=True, init_state=True)
    g = torch.Generator().manual_seed(44)
    inp["dy"] = torch.randn((1, 1000, 1, 2, 32), generator=g)
    inp["dfinal"] = torch.randn((1, 2, 32, 32), generator=g)
    got, ref = _gpu(inp), _oracle(inp)
    for k in KEYS:
        _check(got[k], ref[k], k, f"slow {k}")


def test_backward_dinit_optional_and_repeatable():
    cfg = CASES[0]
    inp = _draw(cfg, 45, True)
    d = {k: (v.cuda() if v is not None else None) for k, v in inp.items()}
    a = pkg.ssd_chunked_backward(d["x"], d["dA"], d["B"], d["C"], d["dy"],
                                 init_state=d["init_state"], dfinal=d["dfinal"],
                                 return_dinit=False)
    b = pkg.ssd_chunked_backward(d["x"], d["dA"], d["B"], d["C"], d["dy"],
                                 init_state=d["init_state"], dfinal=d["dfinal"])
    torch.cuda.synchronize()
    assert a["dinit"] is None
    for k in ("dx", "ddA"):   # no atomics: bit-identical between calls
        assert torch.equal(a[k], b[k]), k
    for k in ("dB", "dC"):    # atomics over the 2 heads of a group: order may differ
        check_close(to_np(a[k]), to_np(b[k]), 1e-6, k)


def test_backward_rejections():
    lib = pkg.load_library()
    ok = pkg.make_shape(1, 64, 2, 16, 16, 1, 1, 64, "f32", False)
    assert lib.ssd_backward_workspace_bytes(ctypes.byref(ok)) > 0
    rot = pkg.make_shape(1, 64, 2, 16, 16, 1, 1, 64, "f32", True)
    assert lib.ssd_backward_workspace_bytes(ctypes.byref(rot)) > \
        lib.ssd_backward_workspace_bytes(ctypes.byref(ok))
    for bad in (pkg.make_shape(1, 64, 2, 128, 16, 1, 1, 64, "f32", False),   # headdim > 64
                pkg.make_shape(1, 64, 2, 16, 256, 1, 1, 64, "f32", False),   # dstate > 128
                pkg.make_shape(1, 64, 2, 16, 16, 1, 128, 64, "f32", False),  # rank > 64
                pkg.make_shape(1, 64, 2, 16, 18, 1, 1, 64, "f32", False)):   # dstate % 4
        assert lib.ssd_backward_workspace_bytes(ctypes.byref(bad)) == 0
        st = lib.ssd_chunked_backward(ctypes.byref(bad), *([None] * 15), ctypes.c_size_t(0),
                                      None)
        assert pkg.STATUS[st] == "SSD_ERR_UNSUPPORTED"
    x = torch.zeros((1, 64, 1, 2, 16), device="cuda")
    B = torch.zeros((1, 64, 1, 1, 16), device="cuda")
    dA = torch.zeros((1, 64, 2), device="cuda")
    th = torch.zeros((1, 64, 2, 8), device="cuda")
    P_ = pkg._ptr

    def call(shape, theta, ddA, dtheta):
        return pkg.STATUS[lib.ssd_chunked_backward(
            ctypes.byref(shape), P_(x), P_(dA), P_(B), P_(B), theta, None, P_(x), None, P_(x),
            ddA, P_(B), P_(B), dtheta, None, None, ctypes.c_size_t(0), None)]

    assert call(ok, None, None, None) == "SSD_ERR_INVALID_ARG"            # ddA missing
    assert call(rot, None, P_(dA), P_(th)) == "SSD_ERR_INVALID_ARG"       # theta missing
    assert call(rot, P_(th), P_(dA), None) == "SSD_ERR_INVALID_ARG"       # dtheta missing
    assert call(ok, P_(th), P_(dA), P_(th)) == "SSD_ERR_INVALID_ARG"      # theta, no has_theta


def test_backward_full_size_sampled():
    """The measured backward shape (4 x 4096 steps, 32 heads, P 64, N 128, bf16 inputs) through
    the launch the bench times; the oracle recomputes two whole sampled sequences (every head,
    so the group sums dB and dC are checked too)."""
    cfg = wl.MAMBA2_BWD_BF16
    inp = wl.make_bwd_inputs(cfg, seed=0)   # the bench's inputs
    got = _gpu(inp)
    for b in (0, 3):
        sub = {k: (v[b:b + 1] if v is not None else None) for k, v in inp.items()}
        ref = _oracle(sub)
        for k in _keys(inp):
            _check(got[k][b:b + 1], ref[k], k, f"{k} batch {b}")


def test_rotated_backward_full_size_sampled():
    """The measured rotated backward shape (T = 131072, 24 heads, P = N = 64, one B/C group per
    head, f32) through the launch the bench times; the oracle recomputes heads 0 and 23 (each
    head its own group, so every gradient of those heads is checked)."""
    cfg = wl.LONG_ROT_BWD_F32
    inp = wl.make_bwd_inputs(cfg, seed=0)   # the bench's inputs
    got = _gpu(inp)
    for h in (0, 23):
        sub = {"x": inp["x"][:, :, :, h:h + 1], "dA": inp["dA"][:, :, h:h + 1],
               "B": inp["B"][:, :, :, h:h + 1], "C": inp["C"][:, :, :, h:h + 1],
               "theta": inp["theta"][:, :, h:h + 1], "dy": inp["dy"][:, :, :, h:h + 1],
               "init_state": inp["init_state"][:, h:h + 1], "dfinal": inp["dfinal"][:, h:h + 1]}
        ref = _oracle(sub)
        view = {"dx": got["dx"][:, :, :, h:h + 1], "ddA": got["ddA"][:, :, h:h + 1],
                "dB": got["dB"][:, :, :, h:h + 1], "dC": got["dC"][:, :, :, h:h + 1],
                "dtheta": got["dtheta"][:, :, h:h + 1], "dinit": got["dinit"][:, h:h + 1]}
        for k in _keys(sub):
            _check(view[k], ref[k], k, f"{k} head {h}")

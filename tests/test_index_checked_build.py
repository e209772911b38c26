"""The index-checked debug library (GPU): every checked output store of the kernels compares its
element index with its buffer's extent, skips the store if it falls outside and latches
SSD_ERR_INDEX with the store's site in the workspace.  The shapes here are the ones whose edges
an out-of-bounds store would hide in: ragged last tiles and chunks, MIMO ranks, time segments,
valid lengths ending mid-tile, partial channel blocks of the selective scan, both trapezoid
forms.  Each runs through the checked library and the normal one on the same inputs: no check
may fire and the outputs must agree.
"""
import ctypes

import pytest
import torch

import chunked_ssd_scan_gb300 as pkg
from chunked_ssd_scan_gb300 import _build
from chunked_ssd_scan_gb300 import workloads as wl
from tests.parity_util import check_close, to_np

pytestmark = pytest.mark.gpu

T = dict(trapezoidal=True)
SSD_SHAPES = [
    (wl.SSDConfig("ck_fused_ragged", 2, 700, 4, 64, 128, 256, 1, 1, "bf16"), None),
    (wl.SSDConfig("ck_fused_mimo_segments", 1, 1000, 4, 64, 128, 64, 4, 4, "bf16"), None),
    (wl.SSDConfig("ck_fused_varlen", 3, 300, 4, 64, 128, 64, 2, 2, "bf16"), [300, 97, 1]),
    (wl.SSDConfig("ck_tc32_rot_ragged", 2, 333, 4, 64, 64, 256, 1, 4, "f32", theta=True), None),
    (wl.SSDConfig("ck_generic_mimo", 2, 150, 3, 16, 32, 64, 2, 3, "f32", theta=True), [150, 77]),
]
TRAP_SHAPES = [
    wl.SSDConfig("ck_trap_fused", 2, 300, 4, 64, 128, 64, 2, 2, "bf16", **T),
    wl.SSDConfig("ck_trap_tc32_rot", 1, 200, 4, 64, 64, 64, 2, 4, "f32", theta=True, **T),
]
SS_SHAPES = [
    wl.SelectiveScanConfig("ck_ss_lookback", 2, 1000, 20, 16),
    wl.SelectiveScanConfig("ck_ss_segmented", 1, 333, 50, 32),
]


@pytest.fixture(scope="module")
def checked():
    return pkg.load_library(_build.build_checked())


def _run(fn, args):
    st = fn(*args)
    assert st == 0, pkg.STATUS.get(st, st)
    torch.cuda.synchronize()


@pytest.mark.parametrize("case", SSD_SHAPES, ids=lambda c: c[0].name)
def test_forward_shapes_fire_no_index_check(checked, case):
    cfg, lens = case
    inp = {k: (None if v is None else v.cuda())
           for k, v in wl.make_ssd_inputs(cfg, seed=41, slow_decay=True, init_state=True).items()}
    vl = None if lens is None else torch.tensor(lens, dtype=torch.int64, device="cuda")
    outs = []
    for lib in (None, checked):
        plan = pkg.SSDForwardPlan(inp["x"], inp["dA"], inp["B"], inp["C"], chunk_len=cfg.chunk_len,
                                  theta=inp["theta"], init_state=inp["init_state"], valid_len=vl)
        if lib is None:
            plan()
        else:
            _run(getattr(lib, plan._name), plan._args)
        torch.cuda.synchronize()
        assert pkg.workspace_status(plan.workspace) == ("SSD_OK", 0), cfg.name
        outs.append((to_np(plan.y), to_np(plan.final_state)))
    (y0, f0), (y1, f1) = outs
    if lens is not None:   # y past each length is not written: compare the real steps only
        for b, L in enumerate(lens):
            check_close(y1[b, :L], y0[b, :L], 1e-6, f"{cfg.name} y seq {b}")
    else:
        check_close(y1, y0, 1e-6, f"{cfg.name} y")
    check_close(f1, f0, 1e-6, f"{cfg.name} final_state")


@pytest.mark.parametrize("cfg", TRAP_SHAPES, ids=lambda c: c.name)
def test_trapezoid_shapes_fire_no_index_check(checked, cfg):
    inp = {k: (None if v is None else v.cuda())
           for k, v in wl.make_trap_inputs(cfg, seed=42, prev=True, init_state=True).items()}
    outs = []
    for lib in (None, checked):
        plan = pkg.SSDTrapezoidalPlan(inp["x"], inp["dA"], inp["B"], inp["C"], inp["gamma"],
                                      inp["beta"], chunk_len=cfg.chunk_len, theta=inp["theta"],
                                      prev_x=inp["prev_x"], prev_B=inp["prev_B"],
                                      init_state=inp["init_state"])
        if lib is None:
            plan()
        else:
            _run(getattr(lib, plan._name), plan._args)
        torch.cuda.synchronize()
        assert pkg.workspace_status(plan.workspace) == ("SSD_OK", 0), cfg.name
        outs.append((to_np(plan.y), to_np(plan.final_state)))
    check_close(outs[1][0], outs[0][0], 1e-6, f"{cfg.name} y")
    check_close(outs[1][1], outs[0][1], 1e-6, f"{cfg.name} final_state")


@pytest.mark.parametrize("cfg", SS_SHAPES, ids=lambda c: c.name)
def test_selective_scan_shapes_fire_no_index_check(checked, cfg):
    s = wl.make_selective_scan_inputs(cfg, seed=43, device="cuda")
    ref = pkg.selective_scan_forward(s["u"], s["delta"], s["A"], s["B"], s["C"], s["skip"])
    fn = checked.selective_scan_forward
    fn.restype = ctypes.c_int
    fn.argtypes = [ctypes.c_void_p] * 7 + [ctypes.c_int64] * 4 + [ctypes.c_void_p, ctypes.c_size_t,
                                                                   ctypes.c_void_p]
    n = int(pkg.load_library().selective_scan_workspace_bytes(cfg.batch, cfg.seqlen, cfg.d_model,
                                                             cfg.d_state))
    ws = torch.zeros(n, dtype=torch.uint8, device="cuda")
    y = torch.full_like(s["u"], float("nan"))
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    _run(fn, [p(s[k]) for k in ("u", "delta", "A", "B", "C", "skip")] + [
        p(y), cfg.batch, cfg.seqlen, cfg.d_model, cfg.d_state, p(ws), ctypes.c_size_t(n),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)])
    assert pkg.workspace_status(ws) == ("SSD_OK", 0), cfg.name
    check_close(to_np(y), to_np(ref), 1e-6, f"{cfg.name} y")

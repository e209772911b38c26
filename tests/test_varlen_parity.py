"""Per-sequence valid lengths: ssd_chunked_forward_varlen and ssd_trapezoidal_forward_varlen
against the fp64 oracle run on each sequence cut at its length.

moments.rs page (module header and state_moments_phys): a batch of sequences of different
lengths is zero-padded to one length; a pad step has zero log-decay (an identity decay) and a
zero write, so the state passes through unchanged and the carry is the state at the last real
step; the rotation at pads is irrelevant.  So y at the real steps and the final state are those
of the sequence cut at its length, which the oracle computes by its own definition.

Every input at pad steps is set to NaN here: a kernel that read one into a real output would
show it.  y starts as NaN bytes inside guard bands: pad steps must still hold the exact bytes
afterwards (never written), and nothing may be written outside the buffers.
"""
import ctypes

import numpy as np
import pytest
import torch

import chunked_ssd_scan_gb300 as pkg
import oracle
from chunked_ssd_scan_gb300 import workloads as wl
from tests.parity_util import (GUARD_FILL, TOL, Guarded, check_close, oracle_ssd, oracle_trap,
                               to_np)

# (config, valid lengths per sequence, the kernel family the shape selects)
SSD_CASES = [
    # tensor-core path: a full sequence, one ending inside a tile, one on a tile boundary, empty
    (wl.SSDConfig("vl_fused_siso_bf16", 4, 700, 4, 64, 128, 256, 1, 1, "bf16"),
     [700, 513, 128, 0], "tc_bf16"),
    # MIMO rank 4: 32 steps per tile, the end inside a 32-row quarter
    (wl.SSDConfig("vl_fused_mimo_bf16", 3, 300, 4, 64, 128, 64, 4, 4, "bf16"),
     [300, 97, 1], "tc_bf16"),
    # few sequences on a long axis: time segments with the state-only pre-pass; the second
    # sequence ends in its third segment, so later segments run on padding only
    (wl.SSDConfig("vl_fused_segmented_bf16", 2, 4096, 4, 64, 128, 256, 1, 1, "bf16"),
     [4096, 1234], "tc_bf16"),
    (wl.SSDConfig("vl_tc32_f32", 3, 600, 4, 64, 64, 256, 1, 2, "f32"),
     [600, 300, 37], "tc_tf32"),
    (wl.SSDConfig("vl_tc32_rot_f32", 2, 700, 4, 64, 64, 256, 1, 4, "f32", theta=True),
     [513, 700], "tc_tf32"),
    (wl.SSDConfig("vl_generic_rot_mimo_f32", 3, 333, 3, 16, 32, 64, 2, 3, "f32", theta=True),
     [333, 200, 64], "generic"),
    (wl.SSDConfig("vl_generic_bf16", 2, 257, 2, 32, 32, 128, 1, 1, "bf16"),
     [100, 257], "generic"),
]

T = dict(trapezoidal=True)
TRAP_CASES = [
    (wl.SSDConfig("vl_trap_rot_f32", 3, 300, 4, 16, 32, 64, 2, 2, "f32", theta=True, **T),
     [300, 129, 0]),
    (wl.SSDConfig("vl_trap_bf16", 2, 256, 4, 64, 64, 64, 2, 2, "bf16", **T), [77, 256]),
    # the tensor-core form of the trapezoid
    (wl.SSDConfig("vl_trap_fused_bf16", 3, 300, 4, 64, 128, 64, 2, 2, "bf16", **T),
     [300, 129, 1]),
]

SSD_KEYS = ("x", "dA", "B", "C", "theta")
TRAP_KEYS = ("x", "dA", "B", "C", "theta", "gamma", "beta")


def _poison_pads(inp, lens, keys):
    """Every input at a pad step set to NaN (axis 1 is time for all of them)."""
    out = dict(inp)
    for k in keys:
        v = inp[k]
        if v is None:
            continue
        v = v.clone()
        for b, L in enumerate(lens):
            v[b, L:] = float("nan")
        out[k] = v
    return out


def _cut(inp, b, L, keys):
    sub = {}
    for k, v in inp.items():
        if v is None:
            sub[k] = None
        elif k in keys:
            sub[k] = v[b:b + 1, :L].contiguous()
        else:   # per-sequence tensors: init_state, prev_x, prev_B
            sub[k] = v[b:b + 1].contiguous()
    return sub


def _check(y, fin, inp, lens, keys, ref_fn, tol, what):
    """y [b,T,...] bytes at pads untouched; real steps and the final state vs the oracle."""
    for b, L in enumerate(lens):
        pad = y[b, L:]
        bad = int((pad.contiguous().view(torch.uint8) != GUARD_FILL).sum().item())
        assert bad == 0, f"{what}: {bad} bytes of y written at the pad steps of sequence {b}"
        if L == 0:   # nothing real: the final state is the initial one
            init = inp["init_state"]
            ref_f = np.zeros(fin[b].shape) if init is None else to_np(init[b])
            check_close(to_np(fin[b]), ref_f, tol, f"{what} seq {b} (empty) final")
            continue
        yr, fr = ref_fn(_cut(inp, b, L, keys))
        check_close(to_np(y[b:b + 1, :L]), yr, tol, f"{what} seq {b} (len {L}) y")
        check_close(to_np(fin[b:b + 1]), fr, tol, f"{what} seq {b} (len {L}) final")


@pytest.mark.gpu
@pytest.mark.parametrize("case", SSD_CASES, ids=lambda c: c[0].name)
def test_varlen_forward_matches_the_cut_sequences(case):
    cfg, lens, family = case
    inp = wl.make_ssd_inputs(cfg, seed=31, slow_decay=True, init_state=True)
    d = {k: (None if v is None else v.cuda()) for k, v in _poison_pads(inp, lens, SSD_KEYS).items()}
    x, B = d["x"], d["B"]
    b, Tn, R, H, P = x.shape
    N = B.shape[4]
    shape = pkg.shape_of(x, B, cfg.chunk_len, d["theta"] is not None)
    assert pkg.ssd_chunked_variant(shape) == family, cfg.name
    gy = Guarded(x.numel() * x.element_size(), "cuda", fill_inner=GUARD_FILL)
    gf = Guarded(b * H * P * N * 4, "cuda", fill_inner=GUARD_FILL)
    nws = int(pkg.load_library().ssd_chunked_workspace_bytes(ctypes.byref(shape)))
    gw = Guarded(nws, "cuda", fill_inner=0)
    vl = torch.tensor(lens, dtype=torch.int64, device="cuda")
    plan = pkg.SSDForwardPlan(x, d["dA"], B, d["C"], chunk_len=cfg.chunk_len, theta=d["theta"],
                              init_state=d["init_state"], y=gy.view(x.dtype, x.shape),
                              final_state=gf.view(torch.float32, (b, H, P, N)),
                              workspace=gw.inner, valid_len=vl)
    y, fin = plan()
    torch.cuda.synchronize()
    assert pkg.workspace_status(plan.workspace) == ("SSD_OK", 0)
    for g, what in ((gy, "y"), (gf, "final_state"), (gw, "workspace")):
        g.check(f"{cfg.name} {what}")
    _check(y, fin, inp, lens, SSD_KEYS, oracle_ssd, TOL[cfg.dtype], cfg.name)


@pytest.mark.gpu
def test_varlen_at_full_length_equals_the_plain_entry_point():
    """valid_len = seqlen everywhere: the same kernels and the same bits as ssd_chunked_forward."""
    cfg = wl.SSDConfig("vl_full_bf16", 2, 1000, 4, 64, 128, 256, 1, 1, "bf16")
    inp = {k: (None if v is None else v.cuda())
           for k, v in wl.make_ssd_inputs(cfg, seed=32, init_state=True).items()}
    args = (inp["x"], inp["dA"], inp["B"], inp["C"])
    kw = dict(chunk_len=cfg.chunk_len, init_state=inp["init_state"])
    y0, f0 = pkg.ssd_chunked_forward(*args, **kw)
    vl = torch.full((cfg.batch,), cfg.seqlen, dtype=torch.int64, device="cuda")
    y1, f1 = pkg.ssd_chunked_forward(*args, valid_len=vl, **kw)
    torch.cuda.synchronize()
    assert torch.equal(y0.view(torch.int16), y1.view(torch.int16))
    assert torch.equal(f0, f1)


@pytest.mark.gpu
@pytest.mark.parametrize("case", TRAP_CASES, ids=lambda c: c[0].name)
def test_varlen_trapezoidal_matches_the_cut_sequences(case):
    cfg, lens = case
    inp = wl.make_trap_inputs(cfg, seed=33, prev=True, slow_decay=True, init_state=True)
    d = {k: (None if v is None else v.cuda())
         for k, v in _poison_pads(inp, lens, TRAP_KEYS).items()}
    x = d["x"]
    b, Tn, R, H, P = x.shape
    N = d["B"].shape[4]
    gy = Guarded(x.numel() * x.element_size(), "cuda", fill_inner=GUARD_FILL)
    vl = torch.tensor(lens, dtype=torch.int64, device="cuda")
    plan = pkg.SSDTrapezoidalPlan(x, d["dA"], d["B"], d["C"], d["gamma"], d["beta"],
                                  chunk_len=cfg.chunk_len, theta=d["theta"], prev_x=d["prev_x"],
                                  prev_B=d["prev_B"], init_state=d["init_state"],
                                  y=gy.view(x.dtype, x.shape), valid_len=vl)
    y, fin = plan()
    torch.cuda.synchronize()
    assert pkg.workspace_status(plan.workspace) == ("SSD_OK", 0)
    gy.check(f"{cfg.name} y")
    _check(y, fin, inp, lens, TRAP_KEYS, oracle_trap, TOL[cfg.dtype], cfg.name)


@pytest.mark.gpu
def test_varlen_rejects_a_missing_or_misaligned_length_array():
    cfg = wl.SSDConfig("vl_reject", 1, 64, 2, 16, 16, 64, 1, 1, "f32")
    inp = {k: (None if v is None else v.cuda()) for k, v in wl.make_ssd_inputs(cfg).items()}
    shape = pkg.shape_of(inp["x"], inp["B"], cfg.chunk_len, False)
    lib = pkg.load_library()
    ws = torch.zeros(int(lib.ssd_chunked_workspace_bytes(ctypes.byref(shape))), dtype=torch.uint8,
                     device="cuda")
    y = torch.empty_like(inp["x"])
    raw = torch.zeros(3, dtype=torch.int64, device="cuda")
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    for vl in (ctypes.c_void_p(None), ctypes.c_void_p(raw.data_ptr() + 4)):
        st = lib.ssd_chunked_forward_varlen(ctypes.byref(shape), p(inp["x"]), p(inp["dA"]),
                                            p(inp["B"]), p(inp["C"]), None, vl, None, p(y), None,
                                            p(ws), ctypes.c_size_t(ws.numel()), None)
        assert st == 1, pkg.STATUS.get(st, st)   # INVALID_ARG, before any launch


def test_oracle_zero_pads_carry_the_state_through():
    """The reading the varlen entry points rest on, checked on the oracle: appending zero pad
    steps (dA = 0, x = 0, B = 0, theta = 0; C and the rest anything) leaves y at the real steps
    and the final state unchanged."""
    cfg = wl.SSDConfig("pad_pin", 1, 50, 2, 4, 6, 16, 2, 1, "f32", theta=True)
    inp = wl.make_ssd_inputs(cfg, seed=34, init_state=True)
    base = {k: to_np(v) for k, v in inp.items()}
    pad = 13
    rng = np.random.default_rng(0)
    padded = dict(base)
    for k in ("x", "dA", "B", "theta"):
        v = base[k]
        padded[k] = np.concatenate([v, np.zeros((1, pad) + v.shape[2:])], axis=1)
    c = base["C"]
    padded["C"] = np.concatenate([c, rng.standard_normal((1, pad) + c.shape[2:])], axis=1)
    y0, f0 = oracle.ssd(base["x"], base["dA"], base["B"], base["C"], base["theta"],
                        base["init_state"])
    y1, f1 = oracle.ssd(padded["x"], padded["dA"], padded["B"], padded["C"], padded["theta"],
                        padded["init_state"])
    np.testing.assert_allclose(y1[:, :cfg.seqlen], y0, rtol=0, atol=1e-12)
    np.testing.assert_allclose(f1, f0, rtol=0, atol=1e-12)

"""Quaternion rotation (moments.rs page, RotationSeq::Quaternion { cum_bshj4 }) on the GPU
through the C ABI vs the fp64 oracle, element by element (GPU)."""
import ctypes

import numpy as np
import pytest
import torch

import chunked_ssd_scan_gb300 as pkg
import oracle
from chunked_ssd_scan_gb300 import workloads as wl
from tests.parity_util import TOL, check_close, to_np

pytestmark = pytest.mark.gpu

CASES = [
    # fp32 P = N = 64 path after the turn (tf32 tensor-core chunk scan), several chunks
    wl.SSDConfig("quat_tc32_f32", 2, 600, 4, 64, 64, 128, 1, 2, "f32"),
    # generic path: MIMO rank 2, a group shared by three heads, ragged T, small odd P
    wl.SSDConfig("quat_generic_mimo_f32", 1, 203, 3, 5, 12, 32, 2, 1, "f32"),
    # bf16 I/O: widened around the fp32 problem
    wl.SSDConfig("quat_bf16", 2, 256, 4, 64, 128, 64, 1, 1, "bf16"),
]


def _run(cfg, inp, Q):
    d = {k: (v.cuda() if v is not None else None) for k, v in inp.items()}
    y, fin = pkg.ssd_quaternion_forward(d["x"], d["dA"], d["B"], d["C"], Q.cuda(),
                                        chunk_len=cfg.chunk_len, init_state=d["init_state"])
    torch.cuda.synchronize()
    return to_np(y), to_np(fin)


@pytest.mark.parametrize("cfg", CASES, ids=lambda c: c.name)
@pytest.mark.parametrize("variant", ["stated", "slow_decay_init"])
def test_quaternion_matches_oracle(cfg, variant):
    kw = dict(slow_decay=True, init_state=True) if variant == "slow_decay_init" else {}
    inp = wl.make_ssd_inputs(cfg, seed=4, **kw)
    Q = wl.make_quaternions(cfg.batch, cfg.seqlen, cfg.nheads, cfg.dstate, seed=5)
    y, fin = _run(cfg, inp, Q)
    yr, fr = oracle.ssd_quaternion(to_np(inp["x"]), to_np(inp["dA"]), to_np(inp["B"]),
                                   to_np(inp["C"]), to_np(Q), to_np(inp["init_state"]))
    check_close(y, yr, TOL[cfg.dtype], f"{cfg.name}/{variant} y")
    check_close(fin, fr, TOL[cfg.dtype], f"{cfg.name}/{variant} final_state")


def test_quaternion_i_axis_equals_angle_rotation_on_gpu():
    """Q = cos(Phi) + i sin(Phi) turns both pairs of each block like the angle rotation with the
    block's step angle on both of its pairs: the two GPU entry points agree."""
    cfg = wl.SSDConfig("quat_vs_angles", 1, 300, 2, 64, 64, 64, 1, 2, "f32", theta=True)
    inp = wl.make_ssd_inputs(cfg, seed=6, slow_decay=True, init_state=True)
    th = inp["theta"][..., ::2].contiguous()              # one angle per 4-block
    phi = torch.cumsum(th.double(), dim=1)
    Q = torch.zeros(th.shape + (4,), dtype=torch.float64)
    Q[..., 0], Q[..., 1] = torch.cos(phi), torch.sin(phi)
    yq, fq = _run(cfg, {**inp, "theta": None}, Q.float().contiguous())
    d = {k: (v.cuda() if v is not None else None) for k, v in inp.items()}
    th2 = th.repeat_interleave(2, dim=3).contiguous().cuda()
    ya, fa = pkg.ssd_chunked_forward(d["x"], d["dA"], d["B"], d["C"], chunk_len=cfg.chunk_len,
                                     theta=th2, init_state=d["init_state"])
    torch.cuda.synchronize()
    check_close(yq, to_np(ya), TOL["f32"], "quaternion vs angle rotation y")
    check_close(fq, to_np(fa), TOL["f32"], "quaternion vs angle rotation final_state")


def test_quaternion_rejections():
    cfg = wl.SSDConfig("quat_bad", 1, 64, 2, 8, 6, 32, 1, 1, "f32")   # dstate 6: not 4-blocks
    shape = pkg.make_shape(cfg.batch, cfg.seqlen, cfg.nheads, cfg.headdim, cfg.dstate,
                           cfg.ngroups, cfg.mimo_rank, cfg.chunk_len, cfg.dtype, False)
    lib = pkg.load_library()
    assert lib.ssd_quaternion_workspace_bytes(ctypes.byref(shape)) == 0
    ok = pkg.make_shape(1, 64, 2, 8, 8, 1, 1, 32, "f32", True)     # has_theta set: rejected
    assert lib.ssd_quaternion_workspace_bytes(ctypes.byref(ok)) == 0

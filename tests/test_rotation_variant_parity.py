"""Rotation variants (partial rope_dim, split-halves pairing) through the C ABI vs the fp64
oracle, element by element (GPU)."""
import pytest
import torch

import chunked_ssd_scan_gb300 as pkg
from chunked_ssd_scan_gb300 import workloads as wl
from tests.parity_util import TOL, check_close, to_np
import oracle

pytestmark = pytest.mark.gpu

CASES = [
    # generic path (P, N small), MIMO with groups, ragged T
    wl.SSDConfig("rot_generic_f32", 2, 150, 4, 16, 16, 64, 2, 2, "f32", theta=True),
    # fp32 P = N = 64 path (tf32 tensor-core chunk scan)
    wl.SSDConfig("rot_tc32_f32", 1, 256, 3, 64, 64, 64, 1, 1, "f32", theta=True),
    # bf16 I/O (rotation runs on the generic path)
    wl.SSDConfig("rot_bf16", 1, 128, 2, 32, 32, 32, 1, 2, "bf16", theta=True),
]


def _run(inp, cfg, rope_dim, halves):
    d = {k: (v.cuda() if v is not None else None) for k, v in inp.items()}
    shape = pkg.shape_of(d["x"], d["B"], cfg.chunk_len, True)
    ws = torch.zeros(pkg.load_library().ssd_rotation_variant_workspace_bytes(
        __import__("ctypes").byref(shape), rope_dim, int(halves)), dtype=torch.uint8,
        device="cuda")
    y, fin = pkg.ssd_rotation_variant_forward(d["x"], d["dA"], d["B"], d["C"], d["theta"],
                                              chunk_len=cfg.chunk_len, rope_dim=rope_dim,
                                              halves=halves, init_state=d["init_state"],
                                              workspace=ws)
    assert pkg.workspace_status(ws) == ("SSD_OK", 0)
    torch.cuda.synchronize()
    return to_np(y), to_np(fin)


@pytest.mark.parametrize("cfg", CASES, ids=lambda c: c.name)
@pytest.mark.parametrize("rope_frac,halves", [(1, True), (2, False), (2, True), (4, True)])
def test_rotation_variant_parity(cfg, rope_frac, halves):
    rope_dim = cfg.dstate // rope_frac
    inp = wl.make_ssd_inputs(cfg, seed=31, slow_decay=True, init_state=True)
    g = torch.Generator().manual_seed(32)
    b, T, H = cfg.batch, cfg.seqlen, cfg.nheads
    inp["theta"] = torch.rand((b, T, H, rope_dim // 2), generator=g) * 0.2 - 0.1
    y, fin = _run(inp, cfg, rope_dim, halves)
    yr, fr = oracle.ssd_rotation_variant(to_np(inp["x"]), to_np(inp["dA"]), to_np(inp["B"]),
                                         to_np(inp["C"]), to_np(inp["theta"]),
                                         to_np(inp["init_state"]), rope_dim=rope_dim,
                                         halves=halves)
    tag = f"{cfg.name}/rope{rope_dim}/{'halves' if halves else 'pairs'}"
    check_close(y, yr, TOL[cfg.dtype], f"{tag} y")
    check_close(fin, fr, TOL[cfg.dtype], f"{tag} final_state")


def test_rotation_variant_rejections():
    cfg = CASES[0]
    d = wl.make_ssd_inputs(cfg, seed=33, device="cuda")
    with pytest.raises(pkg.SSDError):        # odd rope_dim
        pkg.ssd_rotation_variant_forward(d["x"], d["dA"], d["B"], d["C"],
                                         torch.zeros((2, 150, 4, 1), device="cuda"),
                                         chunk_len=64, rope_dim=3)

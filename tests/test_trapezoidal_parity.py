"""Trapezoidal Mamba-3 forward through the C ABI vs the fp64 oracle, element by element (GPU)."""
import numpy as np
import pytest
import torch

import chunked_ssd_scan_gb300 as pkg
from chunked_ssd_scan_gb300 import workloads as wl
from tests.parity_util import TOL, check_close, gpu_ssd, gpu_trap, oracle_trap

pytestmark = pytest.mark.gpu

T = dict(trapezoidal=True)
CASES = [
    wl.SSDConfig("trap_siso_f32", 2, 200, 3, 16, 16, 64, 1, 3, "f32", **T),
    wl.SSDConfig("trap_mimo_rot_f32", 1, 256, 4, 16, 32, 64, 2, 2, "f32", theta=True, **T),
    wl.SSDConfig("trap_rank4_groups_f32", 2, 96, 4, 8, 12, 32, 4, 1, "f32", **T),
    wl.SSDConfig("trap_ragged_rot_shared_f32", 1, 150, 6, 12, 8, 64, 1, 1, "f32", theta=True, **T),
    wl.SSDConfig("trap_bf16", 1, 256, 4, 64, 64, 64, 2, 2, "bf16", **T),
    wl.SSDConfig("trap_rot_bf16", 1, 190, 2, 32, 32, 64, 1, 1, "bf16", theta=True, **T),
    wl.TRAP_MIMO_ROT_F32.with_(seqlen=512),
    # bf16 without rotation at P = 64, N = 128: the fused tensor-core kernel with gamma and beta
    # as per-row write weights (ragged T; MIMO rank 4 with time segments and pre-pass pieces)
    wl.SSDConfig("trap_fused_bf16", 2, 300, 4, 64, 128, 64, 2, 2, "bf16", **T),
    wl.SSDConfig("trap_fused_mimo_bf16", 1, 1000, 4, 64, 128, 64, 4, 4, "bf16", **T),
]

FUSED = {"trap_fused_bf16", "trap_fused_mimo_bf16"}


@pytest.mark.parametrize("cfg", CASES, ids=lambda c: c.name)
@pytest.mark.parametrize("variant", ["stated", "slow_decay_init_prev", "no_prev"])
def test_trapezoidal_parity(cfg, variant):
    kw = dict(slow_decay=True, init_state=True) if variant == "slow_decay_init_prev" else {}
    inp = wl.make_trap_inputs(cfg, seed=21, prev=variant != "no_prev", **kw)
    x, B = inp["x"], inp["B"]
    shape = pkg.shape_of(x, B, cfg.chunk_len, inp["theta"] is not None)
    want = "tc_bf16" if cfg.name in FUSED else ("tc_tf32", "generic")
    got = pkg.ssd_trapezoidal_variant(shape)
    assert got == want if isinstance(want, str) else got in want, (cfg.name, got)
    y, fin = gpu_trap(inp, cfg.chunk_len)
    yr, fr = oracle_trap(inp)
    check_close(y, yr, TOL[cfg.dtype], f"{cfg.name}/{variant} y")
    check_close(fin, fr, TOL[cfg.dtype], f"{cfg.name}/{variant} final_state")


def test_trapezoidal_reduces_to_the_plain_scan():
    """gamma = 1, beta = 0: the trapezoidal call equals ssd_chunked_forward on the same data."""
    cfg = wl.SSDConfig("trap_plain", 1, 256, 4, 16, 32, 64, 2, 2, "f32", theta=True, **T)
    inp = wl.make_trap_inputs(cfg, seed=22, init_state=True)
    inp["gamma"] = torch.ones_like(inp["gamma"])
    inp["beta"] = torch.zeros_like(inp["beta"])
    y, fin = gpu_trap(inp, cfg.chunk_len)
    y2, f2 = gpu_ssd({k: inp[k] for k in ("x", "dA", "B", "C", "theta", "init_state")},
                     cfg.chunk_len)
    check_close(y, y2, 1e-5, "trapezoidal(beta=0) vs plain y")
    check_close(fin, f2, 1e-5, "trapezoidal(beta=0) vs plain final")


@pytest.mark.parametrize("split", [128, 77])
def test_trapezoidal_streaming(split):
    """A stream cut anywhere continues through final_state -> init_state with the last step's
    (x, B) as the next call's previous write."""
    cfg = wl.SSDConfig("trap_stream", 1, 300, 4, 16, 32, 64, 2, 2, "f32", theta=True, **T)
    inp = wl.make_trap_inputs(cfg, seed=23, init_state=True)
    yr, fr = oracle_trap(inp)
    cut = lambda v, lo, hi: v[:, lo:hi].contiguous()
    first = dict(inp)
    for k in ("x", "dA", "B", "C", "theta", "gamma", "beta"):
        first[k] = cut(inp[k], 0, split)
    y1, f1 = gpu_trap(first, cfg.chunk_len)
    second = dict(inp)
    for k in ("x", "dA", "B", "C", "theta", "gamma", "beta"):
        second[k] = cut(inp[k], split, cfg.seqlen)
    second["init_state"] = torch.from_numpy(f1).float()
    second["prev_x"] = inp["x"][:, split - 1].contiguous()
    second["prev_B"] = inp["B"][:, split - 1].contiguous()
    y2, f2 = gpu_trap(second, cfg.chunk_len)
    check_close(np.concatenate([y1, y2], axis=1), yr, TOL["f32"], "stream y")
    check_close(f2, fr, TOL["f32"], "stream final")


def test_trapezoidal_full_size_sampled_heads():
    """The measured trapezoidal shape at full length; the oracle recomputes two heads in full."""
    cfg = wl.TRAP_MIMO_ROT_F32
    inp = wl.make_trap_inputs(cfg, seed=0)
    y, fin = gpu_trap(inp, cfg.chunk_len)
    assert np.all(np.isfinite(y)) and np.all(np.isfinite(fin))
    for h in (0, 13):
        sub = {k: (None if v is None else v) for k, v in inp.items()}
        for k in ("x", "prev_x"):
            sub[k] = inp[k][..., h:h + 1, :].contiguous()
        for k in ("dA", "gamma", "beta"):
            sub[k] = inp[k][..., h:h + 1].contiguous()
        for k in ("B", "C", "prev_B"):          # one group per head in this shape
            sub[k] = inp[k][..., h:h + 1, :].contiguous()
        sub["theta"] = inp["theta"][:, :, h:h + 1].contiguous()
        yr, fr = oracle_trap(sub)
        check_close(y[..., h:h + 1, :], yr, TOL["f32"], f"full y[h={h}]")
        check_close(fin[:, h:h + 1], fr, TOL["f32"], f"full final[h={h}]")


def test_trapezoidal_host_rejections():
    cfg = wl.SSDConfig("trap_rej", 1, 64, 2, 8, 8, 64, 1, 1, "f32", **T)
    d = wl.make_trap_inputs(cfg, seed=24, device="cuda")
    with pytest.raises(ValueError):     # prev_x without prev_B
        pkg.ssd_trapezoidal_forward(d["x"], d["dA"], d["B"], d["C"], d["gamma"], d["beta"],
                                    chunk_len=64, prev_x=d["prev_x"])
    with pytest.raises(pkg.SSDError) as e:   # 2R-channel chunk beyond the pipeline's limit
        pkg.ssd_trapezoidal_forward(d["x"], d["dA"], d["B"], d["C"], d["gamma"], d["beta"],
                                    chunk_len=4096)
    assert e.value.status == 2

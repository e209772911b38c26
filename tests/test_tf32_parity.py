"""ssd_chunked_forward_tf32 (fp32 I/O, P = N = 64: the chunk scan as tcgen05 kind::tf32 products
with split operands) against the fp64 oracle at the fp32 gate |got - ref| <= 1e-4 (1 + |ref|),
element by element, through the C ABI.

The slow-decay cases with an initial state are the hard ones: the state grows large, y is a sum
of terms much larger than itself, and the tensor core's truncating accumulation acts on those
terms.  Chunks of 128 fused rows span several chunks, ragged tails, MIMO ranks, groups and the
rotation (scan.py page: B and C turned by the cumulative angle)."""
import ctypes

import numpy as np
import pytest

import chunked_ssd_scan_gb300 as pkg
from chunked_ssd_scan_gb300 import workloads as wl
from tests.parity_util import TOL, check_close, gpu_ssd, oracle_ssd, slice_heads

CASES = [
    wl.SSDConfig("tf32_l64_g2", 2, 512, 4, 64, 64, 64, 1, 2, "f32"),
    wl.SSDConfig("tf32_l384_theta_shared", 1, 768, 3, 64, 64, 384, 1, 1, "f32", theta=True),
    wl.SSDConfig("tf32_mimo_r2_theta_ragged", 1, 200, 2, 64, 64, 64, 2, 1, "f32", theta=True),
    wl.SSDConfig("tf32_mimo_r4_groups", 2, 96, 4, 64, 64, 128, 4, 2, "f32"),
    wl.SSDConfig("tf32_ragged", 1, 200, 2, 64, 64, 64, 1, 1, "f32"),
    wl.SSDConfig("tf32_ragged_theta", 2, 130, 3, 64, 64, 128, 1, 1, "f32", theta=True),
    wl.SSDConfig("tf32_one_step", 1, 1, 2, 64, 64, 64, 1, 1, "f32", theta=True),
    wl.LONG_ROT_F32.with_(seqlen=2048),
    # chunk_len 1000 sends ssd_chunked_forward to the generic path with long chunks; the common
    # workspace size must still hold the tf32 entry's 128-row chunk states
    wl.SSDConfig("tf32_chunk1000", 1, 2000, 2, 64, 64, 1000, 1, 1, "f32", theta=True),
]


@pytest.mark.gpu
@pytest.mark.parametrize("cfg", CASES, ids=lambda c: c.name)
@pytest.mark.parametrize("variant", ["stated", "slow_decay_init"])
def test_tf32_scan_matches_oracle(cfg, variant):
    kw = dict(slow_decay=True, init_state=True) if variant == "slow_decay_init" else {}
    inp = wl.make_ssd_inputs(cfg, seed=3, **kw)
    y, fin = gpu_ssd(inp, cfg.chunk_len, guard=True, tf32=True)
    yr, fr = oracle_ssd(inp)
    check_close(y, yr, TOL["f32"], f"{cfg.name}/{variant} y")
    check_close(fin, fr, TOL["f32"], f"{cfg.name}/{variant} final_state")


@pytest.mark.gpu
def test_tf32_scan_full_size_sampled_heads():
    """The long-rotation workload at full size through the tf32 entry; sampled (batch, head)
    problems recomputed by the oracle in full."""
    cfg = wl.LONG_ROT_F32
    inp = wl.make_ssd_inputs(cfg, seed=0)
    y, fin = gpu_ssd(inp, cfg.chunk_len, tf32=True)
    assert np.all(np.isfinite(y)) and np.all(np.isfinite(fin))
    for (b, h) in [(0, 0), (0, 13)]:
        sub = slice_heads(inp, cfg, b, h)
        yr, fr = oracle_ssd(sub)
        check_close(y[b:b + 1, :, :, h:h + 1], yr, TOL["f32"], f"y[b={b},h={h}]")
        check_close(fin[b:b + 1, h:h + 1], fr, TOL["f32"], f"final[b={b},h={h}]")


@pytest.mark.gpu
def test_tf32_scan_valid_lengths():
    """Per-sequence valid lengths through the tf32 entry (moments.rs page pad semantics): inputs
    at pad steps are NaN and must not reach any output; each sequence matches the oracle on the
    sequence cut at its length."""
    cfg = wl.SSDConfig("tf32_vl", 3, 600, 4, 64, 64, 256, 1, 2, "f32", theta=True)
    lens = [600, 301, 128]
    inp = wl.make_ssd_inputs(cfg, seed=11, slow_decay=True, init_state=True)
    for b, n in enumerate(lens):
        for k in ("x", "dA", "B", "C", "theta"):
            inp[k][b, n:] = float("nan")
    y, fin = gpu_ssd(inp, cfg.chunk_len, tf32=True, valid_len=lens)
    for b, n in enumerate(lens):
        sub = {k: (v[b:b + 1, :n].contiguous() if k != "init_state" else v[b:b + 1])
               for k, v in inp.items() if v is not None}
        yr, fr = oracle_ssd(sub)
        check_close(y[b:b + 1, :n], yr, TOL["f32"], f"y[b={b}, :{n}]")
        check_close(fin[b:b + 1], fr, TOL["f32"], f"final[b={b}]")


def test_tf32_entry_rejects_other_shapes_on_the_host():
    """bf16 I/O, P or N other than 64 and ranks that do not divide 128 are UNSUPPORTED before any
    pointer is touched (null pointers here)."""
    lib = pkg.load_library()
    for args in ((1, 256, 2, 64, 64, 1, 64, "bf16"), (1, 256, 2, 32, 64, 1, 64, "f32"),
                 (1, 256, 2, 64, 32, 1, 64, "f32"), (1, 256, 2, 64, 64, 3, 64, "f32")):
        b, T, H, P, N, R, l, dt = args
        shape = pkg.make_shape(b, T, H, P, N, 1, R, l, dt, False)
        st = lib.ssd_chunked_forward_tf32(ctypes.byref(shape), *([None] * 10),
                                          ctypes.c_size_t(0), None)
        assert pkg.STATUS.get(st) == "SSD_ERR_UNSUPPORTED", (args, st)

"""CUDA SSD path vs the fp64 oracle, element by element, through the C ABI (GPU)."""
import numpy as np
import pytest
import torch

import chunked_ssd_scan_gb300 as pkg
from chunked_ssd_scan_gb300 import workloads as wl
from tests.parity_util import TOL, check_close, gpu_ssd, oracle_ssd, slice_heads

pytestmark = pytest.mark.gpu

# Reduced-T versions of the four SSD workloads: several chunks and tiles, oracle in seconds.
REDUCED = [
    wl.TINY_SISO_F32,
    wl.MAMBA2_SISO_BF16.with_(batch=2, seqlen=1024),
    wl.MAMBA3_MIMO_BF16.with_(batch=1, seqlen=512),
    wl.LONG_ROT_F32.with_(seqlen=2048),
]


@pytest.mark.parametrize("cfg", REDUCED, ids=lambda c: c.name)
@pytest.mark.parametrize("variant", ["stated", "slow_decay_init", "seed1", "seed2"])
def test_reduced_workloads(cfg, variant):
    kw = dict(slow_decay=True, init_state=True) if variant == "slow_decay_init" else {}
    seed = {"seed1": 1, "seed2": 2}.get(variant, 0)
    inp = wl.make_ssd_inputs(cfg, seed=seed, **kw)
    y, fin = gpu_ssd(inp, cfg.chunk_len)
    yr, fr = oracle_ssd(inp)
    check_close(y, yr, TOL[cfg.dtype], f"{cfg.name}/{variant} y")
    check_close(fin, fr, TOL[cfg.dtype], f"{cfg.name}/{variant} final_state")


FULL = [wl.MAMBA2_SISO_BF16, wl.MAMBA3_MIMO_BF16, wl.LONG_ROT_F32]
SAMPLES = {"mamba2_siso_bf16": [(0, 0), (3, 31), (2, 17)],
           "mamba3_mimo_bf16": [(0, 5), (1, 30)],
           "long_rotation_f32": [(0, 0), (0, 23)]}


@pytest.mark.parametrize("cfg", FULL, ids=lambda c: c.name)
def test_full_size_sampled_heads(cfg):
    """Full workload sizes in the benchmark's launch configuration; the oracle recomputes a few
    independent (batch, head) problems in full and compares every one of their outputs."""
    inp = wl.make_ssd_inputs(cfg, seed=0)
    y, fin = gpu_ssd(inp, cfg.chunk_len)
    assert np.all(np.isfinite(y)) and np.all(np.isfinite(fin))
    for (b, h) in SAMPLES[cfg.name]:
        sub = slice_heads(inp, cfg, b, h)
        yr, fr = oracle_ssd(sub)
        check_close(y[b:b + 1, :, :, h:h + 1], yr, TOL[cfg.dtype], f"{cfg.name} y[b={b},h={h}]")
        check_close(fin[b:b + 1, h:h + 1], fr, TOL[cfg.dtype], f"{cfg.name} final[b={b},h={h}]")


def test_full_size_slow_decay_carries_state_across_all_tiles():
    """The Mamba-2-shape workload at full size with slow decay and an initial state, in the one-
    launch configuration the benchmark times (128 sequences on one SM each: every sequence's
    state crosses all 32 tiles on chip).  Under the stated decay the carry between tiles is
    ~e^-127 and invisible; here it dominates y.  Sampled (batch, head) problems, every output."""
    cfg = wl.MAMBA2_SISO_BF16
    shape = pkg.make_shape(cfg.batch, cfg.seqlen, cfg.nheads, cfg.headdim, cfg.dstate, cfg.ngroups,
                           cfg.mimo_rank, cfg.chunk_len, cfg.dtype, cfg.theta)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    if cfg.batch * cfg.nheads * 2 > sms:   # the bench's configuration on this GPU: no segments
        assert pkg.ssd_chunked_launches(shape) == 1
    inp = wl.make_ssd_inputs(cfg, seed=0, slow_decay=True, init_state=True)
    y, fin = gpu_ssd(inp, cfg.chunk_len)
    for (b, h) in [(0, 0), (1, 9), (2, 22), (3, 31)]:
        sub = slice_heads(inp, cfg, b, h)
        yr, fr = oracle_ssd(sub)
        check_close(y[b:b + 1, :, :, h:h + 1], yr, TOL[cfg.dtype], f"slow decay y[b={b},h={h}]")
        check_close(fin[b:b + 1, h:h + 1], fr, TOL[cfg.dtype], f"slow decay final[b={b},h={h}]")


EDGE = [
    # single chunk, one head, tiny dims
    wl.SSDConfig("one_chunk_f32", 1, 64, 1, 8, 8, 64, 1, 1, "f32"),
    wl.SSDConfig("one_chunk_bf16", 1, 256, 2, 64, 128, 256, 1, 1, "bf16"),
    # chunk_len 1 (every step is a chunk) and T == 1
    wl.SSDConfig("chunk1_f32", 1, 24, 2, 4, 6, 1, 1, 2, "f32"),
    wl.SSDConfig("T1_f32", 2, 1, 3, 5, 4, 1, 2, 3, "f32", theta=True),
    # odd head/state sizes, groups, MIMO with ragged fused tiles (L = 3*40 = 120)
    wl.SSDConfig("odd_dims_f32", 2, 120, 6, 5, 6, 40, 3, 2, "f32", theta=True),
    wl.SSDConfig("odd_dims_bf16", 1, 96, 4, 24, 40, 32, 2, 2, "bf16"),
    # shared B/C across all heads with rotation (per-head rotation of shared B/C)
    wl.SSDConfig("shared_bc_theta_f32", 1, 512, 8, 16, 32, 128, 1, 1, "f32", theta=True),
    # largest tile shapes of the bf16 path with several chunks
    wl.SSDConfig("p128_n128_bf16", 1, 512, 2, 128, 128, 128, 1, 2, "bf16"),
    # fused tensor-core path: one tile; rank 2 with 2 groups; rank 8 (16 steps per tile)
    wl.SSDConfig("fused_one_tile", 1, 128, 4, 64, 128, 128, 1, 1, "bf16"),
    wl.SSDConfig("fused_r2_g2", 2, 320, 8, 64, 128, 64, 2, 2, "bf16"),
    wl.SSDConfig("fused_r8_g4", 1, 256, 4, 64, 128, 16, 8, 4, "bf16"),
    # fused kernel with time segments of unequal length (9 tiles on 8 sequences: 5 + 4)
    wl.SSDConfig("fused_uneven_segments", 1, 1152, 8, 64, 128, 128, 1, 1, "bf16"),
    # fp32 path with the tf32 tensor-core chunk scan (128 fused rows per chunk whatever
    # chunk_len says): four chunks without rotation, two groups; six chunks with rotation and
    # one group shared by three heads
    wl.SSDConfig("tc32_f32_l64_g2", 2, 512, 4, 64, 64, 64, 1, 2, "f32"),
    wl.SSDConfig("tc32_f32_l384_theta_shared", 1, 768, 3, 64, 64, 384, 1, 1, "f32", theta=True),
    # the same with MIMO rank-fused rows (128 / R steps per chunk): rank 2 with rotation and a
    # ragged tail; rank 4 with two groups
    wl.SSDConfig("tc32_f32_mimo_r2_theta", 1, 200, 2, 64, 64, 64, 2, 1, "f32", theta=True),
    wl.SSDConfig("tc32_f32_mimo_r4_groups", 2, 96, 4, 64, 64, 128, 4, 2, "f32"),
]


# seqlen not a multiple of chunk_len (and, for the fused kernel, of the 128-row tile): the last
# chunk or tile is short and runs as zero padding; every path, with groups, MIMO, rotation and
# time segments.
RAGGED = [
    wl.SSDConfig("ragged_generic_f32", 2, 250, 3, 16, 16, 64, 1, 3, "f32"),
    wl.SSDConfig("ragged_generic_mimo_theta_f32", 2, 77, 2, 8, 12, 16, 3, 2, "f32", theta=True),
    wl.SSDConfig("ragged_generic_bf16", 1, 100, 4, 24, 40, 32, 2, 2, "bf16"),
    wl.SSDConfig("ragged_fused_bf16", 2, 300, 4, 64, 128, 256, 1, 1, "bf16"),
    wl.SSDConfig("ragged_fused_mimo_bf16", 1, 90, 4, 64, 128, 32, 4, 2, "bf16"),
    wl.SSDConfig("ragged_fused_segments_bf16", 1, 1000, 8, 64, 128, 128, 1, 1, "bf16"),
    wl.SSDConfig("ragged_tc32_f32", 1, 200, 2, 64, 64, 64, 1, 1, "f32"),
    wl.SSDConfig("ragged_tc32_theta_f32", 2, 130, 3, 64, 64, 128, 1, 1, "f32", theta=True),
]


@pytest.mark.parametrize("cfg", RAGGED, ids=lambda c: c.name)
def test_ragged_sequence_lengths(cfg):
    assert cfg.seqlen % cfg.chunk_len != 0
    expect = {"generic": "generic", "fused": "tc_bf16", "tc32": "tc_tf32"}[cfg.name.split("_")[1]]
    shape = pkg.make_shape(cfg.batch, cfg.seqlen, cfg.nheads, cfg.headdim, cfg.dstate,
                           cfg.ngroups, cfg.mimo_rank, cfg.chunk_len, cfg.dtype, cfg.theta)
    assert pkg.ssd_chunked_variant(shape) == expect, cfg.name
    for kw in ({}, dict(slow_decay=True, init_state=True)):
        inp = wl.make_ssd_inputs(cfg, seed=8, **kw)
        y, fin = gpu_ssd(inp, cfg.chunk_len, guard=True)
        yr, fr = oracle_ssd(inp)
        check_close(y, yr, TOL[cfg.dtype], f"{cfg.name} y")
        check_close(fin, fr, TOL[cfg.dtype], f"{cfg.name} final_state")


@pytest.mark.parametrize("cfg", [wl.SSDConfig("vlen_fused", 3, 512, 4, 64, 128, 128, 1, 1, "bf16"),
                                 wl.SSDConfig("vlen_generic", 3, 200, 2, 16, 16, 64, 2, 2, "f32")],
                         ids=lambda c: c.name)
def test_per_sequence_valid_length_by_zero_padding(cfg):
    """Sequences of different lengths in one batch: steps past a sequence's valid length carry
    dA = 0 and x = 0 (the moments.rs page's pad semantics), so its final state is the state at
    its last real step and its y on real steps is that of the truncated sequence."""
    inp = wl.make_ssd_inputs(cfg, seed=10, init_state=True)
    lens = [cfg.seqlen, cfg.seqlen - 77, 1]
    for b, n in enumerate(lens):
        inp["x"][b, n:] = 0
        inp["dA"][b, n:] = 0
    y, fin = gpu_ssd(inp, cfg.chunk_len)
    for b, n in enumerate(lens):
        sub = {k: (v[b:b + 1, :n].contiguous() if k != "init_state" else v[b:b + 1])
               for k, v in inp.items() if v is not None}
        sub.setdefault("theta", None)
        yr, fr = oracle_ssd(sub)
        check_close(y[b:b + 1, :n], yr, TOL[cfg.dtype], f"{cfg.name} y[b={b}, :{n}]")
        check_close(fin[b:b + 1], fr, TOL[cfg.dtype], f"{cfg.name} final[b={b}]")


def test_f32_workloads_use_the_tf32_tensor_core_scan():
    for cfg in (wl.LONG_ROT_F32, EDGE[-1], EDGE[-2], EDGE[-3], EDGE[-4]):
        shape = pkg.make_shape(cfg.batch, cfg.seqlen, cfg.nheads, cfg.headdim, cfg.dstate,
                               cfg.ngroups, cfg.mimo_rank, cfg.chunk_len, cfg.dtype, cfg.theta)
        assert pkg.ssd_chunked_variant(shape) == "tc_tf32", cfg.name


def test_fused_launches_follow_the_segmentation():
    """Fewer sequences than SMs: pre-pass + carry + full pass; otherwise one launch."""
    def launches(cfg):
        return pkg.ssd_chunked_launches(pkg.make_shape(
            cfg.batch, cfg.seqlen, cfg.nheads, cfg.headdim, cfg.dstate, cfg.ngroups,
            cfg.mimo_rank, cfg.chunk_len, cfg.dtype, cfg.theta))
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert launches(wl.MAMBA3_MIMO_BF16) == (3 if 64 * 2 <= sms else 1)
    assert launches(wl.MAMBA2_SISO_BF16) == (3 if 128 * 2 <= sms else 1)


def test_bf16_workloads_use_the_fused_kernel():
    for cfg in (wl.MAMBA2_SISO_BF16, wl.MAMBA3_MIMO_BF16, EDGE[-5], EDGE[-6], EDGE[-7], EDGE[-8]):
        shape = pkg.make_shape(cfg.batch, cfg.seqlen, cfg.nheads, cfg.headdim, cfg.dstate,
                               cfg.ngroups, cfg.mimo_rank, cfg.chunk_len, cfg.dtype, cfg.theta)
        assert pkg.ssd_chunked_variant(shape) == "tc_bf16", cfg.name


@pytest.mark.parametrize("cfg", EDGE, ids=lambda c: c.name)
def test_edge_shapes(cfg):
    inp = wl.make_ssd_inputs(cfg, seed=3, slow_decay=True, init_state=True)
    y, fin = gpu_ssd(inp, cfg.chunk_len, guard=True)
    yr, fr = oracle_ssd(inp)
    check_close(y, yr, TOL[cfg.dtype], f"{cfg.name} y")
    check_close(fin, fr, TOL[cfg.dtype], f"{cfg.name} final_state")


def test_final_state_optional_and_y_unchanged():
    cfg = wl.TINY_SISO_F32
    inp = wl.make_ssd_inputs(cfg, seed=4, init_state=True)
    y1, _ = gpu_ssd(inp, cfg.chunk_len, final=False)
    y2, _ = gpu_ssd(inp, cfg.chunk_len, final=True)
    assert np.array_equal(y1, y2)


def test_chunk_length_invariance_on_gpu():
    """The result does not depend on chunk_len (the serial.rs page's decomposition is exact)."""
    cfg = wl.SSDConfig("inv", 1, 512, 4, 16, 32, 64, 1, 2, "f32", theta=True)
    inp = wl.make_ssd_inputs(cfg, seed=5, slow_decay=True, init_state=True)
    yr, fr = oracle_ssd(inp)
    for l in (16, 64, 128, 256, 512):
        y, fin = gpu_ssd(inp, l)
        check_close(y, yr, TOL["f32"], f"chunk_len {l} y")
        check_close(fin, fr, TOL["f32"], f"chunk_len {l} final")


def test_continuation_through_final_state():
    cfg = wl.SSDConfig("cont", 1, 512, 4, 16, 32, 64, 2, 2, "f32")
    inp = wl.make_ssd_inputs(cfg, seed=6, slow_decay=True, init_state=True)
    yf, ff = gpu_ssd(inp, 64)
    first = {k: (v[:, :256].contiguous() if (v is not None and k != "init_state") else v)
             for k, v in inp.items()}
    y1, f1 = gpu_ssd(first, 64)
    second = {k: (v[:, 256:].contiguous() if (v is not None and k != "init_state") else v)
              for k, v in inp.items()}
    second["init_state"] = torch.from_numpy(f1).float()
    y2, f2 = gpu_ssd(second, 64)
    check_close(np.concatenate([y1, y2], axis=1), yf, 1e-5, "continuation y")
    check_close(f2, ff, 1e-5, "continuation final")


@pytest.mark.parametrize("split", [200, 77])
def test_streaming_continuation_ragged_with_rotation(split):
    """A stream cut at arbitrary steps (short last chunks on both sides) continues exactly through
    final_state -> init_state; with rotation no angle carry is needed because the state crosses
    the boundary in the physical frame."""
    cfg = wl.SSDConfig("stream", 1, 512, 4, 16, 32, 64, 1, 2, "f32", theta=True)
    inp = wl.make_ssd_inputs(cfg, seed=9, slow_decay=True, init_state=True)
    yf, _ = gpu_ssd(inp, 64)
    first = {k: (v[:, :split].contiguous() if (v is not None and k != "init_state") else v)
             for k, v in inp.items()}
    y1, f1 = gpu_ssd(first, 64)
    second = {k: (v[:, split:].contiguous() if (v is not None and k != "init_state") else v)
              for k, v in inp.items()}
    second["init_state"] = torch.from_numpy(f1).float()
    y2, f2 = gpu_ssd(second, 64)
    # the two halves accumulate their angles from different origins, so they match the unsplit
    # call to the fp32 bound, not bitwise: both are checked against the oracle of the whole
    yr, fr = oracle_ssd(inp)
    check_close(np.concatenate([y1, y2], axis=1), yr, TOL["f32"], "stream y")
    check_close(f2, fr, TOL["f32"], "stream final")
    check_close(yf, yr, TOL["f32"], "unsplit y")


def test_deterministic_bitwise():
    cfg = wl.MAMBA2_SISO_BF16.with_(batch=1, seqlen=1024, nheads=8)
    inp = wl.make_ssd_inputs(cfg, seed=7, init_state=True)
    a = gpu_ssd(inp, cfg.chunk_len)
    b = gpu_ssd(inp, cfg.chunk_len)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_host_rejections_with_real_buffers():
    cfg = wl.TINY_SISO_F32
    d = wl.make_ssd_inputs(cfg, seed=0, device="cuda")
    with pytest.raises(pkg.SSDError) as e:   # fused chunk beyond the generic path's limit
        pkg.ssd_chunked_forward(d["x"], d["dA"], d["B"], d["C"], chunk_len=8192)
    assert e.value.status == 2
    with pytest.raises(ValueError):
        pkg.ssd_chunked_forward(d["x"].cpu(), d["dA"], d["B"], d["C"], chunk_len=64)

"""bench.py's workload plumbing on CPU: every named workload resolves, its algorithmic bytes and
FLOPs are positive, the FLOP count of the fp32 tensor-core path uses the 128-row chunks the
kernels tile by, and the backward's bytes grow with the gradients it writes (no GPU involved)."""
import pytest

import bench
import chunked_ssd_scan_gb300 as pkg
from chunked_ssd_scan_gb300 import workloads as wl

NAMES = [c.name for c in wl.SSD_CONFIGS] + [
    wl.SELECTIVE_SCAN_F32.name, wl.TRAP_MIMO_ROT_F32.name, wl.ROT_VARIANT_F32.name,
    wl.MAMBA2_BWD_BF16.name, wl.LONG_ROT_BWD_F32.name, wl.TRAP_BWD_F32.name]


@pytest.mark.parametrize("name", NAMES)
def test_every_workload_resolves(name):
    cfg = bench.workload(name)
    assert cfg.name == name
    assert cfg.io_bytes() > 0
    small = bench.workload(name, batch=1, seqlen=256)
    assert small.batch == 1 and small.seqlen == 256


def test_unknown_workload_is_rejected():
    with pytest.raises(SystemExit):
        bench.workload("no_such_workload")


def test_metric_names():
    assert "backward" in bench.metric_name(wl.MAMBA2_BWD_BF16, False)
    assert bench.metric_name(wl.SELECTIVE_SCAN_F32, True).startswith("selective scan")
    assert bench.metric_name(wl.MAMBA2_SISO_BF16, False) == bench.METRIC


def test_fp32_flops_counted_at_the_kernel_chunk():
    cfg = wl.LONG_ROT_F32
    shape = pkg.make_shape(cfg.batch, cfg.seqlen, cfg.nheads, cfg.headdim, cfg.dstate,
                           cfg.ngroups, cfg.mimo_rank, cfg.chunk_len, "f32", cfg.theta)
    assert pkg.ssd_chunked_variant(shape) == "tc_tf32"
    assert bench.kernel_chunk(pkg, shape, 1, cfg.chunk_len) == 128
    bf = wl.MAMBA2_SISO_BF16
    bshape = pkg.make_shape(bf.batch, bf.seqlen, bf.nheads, bf.headdim, bf.dstate, bf.ngroups,
                            bf.mimo_rank, bf.chunk_len, "bf16", False)
    assert bench.kernel_chunk(pkg, bshape, 1, bf.chunk_len) == bf.chunk_len
    # shorter chunks do less quadratic work
    assert cfg.with_(chunk_len=64).causal_flops() < cfg.causal_flops()


def test_backward_counts():
    plain, rot, trap = wl.MAMBA2_BWD_BF16, wl.LONG_ROT_BWD_F32, wl.TRAP_BWD_F32
    assert plain.backward_flops() > 0 and rot.backward_flops() > 0
    # the backward reads the forward's inputs and dy and writes one gradient per input
    fwd = plain.with_(backward=False)
    assert plain.io_bytes() > fwd.io_bytes()
    # theta adds its read and dtheta's write; the trapezoid adds gamma, beta and the previous write
    assert rot.io_bytes() > rot.with_(theta=False).io_bytes()
    assert trap.io_bytes() > trap.with_(trapezoidal=False).io_bytes()

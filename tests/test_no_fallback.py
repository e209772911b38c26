"""The product path has no CPU fallback: every public entry point refuses host tensors, and a
missing library raises instead of computing anything (no GPU involved)."""
import pytest
import torch

import chunked_ssd_scan_gb300 as pkg
from chunked_ssd_scan_gb300 import workloads as wl

cpu_only = pytest.mark.skipif(torch.cuda.is_available(), reason="checks host tensors on CPU hosts")


def _ssd_inputs(theta=False):
    cfg = wl.SSDConfig("nf", 1, 64, 2, 16, 16, 64, 1, 1, "f32", theta=theta)
    return cfg, wl.make_ssd_inputs(cfg, seed=0, init_state=True)


@cpu_only
def test_forward_refuses_host_tensors():
    cfg, d = _ssd_inputs(theta=True)
    with pytest.raises(ValueError, match="CUDA tensor"):
        pkg.ssd_chunked_forward(d["x"], d["dA"], d["B"], d["C"], chunk_len=cfg.chunk_len,
                                theta=d["theta"], init_state=d["init_state"])
    with pytest.raises(ValueError, match="CUDA tensor"):
        pkg.ssd_rotation_variant_forward(d["x"], d["dA"], d["B"], d["C"], d["theta"],
                                         chunk_len=cfg.chunk_len)


@cpu_only
def test_trapezoidal_refuses_host_tensors():
    cfg = wl.SSDConfig("nf_trap", 1, 64, 2, 16, 16, 64, 1, 1, "f32", trapezoidal=True)
    d = wl.make_trap_bwd_inputs(cfg, seed=0)
    with pytest.raises(ValueError, match="CUDA tensor"):
        pkg.ssd_trapezoidal_forward(d["x"], d["dA"], d["B"], d["C"], d["gamma"], d["beta"],
                                    chunk_len=cfg.chunk_len)
    with pytest.raises(ValueError, match="CUDA tensor"):
        pkg.ssd_trapezoidal_backward(d["x"], d["dA"], d["B"], d["C"], d["gamma"], d["beta"],
                                     d["dy"])


@cpu_only
def test_backward_refuses_host_tensors():
    cfg = wl.SSDConfig("nf_bwd", 1, 64, 2, 16, 16, 64, 1, 1, "f32")
    d = wl.make_bwd_inputs(cfg, seed=0)
    with pytest.raises(ValueError, match="CUDA tensor"):
        pkg.ssd_chunked_backward(d["x"], d["dA"], d["B"], d["C"], d["dy"])


@cpu_only
def test_selective_scan_refuses_host_tensors():
    s = wl.make_selective_scan_inputs(wl.SelectiveScanConfig("nf_ss", 1, 32, 8, 16), seed=0)
    with pytest.raises(ValueError, match="CUDA tensor"):
        pkg.selective_scan_forward(s["u"], s["delta"], s["A"], s["B"], s["C"], s["skip"])


def test_missing_library_raises(tmp_path):
    with pytest.raises(RuntimeError, match="not found"):
        pkg.load_library(str(tmp_path / "libssdscan.so"))

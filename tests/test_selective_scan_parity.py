"""CUDA selective scan vs the fp64 oracle through the C ABI (GPU)."""
import numpy as np
import pytest
import torch

import chunked_ssd_scan_gb300 as pkg
import oracle
from chunked_ssd_scan_gb300 import workloads as wl
from tests.parity_util import check_close, to_np

pytestmark = pytest.mark.gpu

TOL = 1e-4


def run(cfg, seed=0, skip=True):
    s = wl.make_selective_scan_inputs(cfg, seed=seed)
    if not skip:
        s["skip"] = None
    d = {k: (v.cuda() if v is not None else None) for k, v in s.items()}
    y = pkg.selective_scan_forward(d["u"], d["delta"], d["A"], d["B"], d["C"], d["skip"])
    torch.cuda.synchronize()
    ref = oracle.selective_scan(to_np(s["u"]), to_np(s["delta"]), to_np(s["A"]), to_np(s["B"]),
                                to_np(s["C"]), to_np(s["skip"]))
    return to_np(y), ref


def test_full_workload():
    """The full selective-scan workload (batch 4, T 4096, d_model 512, d_state 16), every output."""
    y, ref = run(wl.SELECTIVE_SCAN_F32)
    check_close(y, ref, TOL, "selective scan y")


@pytest.mark.parametrize("cfg", [
    wl.SelectiveScanConfig("T1", 2, 1, 33, 16),
    wl.SelectiveScanConfig("ragged_T", 1, 1000, 130, 16),
    wl.SelectiveScanConfig("N1", 1, 300, 64, 1),
    wl.SelectiveScanConfig("N64", 2, 257, 96, 64),
    wl.SelectiveScanConfig("N32_ragged_D", 1, 333, 50, 32),
    wl.SelectiveScanConfig("N8_ragged_D", 2, 77, 13, 8),
    # one-pass staged kernel (d_model % 4 == 0): ragged channel blocks and ragged stages
    wl.SelectiveScanConfig("onepass_N16_D20", 2, 1000, 20, 16),
    wl.SelectiveScanConfig("onepass_N8_D36", 1, 130, 36, 8),
    wl.SelectiveScanConfig("onepass_N32_D12", 1, 65, 12, 32),
    wl.SelectiveScanConfig("onepass_N64_D8", 1, 200, 8, 64),
    wl.SelectiveScanConfig("onepass_T1", 3, 1, 4, 16),
    wl.SelectiveScanConfig("N17", 1, 129, 40, 17),
    wl.SelectiveScanConfig("D1", 3, 70, 1, 8),
], ids=lambda c: c.name)
def test_edge_sizes(cfg):
    y, ref = run(cfg, seed=1)
    check_close(y, ref, TOL, f"{cfg.name} y")


def test_without_skip():
    y, ref = run(wl.SelectiveScanConfig("noskip", 2, 500, 64, 16), seed=2, skip=False)
    check_close(y, ref, TOL, "no-skip y")


def test_worked_example_on_gpu():
    """The SSM Selective Scan page's worked example through the CUDA path."""
    from tests.pins import load_golden
    g = load_golden("selective_scan_worked_example.txt")
    dev = "cuda"
    t = lambda k, shp: torch.tensor(g[k], dtype=torch.float32, device=dev).reshape(shp)
    y = pkg.selective_scan_forward(t("u", (1, 4, 2)), t("delta", (1, 4, 2)), t("A", (2, 2)),
                                   t("B", (1, 4, 2)), t("C", (1, 4, 2)), t("skip", (2,)))
    np.testing.assert_allclose(y.cpu().numpy().reshape(-1), g["y"], atol=g["tolerance"][0] + 1e-6)


def test_exponent_range_of_the_decay():
    """Decay factors exp(delta A) from about e^-120 (underflowing to zero) up to nearly 1
    (A from -20 to -0.5, delta doubled): every exponential over that range, on a problem whose
    memory stays short enough for the fp32 recurrence to meet the gate."""
    cfg = wl.SelectiveScanConfig("exp_range", 2, 700, 64, 16)
    s = wl.make_selective_scan_inputs(cfg, seed=5)
    g = torch.Generator().manual_seed(5)
    s["A"] = -(torch.rand((cfg.d_model, cfg.d_state), generator=g) * 19.5 + 0.5)
    s["delta"] = s["delta"] * 2.0
    d = {k: v.cuda() for k, v in s.items()}
    y = pkg.selective_scan_forward(d["u"], d["delta"], d["A"], d["B"], d["C"], d["skip"])
    torch.cuda.synchronize()
    ref = oracle.selective_scan(*(to_np(s[k]) for k in ("u", "delta", "A", "B", "C", "skip")))
    check_close(to_np(y), ref, TOL, "exponent-range y")

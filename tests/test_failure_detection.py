"""Failure detection without a GPU fault: a bounded device wait that nothing satisfies gives up,
latches SSD_ERR_TIMEOUT in the workspace header, and the context stays usable (GPU)."""
import numpy as np
import pytest
import torch

import chunked_ssd_scan_gb300 as pkg
from chunked_ssd_scan_gb300 import workloads as wl
from tests.parity_util import TOL, check_close, gpu_ssd, oracle_ssd

pytestmark = pytest.mark.gpu


def test_wait_gives_up_latches_timeout_and_context_survives():
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    assert pkg.workspace_status(ws) == ("SSD_OK", 0)
    pkg.wait_selftest(ws, 2_000_000)                 # 2 ms bound on a barrier nobody arrives on
    assert pkg.workspace_status(ws) == ("SSD_ERR_TIMEOUT", 900)
    assert pkg.workspace_status(ws) == ("SSD_OK", 0)  # reading clears the latch
    # the same context still runs the forward correctly afterwards
    cfg = wl.SSDConfig("after_timeout", 1, 256, 4, 64, 128, 128, 1, 1, "bf16")
    inp = wl.make_ssd_inputs(cfg, seed=11)
    y, fin = gpu_ssd(inp, cfg.chunk_len)
    yr, fr = oracle_ssd(inp)
    check_close(y, yr, TOL["bf16"], "y after timeout")
    check_close(fin, fr, TOL["bf16"], "final after timeout")


def test_forward_leaves_a_clean_workspace_clean():
    cfg = wl.MAMBA2_SISO_BF16.with_(batch=1, seqlen=512, nheads=4)
    d = wl.make_ssd_inputs(cfg, seed=12, device="cuda")
    plan = pkg.SSDForwardPlan(d["x"], d["dA"], d["B"], d["C"], chunk_len=cfg.chunk_len)
    plan()
    assert pkg.workspace_status(plan.workspace) == ("SSD_OK", 0)
    assert np.all(np.isfinite(plan.y.float().cpu().numpy()))

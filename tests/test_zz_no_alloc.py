"""Allocation-free selective scan entry point (GPU).

``selective_scan_forward_noalloc`` serves callers that cannot allocate device memory (for example
code that receives only its input and output buffers through a fixed plugin interface): instead
of a caller workspace it uses one fixed scratch array inside the library.  Called through the C
ABI, it must agree with ``selective_scan_forward`` (the workspace entry point) and with the fp64
oracle, on calls in a row with different inputs.  The second call repeats the first call's sizes
with other seeds, so the whole scratch region the first call filled is read again: any contents
leaking from one call into the next would show.

This file is named so that pytest collects it last.
"""
import ctypes

import pytest
import torch

import chunked_ssd_scan_gb300 as pkg
import oracle
from chunked_ssd_scan_gb300 import workloads as wl
from tests.parity_util import check_close, to_np

pytestmark = pytest.mark.gpu

TOL = 1e-4   # the selective-scan parity tolerance: |got - ref| <= 1e-4 * (1 + |ref|)
_VP = ctypes.c_void_p


def _fn():
    lib = pkg.load_library()
    f = lib.selective_scan_forward_noalloc
    f.restype = ctypes.c_int
    f.argtypes = [_VP] * 7 + [ctypes.c_int64] * 4 + [_VP]
    return f


def _p(t):
    return _VP(None) if t is None else _VP(t.data_ptr())


def test_noalloc_matches_workspace_entry_point_and_oracle_on_calls_in_a_row():
    f = _fn()
    stream = _VP(torch.cuda.current_stream().cuda_stream)
    small = wl.SelectiveScanConfig("second", 2, 1000, 96, 7)
    # the full workload twice (other seeds the second time), then a smaller odd shape
    cases = [(wl.SELECTIVE_SCAN_F32, 0), (wl.SELECTIVE_SCAN_F32, 3), (small, 1)]
    for cfg, seed in cases:
        s = wl.make_selective_scan_inputs(cfg, seed=seed, device="cuda")
        ref = pkg.selective_scan_forward(s["u"], s["delta"], s["A"], s["B"], s["C"], s["skip"])
        y = torch.full_like(s["u"], float("nan"))
        st = f(_p(s["u"]), _p(s["delta"]), _p(s["A"]), _p(s["B"]), _p(s["C"]), _p(s["skip"]),
               _p(y), cfg.batch, cfg.seqlen, cfg.d_model, cfg.d_state, stream)
        assert st == 0, pkg.STATUS.get(st, st)
        torch.cuda.synchronize()
        what = f"{cfg.name}, seed {seed}"
        check_close(to_np(y), to_np(ref), TOL, f"noalloc vs workspace entry point ({what})")
        yo = oracle.selective_scan(*(to_np(s[k]) for k in ("u", "delta", "A", "B", "C", "skip")))
        check_close(to_np(y), yo, TOL, f"noalloc vs oracle ({what})")


def test_noalloc_rejects_sizes_beyond_its_scratch():
    f = _fn()
    u = torch.zeros(16, device="cuda")
    # 64 x 4096 x 4096 x 16 needs far more than the 16 MiB scratch: rejected before any launch
    st = f(*[_p(u)] * 7, 64, 4096, 4096, 16, _VP(None))
    assert st == 2

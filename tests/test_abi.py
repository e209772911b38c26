"""The C-ABI library loads and exports every declared symbol; host-side validation (CPU only).

No test here launches device work: every call either needs no GPU (sizes, status strings) or is
rejected by host validation before any launch.
"""
import ctypes
import os
import re

import pytest
import torch

import chunked_ssd_scan_gb300 as pkg
from chunked_ssd_scan_gb300 import _build
from chunked_ssd_scan_gb300 import workloads as wl

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "ssdscan.h")


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    src = re.sub(r"//[^\n]*", "", src)
    names = re.findall(r"^(?!typedef|#)[A-Za-z_][\w \t\*]*?\b([a-z_][a-z0-9_]*)\s*\(", src,
                       flags=re.M)
    return sorted(set(names))


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return pkg.load_library()


def test_header_declares_the_abi():
    names = declared_functions()
    for expected in ("ssd_chunked_forward", "ssd_chunked_workspace_bytes", "ssd_chunked_variant",
                     "selective_scan_forward", "selective_scan_workspace_bytes",
                     "ssd_workspace_status", "ssd_status_string", "ssd_abi_version",
                     "ssd_trapezoidal_forward", "ssd_trapezoidal_workspace_bytes",
                     "ssd_rotation_variant_forward", "ssd_rotation_variant_workspace_bytes",
                     "ssd_quaternion_forward", "ssd_quaternion_workspace_bytes",
                     "ssd_chunked_backward", "ssd_backward_workspace_bytes",
                     "ssd_chunked_forward_varlen", "ssd_trapezoidal_forward_varlen",
                     "ssd_trapezoidal_variant"):
        assert expected in names


def test_library_exports_every_declared_symbol(lib):
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, f"not exported: {missing}"


def test_library_is_sm103a_build():
    # the in-tree build targets exactly sm_103a
    assert "arch=compute_103a,code=sm_103a" in " ".join(_build.ARCH)


def test_status_strings(lib):
    for code, name in pkg.STATUS.items():
        assert lib.ssd_status_string(code).decode() == name
    assert lib.ssd_abi_version() >= 1


def _shape(cfg: wl.SSDConfig, **kw):
    d = dict(batch=cfg.batch, seqlen=cfg.seqlen, nheads=cfg.nheads, headdim=cfg.headdim,
             dstate=cfg.dstate, ngroups=cfg.ngroups, mimo_rank=cfg.mimo_rank,
             chunk_len=cfg.chunk_len, io_dtype=1 if cfg.dtype == "bf16" else 0,
             has_theta=1 if cfg.theta else 0)
    d.update(kw)
    return pkg.ssd_shape(**d)


@pytest.mark.parametrize("cfg", wl.SSD_CONFIGS, ids=lambda c: c.name)
def test_workspace_sizes_for_every_workload(lib, cfg):
    s = _shape(cfg)
    n = lib.ssd_chunked_workspace_bytes(ctypes.byref(s))
    assert n > 0 and n % 256 == 0
    assert lib.ssd_chunked_variant(ctypes.byref(s)) != 0


def test_selective_scan_workspace(lib):
    c = wl.SELECTIVE_SCAN_F32
    assert lib.selective_scan_workspace_bytes(c.batch, c.seqlen, c.d_model, c.d_state) > 0
    assert lib.selective_scan_workspace_bytes(1, 10, 4, 65) == 0
    assert lib.selective_scan_workspace_bytes(0, 10, 4, 16) == 0


@pytest.mark.parametrize("kw", [dict(batch=0), dict(seqlen=0), dict(nheads=0), dict(headdim=-1),
                                dict(ngroups=3), dict(io_dtype=7), dict(has_theta=1, dstate=15),
                                dict(mimo_rank=0), dict(chunk_len=0)])
def test_invalid_shapes_have_no_workspace(lib, kw):
    s = _shape(wl.TINY_SISO_F32, **kw)
    assert lib.ssd_chunked_workspace_bytes(ctypes.byref(s)) == 0
    assert lib.ssd_chunked_variant(ctypes.byref(s)) == 0


# The fake pointers below are never dereferenced because validation rejects each call before
# any launch.  They are only used where no GPU is present.
no_gpu_only = pytest.mark.skipif(torch.cuda.is_available(),
                                 reason="fake-pointer validation tests run on CPU-only hosts")

_VP = ctypes.c_void_p
A16 = 0x100000


def _call(lib, shape, x=A16, dA=A16, B=A16, C=A16, theta=None, init=None, y=A16, fin=None,
          ws=A16, ws_bytes=None):
    if ws_bytes is None:
        ws_bytes = lib.ssd_chunked_workspace_bytes(ctypes.byref(shape))
    return lib.ssd_chunked_forward(ctypes.byref(shape), _VP(x), _VP(dA), _VP(B), _VP(C),
                                   _VP(theta), _VP(init), _VP(y), _VP(fin), _VP(ws),
                                   ctypes.c_size_t(ws_bytes), _VP(None))


@no_gpu_only
def test_null_and_misaligned_pointers_rejected(lib):
    s = _shape(wl.TINY_SISO_F32)
    assert _call(lib, s, x=None) == 1
    assert _call(lib, s, dA=None) == 1
    assert _call(lib, s, y=None) == 1
    assert _call(lib, s, B=A16 + 2) == 1
    assert _call(lib, s, fin=A16 + 8) == 1
    assert _call(lib, s, theta=A16) == 1           # theta given but has_theta == 0
    st = _shape(wl.TINY_SISO_F32, has_theta=1)
    assert _call(lib, st, theta=None) == 1         # has_theta == 1 but no theta


@no_gpu_only
def test_workspace_errors(lib):
    s = _shape(wl.TINY_SISO_F32)
    need = lib.ssd_chunked_workspace_bytes(ctypes.byref(s))
    assert _call(lib, s, ws=None) == 4
    assert _call(lib, s, ws_bytes=need - 1) == 4
    assert _call(lib, s, ws=A16 + 16) == 4


@no_gpu_only
def test_unsupported_shapes(lib):
    s = _shape(wl.TINY_SISO_F32, chunk_len=8192)   # fused chunk beyond every path's limit
    assert _call(lib, s, ws_bytes=1 << 30) == 2
    s = _shape(wl.TINY_SISO_F32, headdim=512)
    assert _call(lib, s, ws_bytes=1 << 30) == 2


@no_gpu_only
def test_selective_scan_rejections(lib):
    f = lib.selective_scan_forward
    args = [_VP(A16)] * 7
    assert f(*args, 1, 16, 8, 65, _VP(A16), ctypes.c_size_t(1 << 20), _VP(None)) == 2
    bad = list(args)
    bad[0] = _VP(None)
    assert f(*bad, 1, 16, 8, 16, _VP(A16), ctypes.c_size_t(1 << 20), _VP(None)) == 1
    assert f(*args, 1, 16, 8, 16, _VP(A16), ctypes.c_size_t(8), _VP(None)) == 4


@no_gpu_only
def test_wait_selftest_argument_checks(lib):
    """Rejected on the host before any launch (no GPU needed)."""
    f = lib.ssd_wait_selftest
    f.restype = ctypes.c_int
    f.argtypes = [_VP, ctypes.c_size_t, ctypes.c_uint64, _VP]
    assert f(None, 256, 1000, None) == 4                      # no workspace
    assert f(_VP(A16 + 16), 256, 1000, None) == 4             # not 256-byte aligned
    assert f(_VP(A16), 128, 1000, None) == 4                  # smaller than the header
    assert f(_VP(A16), 256, 0, None) == 1                     # no wait
    assert f(_VP(A16), 256, 200_000_000, None) == 1           # above the 100 ms cap


def _bwd(lib, shape, theta=None, dtheta=None, dx=A16, ddA=A16, x=A16, ws=A16, ws_bytes=None):
    if ws_bytes is None:
        ws_bytes = lib.ssd_backward_workspace_bytes(ctypes.byref(shape))
    return lib.ssd_chunked_backward(ctypes.byref(shape), _VP(x), _VP(A16), _VP(A16), _VP(A16),
                                    _VP(theta), _VP(None), _VP(A16), _VP(None), _VP(dx),
                                    _VP(ddA), _VP(A16), _VP(A16), _VP(dtheta), _VP(None),
                                    _VP(ws), ctypes.c_size_t(ws_bytes), _VP(None))


def test_backward_workspace_sizes(lib):
    plain = _shape(wl.TINY_SISO_F32)
    rot = _shape(wl.TINY_SISO_F32, has_theta=1)
    assert lib.ssd_backward_workspace_bytes(ctypes.byref(plain)) > 0
    assert (lib.ssd_backward_workspace_bytes(ctypes.byref(rot))
            > lib.ssd_backward_workspace_bytes(ctypes.byref(plain)))
    for bad in (_shape(wl.TINY_SISO_F32, headdim=128), _shape(wl.TINY_SISO_F32, dstate=18),
                _shape(wl.TINY_SISO_F32, dstate=256), _shape(wl.TINY_SISO_F32, mimo_rank=128)):
        assert lib.ssd_backward_workspace_bytes(ctypes.byref(bad)) == 0
    trap = _shape(wl.TINY_SISO_F32, mimo_rank=2)
    assert lib.ssd_trapezoidal_backward_workspace_bytes(ctypes.byref(trap)) > 0
    wide = _shape(wl.TINY_SISO_F32, mimo_rank=64)   # 128 write channels after the expansion
    assert lib.ssd_trapezoidal_backward_workspace_bytes(ctypes.byref(wide)) == 0


@no_gpu_only
def test_backward_host_rejections(lib):
    """Rejected on the host before any launch (no GPU needed)."""
    plain = _shape(wl.TINY_SISO_F32)
    rot = _shape(wl.TINY_SISO_F32, has_theta=1)
    assert _bwd(lib, plain, x=None) == 1                       # x missing
    assert _bwd(lib, plain, ddA=None) == 1                     # ddA missing
    assert _bwd(lib, plain, dx=A16 + 4) == 1                   # misaligned gradient
    assert _bwd(lib, plain, theta=A16, dtheta=A16) == 1        # theta without has_theta
    assert _bwd(lib, rot, theta=None, dtheta=A16) == 1         # has_theta without theta
    assert _bwd(lib, rot, theta=A16, dtheta=None) == 1         # no dtheta for theta
    assert _bwd(lib, plain, ws=None) == 4
    assert _bwd(lib, plain, ws_bytes=64) == 4
    assert _bwd(lib, plain, ws=A16 + 16) == 4
    assert _bwd(lib, _shape(wl.TINY_SISO_F32, dstate=18), ws_bytes=1 << 30) == 2
    f = lib.ssd_trapezoidal_backward
    trap = _shape(wl.TINY_SISO_F32, mimo_rank=2)
    need = lib.ssd_trapezoidal_backward_workspace_bytes(ctypes.byref(trap))
    # x dA B C gamma beta | theta prev_x prev_B init | dy | dfinal | dx ddA dB dC dgamma dbeta |
    # dtheta dinit dprev_x dprev_B | workspace
    ptrs = ([_VP(A16)] * 6 + [_VP(None)] * 4 + [_VP(A16)] + [_VP(None)] + [_VP(A16)] * 6
            + [_VP(None)] * 4 + [_VP(A16)])
    assert len(ptrs) == 23
    args = lambda p, nbytes: (ctypes.byref(trap), *p, ctypes.c_size_t(nbytes), _VP(None))
    assert f(*args(ptrs, need - 1)) == 4                        # workspace too small
    bad = list(ptrs)
    bad[4] = _VP(None)                                          # gamma missing
    assert f(*args(bad, need)) == 1
    bad = list(ptrs)
    bad[7] = _VP(A16)                                           # prev_x without prev_B
    assert f(*args(bad, need)) == 1


def declared_parameter_counts():
    """Number of parameters of every function declared in the header."""
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    src = re.sub(r"//[^\n]*", "", src)
    counts = {}
    for m in re.finditer(r"^(?!typedef|#)[A-Za-z_][\w \t\*]*?\b([a-z_][a-z0-9_]*)\s*\(([^)]*)\)\s*;",
                         src, flags=re.M):
        params = m.group(2).strip()
        counts[m.group(1)] = 0 if params in ("", "void") else len(params.split(","))
    return counts


def test_binding_argument_counts_match_the_header(lib):
    """Every function the binding gives argtypes to takes as many arguments as the header
    declares (a miscounted binding would fail only when called on a GPU)."""
    counts = declared_parameter_counts()
    assert counts, "no declarations parsed"
    checked = 0
    for name, n in counts.items():
        argtypes = getattr(getattr(lib, name), "argtypes", None)
        if argtypes is None:
            continue
        assert len(argtypes) == n, f"{name}: binding has {len(argtypes)} arguments, header {n}"
        checked += 1
    assert checked >= 10

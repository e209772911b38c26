"""chunked_ssd_scan_gb300 -- chunked SSD scan and selective scan on GB300 (sm_103a).

Thin Python binding over the C ABI in include/ssdscan.h (libssdscan.so, built in-tree by
``_build.build()``).  PyTorch supplies device memory and the current stream; every step of the
computation runs in the library's CUDA kernels.  If the shared library is missing this module
raises: there is no Python or CPU fallback.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

from . import workloads  # noqa: F401  (seeded synthetic inputs; no scan arithmetic)

__all__ = [
    "SSDError", "load_library", "ssd_shape", "ssd_chunked_workspace_bytes", "ssd_chunked_variant",
    "ssd_chunked_launches", "ssd_chunked_forward", "ssd_trapezoidal_variant", "SSDForwardPlan", "SelectiveScanPlan",
    "selective_scan_workspace_bytes", "selective_scan_forward", "ssd_trapezoidal_workspace_bytes",
    "ssd_trapezoidal_forward", "SSDTrapezoidalPlan", "ssd_rotation_variant_forward",
    "ssd_quaternion_forward",
    "ssd_backward_workspace_bytes", "ssd_chunked_backward", "SSDBackwardPlan",
    "ssd_trapezoidal_backward", "ssd_trapezoidal_backward_workspace_bytes",
    "workspace_status", "wait_selftest", "STATUS", "VARIANTS",
]

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libssdscan.so")

STATUS = {0: "SSD_OK", 1: "SSD_ERR_INVALID_ARG", 2: "SSD_ERR_UNSUPPORTED", 3: "SSD_ERR_CUDA",
          4: "SSD_ERR_WORKSPACE", 5: "SSD_ERR_TIMEOUT", 6: "SSD_ERR_INDEX"}
VARIANTS = {0: "none", 1: "generic", 2: "tc_bf16", 3: "tiled_f32", 4: "tc_tf32"}
SSD_F32, SSD_BF16 = 0, 1


class SSDError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = int(status)
        super().__init__(f"{what}: {STATUS.get(int(status), status)}")


class ssd_shape(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int64), ("seqlen", ctypes.c_int64), ("nheads", ctypes.c_int64),
                ("headdim", ctypes.c_int64), ("dstate", ctypes.c_int64),
                ("ngroups", ctypes.c_int64), ("mimo_rank", ctypes.c_int64),
                ("chunk_len", ctypes.c_int64), ("io_dtype", ctypes.c_int32),
                ("has_theta", ctypes.c_int32)]


_LIB = None
_VP = ctypes.c_void_p
_I64 = ctypes.c_int64


def load_library(path: Optional[str] = None):
    """Load libssdscan.so (raises if it has not been built)."""
    global _LIB
    if _LIB is not None and path is None:
        return _LIB
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise RuntimeError(f"libssdscan.so not found at {p}; build it with "
                           "`python -c 'import __graft_entry__ as g; g.build()'`")
    lib = ctypes.CDLL(p)
    SP = ctypes.POINTER(ssd_shape)
    lib.ssd_chunked_workspace_bytes.restype = ctypes.c_size_t
    lib.ssd_chunked_workspace_bytes.argtypes = [SP]
    lib.ssd_chunked_variant.restype = ctypes.c_int32
    lib.ssd_chunked_variant.argtypes = [SP]
    lib.ssd_chunked_launches.restype = ctypes.c_int32
    lib.ssd_chunked_launches.argtypes = [SP]
    lib.ssd_chunked_forward.restype = ctypes.c_int
    lib.ssd_chunked_forward.argtypes = [SP] + [_VP] * 9 + [ctypes.c_size_t, _VP]
    lib.ssd_chunked_forward_varlen.restype = ctypes.c_int
    lib.ssd_chunked_forward_varlen.argtypes = [SP] + [_VP] * 10 + [ctypes.c_size_t, _VP]
    lib.ssd_chunked_forward_tf32.restype = ctypes.c_int
    lib.ssd_chunked_forward_tf32.argtypes = [SP] + [_VP] * 10 + [ctypes.c_size_t, _VP]
    lib.ssd_trapezoidal_workspace_bytes.restype = ctypes.c_size_t
    lib.ssd_trapezoidal_workspace_bytes.argtypes = [SP]
    lib.ssd_trapezoidal_variant.restype = ctypes.c_int32
    lib.ssd_trapezoidal_variant.argtypes = [SP]
    lib.ssd_trapezoidal_forward.restype = ctypes.c_int
    lib.ssd_trapezoidal_forward.argtypes = [SP] + [_VP] * 13 + [ctypes.c_size_t, _VP]
    lib.ssd_trapezoidal_forward_varlen.restype = ctypes.c_int
    lib.ssd_trapezoidal_forward_varlen.argtypes = [SP] + [_VP] * 14 + [ctypes.c_size_t, _VP]
    lib.ssd_quaternion_workspace_bytes.restype = ctypes.c_size_t
    lib.ssd_quaternion_workspace_bytes.argtypes = [SP]
    lib.ssd_quaternion_forward.restype = ctypes.c_int
    lib.ssd_quaternion_forward.argtypes = [SP] + [_VP] * 9 + [ctypes.c_size_t, _VP]
    lib.ssd_rotation_variant_workspace_bytes.restype = ctypes.c_size_t
    lib.ssd_rotation_variant_workspace_bytes.argtypes = [SP, _I64, ctypes.c_int32]
    lib.ssd_rotation_variant_forward.restype = ctypes.c_int
    lib.ssd_rotation_variant_forward.argtypes = ([SP, _I64, ctypes.c_int32] + [_VP] * 9
                                                 + [ctypes.c_size_t, _VP])
    lib.selective_scan_workspace_bytes.restype = ctypes.c_size_t
    lib.ssd_backward_workspace_bytes.restype = ctypes.c_size_t
    lib.ssd_backward_workspace_bytes.argtypes = [SP]
    lib.ssd_chunked_backward.restype = ctypes.c_int
    lib.ssd_chunked_backward.argtypes = [SP] + [_VP] * 15 + [ctypes.c_size_t, _VP]
    lib.ssd_trapezoidal_backward_workspace_bytes.restype = ctypes.c_size_t
    lib.ssd_trapezoidal_backward_workspace_bytes.argtypes = [SP]
    lib.ssd_trapezoidal_backward.restype = ctypes.c_int
    lib.ssd_trapezoidal_backward.argtypes = [SP] + [_VP] * 23 + [ctypes.c_size_t, _VP]
    lib.selective_scan_workspace_bytes.argtypes = [_I64] * 4
    lib.selective_scan_forward.restype = ctypes.c_int
    lib.selective_scan_forward.argtypes = [_VP] * 7 + [_I64] * 4 + [_VP, ctypes.c_size_t, _VP]
    lib.ssd_workspace_status.restype = ctypes.c_int
    lib.ssd_workspace_status.argtypes = [_VP, _VP, ctypes.POINTER(ctypes.c_int64)]
    lib.ssd_status_string.restype = ctypes.c_char_p
    lib.ssd_status_string.argtypes = [ctypes.c_int]
    lib.ssd_wait_selftest.restype = ctypes.c_int
    lib.ssd_wait_selftest.argtypes = [_VP, ctypes.c_size_t, ctypes.c_uint64, _VP]
    lib.ssd_abi_version.restype = ctypes.c_int32
    lib.ssd_abi_version.argtypes = []
    if path is None:
        _LIB = lib
    return lib


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream_handle(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _check_cuda(name, t, dtype=None, shape=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must have dtype {dtype}, got {t.dtype}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")


def make_shape(batch, seqlen, nheads, headdim, dstate, ngroups, mimo_rank, chunk_len,
               io_dtype, has_theta) -> ssd_shape:
    return ssd_shape(batch, seqlen, nheads, headdim, dstate, ngroups, mimo_rank, chunk_len,
                     SSD_BF16 if io_dtype in (torch.bfloat16, SSD_BF16, "bf16") else SSD_F32,
                     1 if has_theta else 0)


def ssd_chunked_workspace_bytes(shape: ssd_shape) -> int:
    return int(load_library().ssd_chunked_workspace_bytes(ctypes.byref(shape)))


def ssd_chunked_variant(shape: ssd_shape) -> str:
    return VARIANTS.get(int(load_library().ssd_chunked_variant(ctypes.byref(shape))), "none")


def ssd_chunked_launches(shape: ssd_shape) -> int:
    """Kernel launches per ``ssd_chunked_forward`` call for ``shape`` on the current device."""
    return int(load_library().ssd_chunked_launches(ctypes.byref(shape)))


def shape_of(x: torch.Tensor, B: torch.Tensor, chunk_len: int, has_theta: bool) -> ssd_shape:
    b, T, R, H, P = x.shape
    G, N = B.shape[3], B.shape[4]
    return make_shape(b, T, H, P, N, G, R, chunk_len, x.dtype, has_theta)


class SSDForwardPlan:
    """Arguments of ``ssd_chunked_forward`` validated once, for repeated calls on the same
    buffers.  Calling the plan makes only the C call (on the stream given here, or the stream
    that is current at construction).  Shapes and dtypes are those of ``ssd_chunked_forward``;
    with ``valid_len`` (int64 [b] on the device) the plan calls ``ssd_chunked_forward_varlen``;
    with ``tf32=True`` (fp32, P = N = 64) it calls ``ssd_chunked_forward_tf32`` (valid_len
    optional), whose chunk scan runs on the tensor core.
    """

    def __init__(self, x: torch.Tensor, dA: torch.Tensor, B: torch.Tensor, C: torch.Tensor, *,
                 chunk_len: int, theta: Optional[torch.Tensor] = None,
                 init_state: Optional[torch.Tensor] = None, y: Optional[torch.Tensor] = None,
                 final_state: Optional[torch.Tensor] = None, return_final_state: bool = True,
                 workspace: Optional[torch.Tensor] = None, stream=None,
                 valid_len: Optional[torch.Tensor] = None, tf32: bool = False):
        if x.dim() != 5 or B.dim() != 5:
            raise ValueError("x must be [b,T,R,H,P] and B/C [b,T,R,G,N]")
        b, T, R, H, P = x.shape
        G, N = B.shape[3], B.shape[4]
        _check_cuda("x", x)
        if x.dtype not in (torch.float32, torch.bfloat16):
            raise ValueError("x/B/C must be float32 or bfloat16")
        _check_cuda("B", B, x.dtype, (b, T, R, G, N))
        _check_cuda("C", C, x.dtype, (b, T, R, G, N))
        _check_cuda("dA", dA, torch.float32, (b, T, H))
        if theta is not None:
            _check_cuda("theta", theta, torch.float32, (b, T, H, N // 2))
        if init_state is not None:
            _check_cuda("init_state", init_state, torch.float32, (b, H, P, N))
        if valid_len is not None:
            _check_cuda("valid_len", valid_len, torch.int64, (b,))
        self.shape = shape_of(x, B, chunk_len, theta is not None)
        self._lib = load_library()
        if y is None:
            y = torch.empty_like(x)
        _check_cuda("y", y, x.dtype, x.shape)
        if final_state is None and return_final_state:
            final_state = torch.empty((b, H, P, N), dtype=torch.float32, device=x.device)
        if final_state is not None:
            _check_cuda("final_state", final_state, torch.float32, (b, H, P, N))
        need = int(self._lib.ssd_chunked_workspace_bytes(ctypes.byref(self.shape)))
        if need == 0:
            raise SSDError(2, "ssd_chunked_workspace_bytes (shape not supported)")
        if workspace is None:
            workspace = torch.zeros(need, dtype=torch.uint8, device=x.device)   # zero header
        _check_cuda("workspace", workspace, torch.uint8)
        # keep every buffer alive as long as the plan
        self.inputs = (x, dA, B, C, theta, init_state, valid_len)
        self.y, self.final_state, self.workspace = y, final_state, workspace
        vl = (_ptr(valid_len),) if (tf32 or valid_len is not None) else ()
        self._args = (ctypes.byref(self.shape), _ptr(x), _ptr(dA), _ptr(B), _ptr(C), _ptr(theta),
                      *vl, _ptr(init_state), _ptr(y), _ptr(final_state), _ptr(workspace),
                      ctypes.c_size_t(workspace.numel()), _stream_handle(stream))
        self._name = "ssd_chunked_forward" + ("_tf32" if tf32 else
                                              "" if valid_len is None else "_varlen")
        self._fn = getattr(self._lib, self._name)

    def __call__(self):
        st = self._fn(*self._args)
        if st != 0:
            raise SSDError(st, self._name)
        return self.y, self.final_state


def ssd_chunked_forward(x: torch.Tensor, dA: torch.Tensor, B: torch.Tensor, C: torch.Tensor, *,
                        chunk_len: int, theta: Optional[torch.Tensor] = None,
                        init_state: Optional[torch.Tensor] = None,
                        y: Optional[torch.Tensor] = None,
                        final_state: Optional[torch.Tensor] = None,
                        return_final_state: bool = True,
                        workspace: Optional[torch.Tensor] = None, stream=None,
                        valid_len: Optional[torch.Tensor] = None, tf32: bool = False):
    """Chunked SSD forward scan through ``ssd_chunked_forward`` (``ssd_chunked_forward_varlen``
    when ``valid_len`` is given, ``ssd_chunked_forward_tf32`` with ``tf32=True``).

    x [b,T,R,H,P], B/C [b,T,R,G,N] (all f32 or all bf16), dA [b,T,H] f32, theta [b,T,H,N/2] f32,
    init_state [b,H,P,N] f32, valid_len [b] int64 (steps from valid_len[b] on are padding; y is
    not written there).  Returns (y, final_state) (final_state None if not requested).
    """
    return SSDForwardPlan(x, dA, B, C, chunk_len=chunk_len, theta=theta, init_state=init_state,
                          y=y, final_state=final_state, return_final_state=return_final_state,
                          workspace=workspace, stream=stream, valid_len=valid_len, tf32=tf32)()


def ssd_trapezoidal_workspace_bytes(shape: ssd_shape) -> int:
    return int(load_library().ssd_trapezoidal_workspace_bytes(ctypes.byref(shape)))


def ssd_trapezoidal_variant(shape: ssd_shape) -> str:
    return VARIANTS.get(int(load_library().ssd_trapezoidal_variant(ctypes.byref(shape))), "none")


class SSDTrapezoidalPlan:
    """Validated buffers for repeated ``ssd_trapezoidal_forward`` calls (C-ABI call only).

    x [b,T,R,H,P], B/C [b,T,R,G,N] (f32 or bf16), dA, gamma, beta [b,T,H] f32,
    theta [b,T,H,N/2] f32, prev_x [b,R,H,P] and prev_B [b,R,G,N] (x's dtype; the previous call's
    last step, both or neither), init_state [b,H,P,N] f32.
    """

    def __init__(self, x, dA, B, C, gamma, beta, *, chunk_len: int, theta=None, prev_x=None,
                 prev_B=None, init_state=None, y=None, final_state=None,
                 return_final_state: bool = True, workspace=None, stream=None, valid_len=None):
        if x.dim() != 5 or B.dim() != 5:
            raise ValueError("x must be [b,T,R,H,P] and B/C [b,T,R,G,N]")
        b, T, R, H, P = x.shape
        G, N = B.shape[3], B.shape[4]
        _check_cuda("x", x)
        if x.dtype not in (torch.float32, torch.bfloat16):
            raise ValueError("x/B/C must be float32 or bfloat16")
        _check_cuda("B", B, x.dtype, (b, T, R, G, N))
        _check_cuda("C", C, x.dtype, (b, T, R, G, N))
        for name, t in (("dA", dA), ("gamma", gamma), ("beta", beta)):
            _check_cuda(name, t, torch.float32, (b, T, H))
        if theta is not None:
            _check_cuda("theta", theta, torch.float32, (b, T, H, N // 2))
        if (prev_x is None) != (prev_B is None):
            raise ValueError("prev_x and prev_B go together")
        if prev_x is not None:
            _check_cuda("prev_x", prev_x, x.dtype, (b, R, H, P))
            _check_cuda("prev_B", prev_B, x.dtype, (b, R, G, N))
        if init_state is not None:
            _check_cuda("init_state", init_state, torch.float32, (b, H, P, N))
        if valid_len is not None:
            _check_cuda("valid_len", valid_len, torch.int64, (b,))
        self.shape = shape_of(x, B, chunk_len, theta is not None)
        self._lib = load_library()
        if y is None:
            y = torch.empty_like(x)
        _check_cuda("y", y, x.dtype, x.shape)
        if final_state is None and return_final_state:
            final_state = torch.empty((b, H, P, N), dtype=torch.float32, device=x.device)
        if final_state is not None:
            _check_cuda("final_state", final_state, torch.float32, (b, H, P, N))
        need = int(self._lib.ssd_trapezoidal_workspace_bytes(ctypes.byref(self.shape)))
        if need == 0:
            raise SSDError(2, "ssd_trapezoidal_workspace_bytes (shape not supported)")
        if workspace is None:
            workspace = torch.zeros(need, dtype=torch.uint8, device=x.device)   # zero header
        _check_cuda("workspace", workspace, torch.uint8)
        self.inputs = (x, dA, B, C, gamma, beta, theta, prev_x, prev_B, init_state, valid_len)
        self.y, self.final_state, self.workspace = y, final_state, workspace
        vl = () if valid_len is None else (_ptr(valid_len),)
        self._args = (ctypes.byref(self.shape), _ptr(x), _ptr(dA), _ptr(B), _ptr(C), _ptr(gamma),
                      _ptr(beta), _ptr(theta), _ptr(prev_x), _ptr(prev_B), *vl,
                      _ptr(init_state), _ptr(y), _ptr(final_state), _ptr(workspace),
                      ctypes.c_size_t(workspace.numel()), _stream_handle(stream))
        self._name = "ssd_trapezoidal_forward" + ("" if valid_len is None else "_varlen")
        self._fn = getattr(self._lib, self._name)

    def __call__(self):
        st = self._fn(*self._args)
        if st != 0:
            raise SSDError(st, self._name)
        return self.y, self.final_state


def ssd_trapezoidal_forward(x, dA, B, C, gamma, beta, *, chunk_len: int, theta=None,
                            prev_x=None, prev_B=None, init_state=None, y=None, final_state=None,
                            return_final_state: bool = True, workspace=None, stream=None,
                            valid_len=None):
    """Trapezoidal Mamba-3 forward through ``ssd_trapezoidal_forward`` (the ``_varlen`` entry
    point when ``valid_len`` [b] int64 is given); returns (y, final)."""
    return SSDTrapezoidalPlan(x, dA, B, C, gamma, beta, chunk_len=chunk_len, theta=theta,
                              prev_x=prev_x, prev_B=prev_B, init_state=init_state, y=y,
                              final_state=final_state, return_final_state=return_final_state,
                              workspace=workspace, stream=stream, valid_len=valid_len)()


def ssd_quaternion_forward(x, dA, B, C, qcum, *, chunk_len: int, init_state=None, y=None,
                           final_state=None, return_final_state: bool = True, workspace=None,
                           stream=None):
    """SSD forward with the quaternion rotation through ``ssd_quaternion_forward``: qcum
    [b,T,H,N/4,4] f32 cumulative unit quaternions (w, x, y, z) of the state's 4-blocks.
    Returns (y, final)."""
    if x.dim() != 5 or B.dim() != 5:
        raise ValueError("x must be [b,T,R,H,P] and B/C [b,T,R,G,N]")
    b, T, R, H, P = x.shape
    G, N = B.shape[3], B.shape[4]
    _check_cuda("x", x)
    _check_cuda("B", B, x.dtype, (b, T, R, G, N))
    _check_cuda("C", C, x.dtype, (b, T, R, G, N))
    _check_cuda("dA", dA, torch.float32, (b, T, H))
    _check_cuda("qcum", qcum, torch.float32, (b, T, H, N // 4, 4))
    if init_state is not None:
        _check_cuda("init_state", init_state, torch.float32, (b, H, P, N))
    shape = shape_of(x, B, chunk_len, False)
    lib = load_library()
    if y is None:
        y = torch.empty_like(x)
    if final_state is None and return_final_state:
        final_state = torch.empty((b, H, P, N), dtype=torch.float32, device=x.device)
    need = int(lib.ssd_quaternion_workspace_bytes(ctypes.byref(shape)))
    if need == 0:
        raise SSDError(2, "ssd_quaternion_workspace_bytes (shape not supported)")
    if workspace is None:
        workspace = torch.zeros(need, dtype=torch.uint8, device=x.device)
    st = lib.ssd_quaternion_forward(ctypes.byref(shape), _ptr(x), _ptr(dA), _ptr(B), _ptr(C),
                                    _ptr(qcum), _ptr(init_state), _ptr(y), _ptr(final_state),
                                    _ptr(workspace), ctypes.c_size_t(workspace.numel()),
                                    _stream_handle(stream))
    if st != 0:
        raise SSDError(st, "ssd_quaternion_forward")
    return y, final_state


def ssd_rotation_variant_forward(x, dA, B, C, theta, *, chunk_len: int, rope_dim: int = 0,
                                 halves: bool = False, init_state=None, y=None,
                                 final_state=None, return_final_state: bool = True,
                                 workspace=None, stream=None):
    """Rotated SSD forward with a partial rotation (the first rope_dim state dims, 0 = all) and
    the interleaved (2k, 2k+1) or split-halves (k, k + rope_dim/2) pairing, through
    ``ssd_rotation_variant_forward``.  theta [b,T,H,rope_dim/2] f32.  Returns (y, final)."""
    if x.dim() != 5 or B.dim() != 5:
        raise ValueError("x must be [b,T,R,H,P] and B/C [b,T,R,G,N]")
    b, T, R, H, P = x.shape
    G, N = B.shape[3], B.shape[4]
    rd = rope_dim or N
    _check_cuda("x", x)
    _check_cuda("B", B, x.dtype, (b, T, R, G, N))
    _check_cuda("C", C, x.dtype, (b, T, R, G, N))
    _check_cuda("dA", dA, torch.float32, (b, T, H))
    _check_cuda("theta", theta, torch.float32, (b, T, H, rd // 2))
    if init_state is not None:
        _check_cuda("init_state", init_state, torch.float32, (b, H, P, N))
    shape = shape_of(x, B, chunk_len, True)
    lib = load_library()
    if y is None:
        y = torch.empty_like(x)
    if final_state is None and return_final_state:
        final_state = torch.empty((b, H, P, N), dtype=torch.float32, device=x.device)
    need = int(lib.ssd_rotation_variant_workspace_bytes(ctypes.byref(shape), int(rope_dim),
                                                        int(bool(halves))))
    if need == 0:
        raise SSDError(2, "ssd_rotation_variant_workspace_bytes (shape not supported)")
    if workspace is None:
        workspace = torch.zeros(need, dtype=torch.uint8, device=x.device)
    st = lib.ssd_rotation_variant_forward(ctypes.byref(shape), int(rope_dim), int(bool(halves)),
                                          _ptr(x), _ptr(dA), _ptr(B), _ptr(C), _ptr(theta),
                                          _ptr(init_state), _ptr(y), _ptr(final_state),
                                          _ptr(workspace), ctypes.c_size_t(workspace.numel()),
                                          _stream_handle(stream))
    if st != 0:
        raise SSDError(st, "ssd_rotation_variant_forward")
    return y, final_state


def ssd_backward_workspace_bytes(shape: ssd_shape) -> int:
    return int(load_library().ssd_backward_workspace_bytes(ctypes.byref(shape)))


class SSDBackwardPlan:
    """Arguments of ``ssd_chunked_backward`` validated once, for repeated calls on the same
    buffers (the gradients are allocated here unless given).  dy [b,T,R,H,P] and dfinal
    [b,H,P,N] are f32; theta [b,T,H,N/2] f32 selects the rotated form (and dtheta); every
    gradient is f32.  Calling the plan makes only the C call and returns the dict dx, ddA, dB,
    dC, dtheta (None without theta) and dinit (None unless return_dinit)."""

    def __init__(self, x: torch.Tensor, dA: torch.Tensor, B: torch.Tensor, C: torch.Tensor,
                 dy: torch.Tensor, *, theta: Optional[torch.Tensor] = None,
                 init_state: Optional[torch.Tensor] = None,
                 dfinal: Optional[torch.Tensor] = None, return_dinit: bool = True,
                 grads: Optional[dict] = None, workspace: Optional[torch.Tensor] = None,
                 stream=None):
        if x.dim() != 5 or B.dim() != 5:
            raise ValueError("x must be [b,T,R,H,P] and B/C [b,T,R,G,N]")
        b, T, R, H, P = x.shape
        G, N = B.shape[3], B.shape[4]
        _check_cuda("x", x)
        if x.dtype not in (torch.float32, torch.bfloat16):
            raise ValueError("x/B/C must be float32 or bfloat16")
        _check_cuda("B", B, x.dtype, (b, T, R, G, N))
        _check_cuda("C", C, x.dtype, (b, T, R, G, N))
        _check_cuda("dA", dA, torch.float32, (b, T, H))
        _check_cuda("dy", dy, torch.float32, (b, T, R, H, P))
        if theta is not None:
            _check_cuda("theta", theta, torch.float32, (b, T, H, N // 2))
        if init_state is not None:
            _check_cuda("init_state", init_state, torch.float32, (b, H, P, N))
        if dfinal is not None:
            _check_cuda("dfinal", dfinal, torch.float32, (b, H, P, N))
        self.shape = shape_of(x, B, 64, theta is not None)
        self._lib = load_library()
        need = int(self._lib.ssd_backward_workspace_bytes(ctypes.byref(self.shape)))
        if need == 0:
            raise SSDError(2, "ssd_backward_workspace_bytes (shape not supported)")
        if workspace is None:
            workspace = torch.zeros(need, dtype=torch.uint8, device=x.device)   # zero header
        _check_cuda("workspace", workspace, torch.uint8)
        shapes = {"dx": (b, T, R, H, P), "ddA": (b, T, H), "dB": (b, T, R, G, N),
                  "dC": (b, T, R, G, N), "dtheta": (b, T, H, N // 2), "dinit": (b, H, P, N)}
        g = dict(grads or {})
        for k, shp in shapes.items():
            if (k == "dinit" and not return_dinit) or (k == "dtheta" and theta is None):
                g[k] = None
                continue
            if g.get(k) is None:
                g[k] = torch.empty(shp, dtype=torch.float32, device=x.device)
            _check_cuda(k, g[k], torch.float32, shp)
        self.inputs = (x, dA, B, C, theta, dy, init_state, dfinal)
        self.grads, self.workspace = g, workspace
        self._args = (ctypes.byref(self.shape), _ptr(x), _ptr(dA), _ptr(B), _ptr(C), _ptr(theta),
                      _ptr(init_state), _ptr(dy), _ptr(dfinal), _ptr(g["dx"]), _ptr(g["ddA"]),
                      _ptr(g["dB"]), _ptr(g["dC"]), _ptr(g["dtheta"]), _ptr(g["dinit"]),
                      _ptr(workspace), ctypes.c_size_t(workspace.numel()),
                      _stream_handle(stream))
        self._fn = self._lib.ssd_chunked_backward

    def __call__(self):
        st = self._fn(*self._args)
        if st != 0:
            raise SSDError(st, "ssd_chunked_backward")
        return self.grads


def ssd_chunked_backward(x, dA, B, C, dy, *, theta=None, init_state=None, dfinal=None,
                         return_dinit: bool = True, grads=None, workspace=None, stream=None):
    """Gradients of <dy, y> + <dfinal, final_state> for the SSD forward (rotated when theta is
    given), through ``ssd_chunked_backward``.  Returns a dict of f32 tensors dx, ddA, dB, dC,
    dtheta and dinit."""
    return SSDBackwardPlan(x, dA, B, C, dy, theta=theta, init_state=init_state, dfinal=dfinal,
                           return_dinit=return_dinit, grads=grads, workspace=workspace,
                           stream=stream)()


def ssd_trapezoidal_backward_workspace_bytes(shape: ssd_shape) -> int:
    return int(load_library().ssd_trapezoidal_backward_workspace_bytes(ctypes.byref(shape)))


def ssd_trapezoidal_backward(x, dA, B, C, gamma, beta, dy, *, theta=None, prev_x=None,
                             prev_B=None, init_state=None, dfinal=None, grads=None,
                             workspace=None, stream=None):
    """Gradients of <dy, y> + <dfinal, final_state> for the trapezoidal forward, through
    ``ssd_trapezoidal_backward``.  Returns a dict of f32 tensors dx, ddA, dB, dC, dgamma, dbeta,
    dtheta (None without theta), dinit, dprev_x and dprev_B (None without a previous write),
    plus the workspace used; `grads` (such a dict) supplies the output tensors."""
    if x.dim() != 5 or B.dim() != 5:
        raise ValueError("x must be [b,T,R,H,P] and B/C [b,T,R,G,N]")
    b, T, R, H, P = x.shape
    G, N = B.shape[3], B.shape[4]
    _check_cuda("x", x)
    _check_cuda("B", B, x.dtype, (b, T, R, G, N))
    _check_cuda("C", C, x.dtype, (b, T, R, G, N))
    for name, v in (("dA", dA), ("gamma", gamma), ("beta", beta)):
        _check_cuda(name, v, torch.float32, (b, T, H))
    _check_cuda("dy", dy, torch.float32, (b, T, R, H, P))
    if theta is not None:
        _check_cuda("theta", theta, torch.float32, (b, T, H, N // 2))
    if (prev_x is None) != (prev_B is None):
        raise ValueError("prev_x and prev_B go together")
    if prev_x is not None:
        _check_cuda("prev_x", prev_x, x.dtype, (b, R, H, P))
        _check_cuda("prev_B", prev_B, x.dtype, (b, R, G, N))
    for name, v in (("init_state", init_state), ("dfinal", dfinal)):
        if v is not None:
            _check_cuda(name, v, torch.float32, (b, H, P, N))
    shape = shape_of(x, B, 64, theta is not None)
    lib = load_library()
    need = int(lib.ssd_trapezoidal_backward_workspace_bytes(ctypes.byref(shape)))
    if need == 0:
        raise SSDError(2, "ssd_trapezoidal_backward_workspace_bytes (shape not supported)")
    if workspace is None:
        workspace = torch.zeros(need, dtype=torch.uint8, device=x.device)
    shapes = {"dx": (b, T, R, H, P), "ddA": (b, T, H), "dB": (b, T, R, G, N),
              "dC": (b, T, R, G, N), "dgamma": (b, T, H), "dbeta": (b, T, H),
              "dtheta": (b, T, H, N // 2) if theta is not None else None,
              "dinit": (b, H, P, N),
              "dprev_x": (b, R, H, P) if prev_x is not None else None,
              "dprev_B": (b, R, G, N) if prev_x is not None else None}
    g = {}
    for k, shp in shapes.items():
        given = (grads or {}).get(k)
        if shp is None:
            g[k] = None
        elif given is not None:
            _check_cuda(k, given, torch.float32, shp)
            g[k] = given
        else:
            g[k] = torch.empty(shp, dtype=torch.float32, device=x.device)
    st = lib.ssd_trapezoidal_backward(
        ctypes.byref(shape), _ptr(x), _ptr(dA), _ptr(B), _ptr(C), _ptr(gamma), _ptr(beta),
        _ptr(theta), _ptr(prev_x), _ptr(prev_B), _ptr(init_state), _ptr(dy), _ptr(dfinal),
        _ptr(g["dx"]), _ptr(g["ddA"]), _ptr(g["dB"]), _ptr(g["dC"]), _ptr(g["dgamma"]),
        _ptr(g["dbeta"]), _ptr(g["dtheta"]), _ptr(g["dinit"]), _ptr(g["dprev_x"]),
        _ptr(g["dprev_B"]), _ptr(workspace), ctypes.c_size_t(workspace.numel()),
        _stream_handle(stream))
    if st != 0:
        raise SSDError(st, "ssd_trapezoidal_backward")
    g["workspace"] = workspace
    return g


def selective_scan_workspace_bytes(batch, seqlen, d_model, d_state) -> int:
    return int(load_library().selective_scan_workspace_bytes(batch, seqlen, d_model, d_state))


class SelectiveScanPlan:
    """Arguments of ``selective_scan_forward`` validated once, for repeated calls on the same
    buffers; calling the plan makes only the C call (stream fixed at construction)."""

    def __init__(self, u, delta, A, B, C, skip=None, *, y=None, workspace=None, stream=None):
        b, T, D = u.shape
        N = A.shape[1]
        f32 = torch.float32
        _check_cuda("u", u, f32)
        _check_cuda("delta", delta, f32, (b, T, D))
        _check_cuda("A", A, f32, (D, N))
        _check_cuda("B", B, f32, (b, T, N))
        _check_cuda("C", C, f32, (b, T, N))
        if skip is not None:
            _check_cuda("skip", skip, f32, (D,))
        self._lib = load_library()
        if y is None:
            y = torch.empty_like(u)
        _check_cuda("y", y, f32, (b, T, D))
        need = int(self._lib.selective_scan_workspace_bytes(b, T, D, N))
        if need == 0:
            raise SSDError(2, "selective_scan_workspace_bytes (sizes not supported)")
        if workspace is None:
            workspace = torch.zeros(need, dtype=torch.uint8, device=u.device)   # zero header
        _check_cuda("workspace", workspace, torch.uint8)
        self.inputs = (u, delta, A, B, C, skip)
        self.y, self.workspace = y, workspace
        self._args = (_ptr(u), _ptr(delta), _ptr(A), _ptr(B), _ptr(C), _ptr(skip), _ptr(y), b, T,
                      D, N, _ptr(workspace), ctypes.c_size_t(workspace.numel()),
                      _stream_handle(stream))
        self._fn = self._lib.selective_scan_forward

    def __call__(self):
        st = self._fn(*self._args)
        if st != 0:
            raise SSDError(st, "selective_scan_forward")
        return self.y


def selective_scan_forward(u, delta, A, B, C, skip=None, *, y=None, workspace=None, stream=None):
    """Diagonal-A selective scan through ``selective_scan_forward`` (all f32).  Returns y."""
    return SelectiveScanPlan(u, delta, A, B, C, skip, y=y, workspace=workspace, stream=stream)()


def wait_selftest(workspace: torch.Tensor, wait_ns: int, stream=None) -> None:
    """Runs the bounded-wait self-test (``ssd_wait_selftest``): a device wait that nothing
    satisfies gives up after ``wait_ns`` and latches SSD_ERR_TIMEOUT in ``workspace``."""
    _check_cuda("workspace", workspace, torch.uint8)
    st = load_library().ssd_wait_selftest(_ptr(workspace), ctypes.c_size_t(workspace.numel()),
                                          ctypes.c_uint64(int(wait_ns)), _stream_handle(stream))
    if st != 0:
        raise SSDError(st, "ssd_wait_selftest")


def workspace_status(workspace: torch.Tensor, stream=None):
    """(status name, detail) of the device-side error word of ``workspace`` (syncs the stream)."""
    detail = ctypes.c_int64(0)
    st = load_library().ssd_workspace_status(_ptr(workspace), _stream_handle(stream),
                                             ctypes.byref(detail))
    return STATUS.get(int(st), str(st)), int(detail.value)

"""fp64 CPU oracle for the chunked SSD scan and the selective scan.

TEST INFRASTRUCTURE ONLY: imported by the test suite, by the smoke check and by the benchmark's
CPU-baseline leg, never by the library.  It shares no code with the CUDA path.

- ``ssd`` / ``ssd_trapezoidal`` / ``selective_scan`` call the plain sequential recurrences in
  ``ssd_oracle.c`` (C, fp64, threads over independent problems).  These are the oracle proper.
- ``chunked_ref`` (numpy, fp64) restates the serial.rs page's K1..K5 chunk decomposition, the
  segsum.rs page's stable segment sum, and the scan.py page's cumulative-angle rotation.  It is
  not an oracle for the GPU; the pin tests use it to check the sequential oracle against the
  pages' own algebra (chunk invariance, rotation absorption).

Inputs are numpy arrays (any float dtype; they are upcast to float64) in the library's layouts:
    x  [b,T,R,H,P]   dA [b,T,H]   B, C [b,T,R,G,N]   theta [b,T,H,N/2]   init [b,H,P,N]
    u, delta [b,T,D] A [D,N]      B, C [b,T,N]       skip [D]
    gamma, beta [b,T,H]   prev_x [b,R,H,P]   prev_B [b,R,G,N]        (trapezoidal form)
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ssd_oracle.c")
_SO = os.path.join(_HERE, "libssd_oracle.so")
_LIB = None

_D = ctypes.POINTER(ctypes.c_double)
_I64 = ctypes.c_int64


def build(force: bool = False) -> str:
    """Compile ssd_oracle.c into libssd_oracle.so next to it (plain gcc, no CPU-specific flags)."""
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        tmp = _SO + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared", "-o", tmp, _SRC,
             "-lm", "-lpthread"])
        os.replace(tmp, _SO)
    return _SO


def _lib():
    global _LIB
    if _LIB is None:
        lib = ctypes.CDLL(build())
        lib.oracle_ssd_ex.restype = ctypes.c_int
        lib.oracle_ssd_ex.argtypes = [_D] * 8 + [_I64] * 8 + [ctypes.c_int]
        lib.oracle_ssd_backward_ex.restype = ctypes.c_int
        lib.oracle_ssd_backward_ex.argtypes = [_D] * 14 + [_I64] * 8 + [ctypes.c_int]
        lib.oracle_ssd_trap_backward_ex.restype = ctypes.c_int
        lib.oracle_ssd_trap_backward_ex.argtypes = [_D] * 22 + [_I64] * 8 + [ctypes.c_int]
        lib.oracle_ssd_rot_ex.restype = ctypes.c_int
        lib.oracle_ssd_rot_ex.argtypes = [_D] * 8 + [_I64] * 8 + [ctypes.c_int, _I64, ctypes.c_int]
        lib.oracle_ssd_quat_ex.restype = ctypes.c_int
        lib.oracle_ssd_quat_ex.argtypes = [_D] * 8 + [_I64] * 8 + [ctypes.c_int]
        lib.oracle_ssd_trap_ex.restype = ctypes.c_int
        lib.oracle_ssd_trap_ex.argtypes = [_D] * 12 + [_I64] * 8 + [ctypes.c_int]
        lib.oracle_selective_scan_ex.restype = ctypes.c_int
        lib.oracle_selective_scan_ex.argtypes = [_D] * 7 + [_I64] * 5 + [ctypes.c_int]
        _LIB = lib
    return _LIB


def _f64(a):
    if a is None:
        return None
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _ptr(a):
    if a is None:
        return ctypes.cast(None, _D)
    return a.ctypes.data_as(_D)


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


def ssd(x, dA, B, C, theta=None, init_state=None, nthreads=None, mutation: int = 0):
    """Sequential fp64 SSD recurrence.  Returns (y [b,T,R,H,P], final_state [b,H,P,N])."""
    x, dA, B, C = _f64(x), _f64(dA), _f64(B), _f64(C)
    theta, init_state = _f64(theta), _f64(init_state)
    b, T, R, H, P = x.shape
    G, N = B.shape[3], B.shape[4]
    assert dA.shape == (b, T, H)
    assert B.shape == (b, T, R, G, N) and C.shape == B.shape
    if theta is not None:
        assert theta.shape == (b, T, H, N // 2)
    if init_state is not None:
        assert init_state.shape == (b, H, P, N)
    y = np.zeros((b, T, R, H, P), np.float64)
    fin = np.zeros((b, H, P, N), np.float64)
    rc = _lib().oracle_ssd_ex(_ptr(x), _ptr(dA), _ptr(B), _ptr(C), _ptr(theta), _ptr(init_state),
                              _ptr(y), _ptr(fin), b, T, R, H, G, P, N,
                              nthreads or default_threads(), int(mutation))
    if rc != 0:
        raise ValueError(f"oracle_ssd rejected its arguments (code {rc})")
    return y, fin


def ssd_backward(x, dA, B, C, dy, init_state=None, dfinal=None, theta=None, nthreads=None,
                 mutation: int = 0):
    """Reverse mode of the SSD recurrence (rotated when theta [b,T,H,N/2] is given, interleaved
    pairs) for the loss <dy, y> + <dfinal, final>.  Returns dict dx [b,T,R,H,P], ddA [b,T,H],
    dB, dC [b,T,R,G,N], dinit [b,H,P,N] and, with theta, dtheta [b,T,H,N/2]."""
    x, dA, B, C, dy = (_f64(v) for v in (x, dA, B, C, dy))
    init_state, dfinal, theta = _f64(init_state), _f64(dfinal), _f64(theta)
    b, T, R, H, P = x.shape
    G, N = B.shape[3], B.shape[4]
    assert dy.shape == x.shape
    if theta is not None:
        assert theta.shape == (b, T, H, N // 2)
    out = {"dx": np.zeros_like(x), "ddA": np.zeros_like(dA), "dB": np.zeros_like(B),
           "dC": np.zeros_like(C), "dinit": np.zeros((b, H, P, N))}
    if theta is not None:
        out["dtheta"] = np.zeros_like(theta)
    rc = _lib().oracle_ssd_backward_ex(_ptr(x), _ptr(dA), _ptr(B), _ptr(C), _ptr(theta),
                                       _ptr(init_state), _ptr(dy), _ptr(dfinal), _ptr(out["dx"]),
                                       _ptr(out["ddA"]), _ptr(out["dB"]), _ptr(out["dC"]),
                                       _ptr(out.get("dtheta")), _ptr(out["dinit"]),
                                       b, T, R, H, G, P, N, nthreads or default_threads(),
                                       int(mutation))
    if rc != 0:
        raise ValueError(f"oracle_ssd_backward rejected its arguments (code {rc})")
    return out


def ssd_trap_backward(x, dA, B, C, gamma, beta, dy, theta=None, init_state=None, prev_x=None,
                      prev_B=None, dfinal=None, nthreads=None, mutation: int = 0):
    """Reverse mode of the trapezoidal SSD recurrence (see ssd_oracle.c) for the loss
    <dy, y> + <dfinal, final>.  Returns dict dx, ddA, dB, dC, dgamma, dbeta, dinit and, when
    given theta / prev_x and prev_B, dtheta / dprev_x and dprev_B."""
    x, dA, B, C, gamma, beta, dy = (_f64(v) for v in (x, dA, B, C, gamma, beta, dy))
    theta, init_state, prev_x, prev_B, dfinal = (_f64(v) for v in
                                                 (theta, init_state, prev_x, prev_B, dfinal))
    b, T, R, H, P = x.shape
    G, N = B.shape[3], B.shape[4]
    assert dy.shape == x.shape and gamma.shape == (b, T, H) and beta.shape == (b, T, H)
    out = {"dx": np.zeros_like(x), "ddA": np.zeros_like(dA), "dB": np.zeros_like(B),
           "dC": np.zeros_like(C), "dgamma": np.zeros_like(gamma), "dbeta": np.zeros_like(beta),
           "dinit": np.zeros((b, H, P, N))}
    if theta is not None:
        assert theta.shape == (b, T, H, N // 2)
        out["dtheta"] = np.zeros_like(theta)
    if prev_x is not None:
        out["dprev_x"] = np.zeros_like(prev_x)
        out["dprev_B"] = np.zeros_like(prev_B)
    rc = _lib().oracle_ssd_trap_backward_ex(
        _ptr(x), _ptr(dA), _ptr(B), _ptr(C), _ptr(gamma), _ptr(beta), _ptr(theta),
        _ptr(init_state), _ptr(prev_x), _ptr(prev_B), _ptr(dy), _ptr(dfinal), _ptr(out["dx"]),
        _ptr(out["ddA"]), _ptr(out["dB"]), _ptr(out["dC"]), _ptr(out["dgamma"]),
        _ptr(out["dbeta"]), _ptr(out.get("dtheta")), _ptr(out["dinit"]), _ptr(out.get("dprev_x")),
        _ptr(out.get("dprev_B")), b, T, R, H, G, P, N, nthreads or default_threads(),
        int(mutation))
    if rc != 0:
        raise ValueError(f"oracle_ssd_trap_backward rejected its arguments (code {rc})")
    return out


def ssd_rotation_variant(x, dA, B, C, theta, init_state=None, rope_dim: int = 0,
                         halves: bool = False, nthreads=None, mutation: int = 0):
    """Sequential fp64 SSD recurrence whose rotation turns only the first rope_dim state dims
    (0 = all), pairing (2k, 2k+1) or, with halves, (k, k + rope_dim/2); theta [b,T,H,rope_dim/2].
    Returns (y, final_state)."""
    x, dA, B, C, theta, init_state = (_f64(v) for v in (x, dA, B, C, theta, init_state))
    b, T, R, H, P = x.shape
    G, N = B.shape[3], B.shape[4]
    rd = rope_dim or N
    assert theta.shape == (b, T, H, rd // 2)
    y = np.zeros((b, T, R, H, P), np.float64)
    fin = np.zeros((b, H, P, N), np.float64)
    rc = _lib().oracle_ssd_rot_ex(_ptr(x), _ptr(dA), _ptr(B), _ptr(C), _ptr(theta),
                                  _ptr(init_state), _ptr(y), _ptr(fin), b, T, R, H, G, P, N,
                                  int(rope_dim), int(bool(halves)), nthreads or default_threads(),
                                  int(mutation))
    if rc != 0:
        raise ValueError(f"oracle_ssd_rot rejected its arguments (code {rc})")
    return y, fin


def ssd_quaternion(x, dA, B, C, qcum, init_state=None, nthreads=None, mutation: int = 0):
    """Sequential fp64 SSD recurrence with the quaternion rotation (see ssd_oracle.c): qcum
    [b,T,H,N/4,4] cumulative unit quaternions (w, x, y, z); block j of the state is turned by
    left multiplication with qcum_t qcum_{t-1}^* before the write.  Returns (y, final_state)."""
    x, dA, B, C, qcum, init_state = (_f64(v) for v in (x, dA, B, C, qcum, init_state))
    b, T, R, H, P = x.shape
    G, N = B.shape[3], B.shape[4]
    assert N % 4 == 0 and qcum.shape == (b, T, H, N // 4, 4)
    y = np.zeros((b, T, R, H, P), np.float64)
    fin = np.zeros((b, H, P, N), np.float64)
    rc = _lib().oracle_ssd_quat_ex(_ptr(x), _ptr(dA), _ptr(B), _ptr(C), _ptr(qcum),
                                   _ptr(init_state), _ptr(y), _ptr(fin), b, T, R, H, G, P, N,
                                   nthreads or default_threads(), int(mutation))
    if rc != 0:
        raise ValueError(f"oracle_ssd_quat rejected its arguments (code {rc})")
    return y, fin


def ssd_trapezoidal(x, dA, B, C, gamma, beta, theta=None, init_state=None, prev_x=None,
                    prev_B=None, nthreads=None, mutation: int = 0):
    """Sequential fp64 trapezoidal SSD recurrence (see ssd_oracle.c).  Returns (y, final_state)."""
    x, dA, B, C, gamma, beta = (_f64(v) for v in (x, dA, B, C, gamma, beta))
    theta, init_state, prev_x, prev_B = (_f64(v) for v in (theta, init_state, prev_x, prev_B))
    b, T, R, H, P = x.shape
    G, N = B.shape[3], B.shape[4]
    assert dA.shape == (b, T, H) and gamma.shape == (b, T, H) and beta.shape == (b, T, H)
    assert B.shape == (b, T, R, G, N) and C.shape == B.shape
    if theta is not None:
        assert theta.shape == (b, T, H, N // 2)
    if init_state is not None:
        assert init_state.shape == (b, H, P, N)
    if prev_x is not None or prev_B is not None:
        assert prev_x.shape == (b, R, H, P) and prev_B.shape == (b, R, G, N)
    y = np.zeros((b, T, R, H, P), np.float64)
    fin = np.zeros((b, H, P, N), np.float64)
    rc = _lib().oracle_ssd_trap_ex(_ptr(x), _ptr(dA), _ptr(B), _ptr(C), _ptr(gamma), _ptr(beta),
                                   _ptr(theta), _ptr(init_state), _ptr(prev_x), _ptr(prev_B),
                                   _ptr(y), _ptr(fin), b, T, R, H, G, P, N,
                                   nthreads or default_threads(), int(mutation))
    if rc != 0:
        raise ValueError(f"oracle_ssd_trap rejected its arguments (code {rc})")
    return y, fin


def selective_scan(u, delta, A, B, C, skip=None, nthreads=None, mutation: int = 0):
    """Sequential fp64 selective scan.  Returns y [b,T,D]."""
    u, delta, A, B, C, skip = (_f64(v) for v in (u, delta, A, B, C, skip))
    b, T, D = u.shape
    N = A.shape[1]
    assert delta.shape == u.shape and A.shape == (D, N)
    assert B.shape == (b, T, N) and C.shape == B.shape
    if skip is not None:
        assert skip.shape == (D,)
    y = np.zeros((b, T, D), np.float64)
    rc = _lib().oracle_selective_scan_ex(_ptr(u), _ptr(delta), _ptr(A), _ptr(B), _ptr(C),
                                         _ptr(skip), _ptr(y), b, T, D, N,
                                         nthreads or default_threads(), int(mutation))
    if rc != 0:
        raise ValueError(f"oracle_selective_scan rejected its arguments (code {rc})")
    return y


# Planted-mistake codes understood by the C oracle (used only by the pin tests).
MUTATIONS_SSD = {
    "no_decay": 1,
    "decay_after_write": 2,
    "swap_B_C": 3,
    "rank_local_output": 4,
    "rotation_sign": 5,
    "group_index": 6,
}
MUTATIONS_TRAP = {
    "no_beta": 9,
    "beta_turned_late": 10,
    "beta_on_current_write": 11,
}
MUTATIONS_ROT = {
    "interleaved_instead_of_halves": 12,
    "rope_on_last_dims": 13,
}
MUTATIONS_QUAT = {
    "quaternion_right_multiplication": 20,
    "cumulative_quaternion_as_step": 21,
}
MUTATIONS_BWD = {
    "dy_added_after_decay": 14,
    "ddA_without_decay_factor": 15,
    "state_gradient_turned_forward": 16,
}
MUTATIONS_TRAP_BWD = {
    "beta_gradient_not_carried": 17,
}
MUTATIONS_SS = {
    "no_skip": 7,
    "no_delta_on_B": 8,
}

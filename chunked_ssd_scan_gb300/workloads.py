"""Seeded synthetic inputs for the SSD scan and the selective scan.

This module only draws random numbers in the shapes, dtypes and distributions of the workloads;
it holds none of the scan's arithmetic.  Tests and the benchmark feed the same tensors to the
CUDA library and to the CPU oracle.

Recipe (one torch CPU ``Generator`` per call, seeded):
- SSD draw order x, B, C, dt, A_h, theta, init_state; all drawn in fp32 and then cast to the
  I/O dtype (x, B, C, y share it; dA, theta and the states stay fp32).
    x ~ N(0,1) * x_scale;  B, C ~ N(0,1) * bc_scale
    dt = softplus(N(0,1) - 2)  [b,T,H];  A_h = -exp(U(0, ln 16))  [H];  dA = dt * A_h
    "slow decay" variant: dA = -U(0, 0.01)  (so the chunk-to-chunk state carry stays visible)
    theta ~ U(-0.1, 0.1)  [b,T,H,N/2];  init_state ~ N(0,1)  [b,H,P,N] when requested
- Trapezoidal form (make_trap_inputs): the SSD draws above, then from a second generator
  (seed + 104729) lam, s, prev_x, prev_B:
    lam = sigmoid(N(0,1)), s = softplus(N(0,1) - 2)  [b,T,H];
    gamma = lam * s;  beta = (1 - lam) * s * exp(dA)   (the generalised trapezoid's weights);
    prev_x ~ N(0,1) * x_scale [b,R,H,P], prev_B ~ N(0,1) * bc_scale [b,R,G,N] when requested
- Selective scan draw order u, delta, A, B, C, skip:
    u ~ N(0,1);  delta = softplus(N(0,1));  A = -U(0.5, 2)  [D,N];  B, C ~ N(0,1)  [b,T,N];
    skip ~ N(0,1)  [D]
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import torch


@dataclasses.dataclass(frozen=True)
class SSDConfig:
    name: str
    batch: int
    seqlen: int
    nheads: int
    headdim: int
    dstate: int
    chunk_len: int
    mimo_rank: int
    ngroups: int
    dtype: str            # "f32" or "bf16": the dtype of x, B, C and y
    theta: bool = False
    x_scale: float = 1.0
    bc_scale: float = 1.0
    trapezoidal: bool = False   # the trapezoidal form (gamma, beta and the previous write)
    rope_dim: int = 0           # rotation variant: rotated state dims (0 = all of dstate)
    halves: bool = False        # rotation variant: split-halves pairing
    backward: bool = False      # the reverse mode (dy, dfinal in; dx, ddA, dB, dC, dinit out)

    @property
    def torch_dtype(self) -> torch.dtype:
        return torch.float32 if self.dtype == "f32" else torch.bfloat16

    @property
    def tokens(self) -> int:
        """Tokens per call: one per (batch, time step); MIMO ranks do not multiply it."""
        return self.batch * self.seqlen

    def with_(self, **kw) -> "SSDConfig":
        return dataclasses.replace(self, **kw)

    def io_bytes(self) -> int:
        """Algorithmic HBM bytes: every input read once and every output written once."""
        e = 4 if self.dtype == "f32" else 2
        b, T, R, H, P, N, G = (self.batch, self.seqlen, self.mimo_rank, self.nheads, self.headdim,
                               self.dstate, self.ngroups)
        if self.backward:   # inputs x, B, C, dA, dy, init, dfinal; f32 gradients out
            nbytes = b * T * R * H * P * (e + 4 + 4)     # x, dy read, dx written
            nbytes += b * T * R * G * N * (e + 4) * 2    # B, C read, dB, dC written
            nbytes += b * T * H * 4 * 2                  # dA read, ddA written
            nbytes += b * H * P * N * 4 * 3              # init, dfinal read, dinit written
            if self.theta:
                nbytes += b * T * H * (N // 2) * 4 * 2   # theta read, dtheta written
            if self.trapezoidal:
                nbytes += b * T * H * 4 * 4              # gamma, beta read; dgamma, dbeta written
                nbytes += b * R * (H * P + G * N) * (e + 4)   # previous write read, its grads
            return nbytes
        nbytes = b * T * R * H * P * e * 2          # x read, y written
        nbytes += b * T * R * G * N * e * 2         # B, C read
        nbytes += b * T * H * 4                     # dA read
        nbytes += b * H * P * N * 4                 # final state written
        if self.theta:
            nbytes += b * T * H * ((self.rope_dim or N) // 2) * 4   # theta read
        if self.trapezoidal:
            nbytes += 2 * b * T * H * 4             # gamma, beta read
            nbytes += b * R * (H * P + G * N) * e   # previous write read
        return nbytes

    def causal_flops(self) -> int:
        """Contraction FLOPs of the chunked method, counting only the causal part of each chunk."""
        b, T, R, H, P, N, G, l = (self.batch, self.seqlen, self.mimo_rank, self.nheads,
                                  self.headdim, self.dstate, self.ngroups, self.chunk_len)
        nch = -(-T // l)
        L = l * R
        pairs = R * R * l * (l + 1) // 2                     # causal (i, j) pairs per chunk
        cb = 2 * pairs * N * b * nch * G                     # K2, once per B/C group
        diag = 2 * pairs * P * b * nch * H                   # K5 intra-chunk
        state = 2 * P * N * L * b * nch * H                  # K3
        off = 2 * L * N * P * b * nch * H                    # K5 inter-chunk
        return cb + diag + state + off

    def backward_flops(self) -> int:
        """FLOPs of the chunked backward at 64 fused rows per chunk (64 / R steps), causal part
        only: the chunk-state recompute and dL/dh_in contribution (2 P N L each), the pairwise
        C.B (per group) and dy.x products, and dx, dB, dC (each a causal pairwise sum plus a
        P x N state product per row)."""
        b, T, R, H, P, N, G = (self.batch, self.seqlen, self.mimo_rank, self.nheads,
                               self.headdim, self.dstate, self.ngroups)
        l = max(1, 64 // R)
        nch = -(-T // l)
        L = l * R
        pairs = R * R * l * (l + 1) // 2
        per_head = (2 * 2 * P * N * L            # state recompute, D_c
                    + 2 * pairs * P              # dy_i . x_j
                    + 2 * pairs * P + 2 * L * N * P    # dx
                    + 2 * pairs * N + 2 * L * P * N    # dB
                    + 2 * pairs * N + 2 * L * P * N)   # dC
        return b * nch * (H * per_head + G * 2 * pairs * N)


@dataclasses.dataclass(frozen=True)
class SelectiveScanConfig:
    name: str
    batch: int
    seqlen: int
    d_model: int
    d_state: int

    @property
    def tokens(self) -> int:
        return self.batch * self.seqlen

    def io_bytes(self) -> int:
        b, T, D, N = self.batch, self.seqlen, self.d_model, self.d_state
        return 4 * (3 * b * T * D + 2 * b * T * N + D * N + D)

    def with_(self, **kw) -> "SelectiveScanConfig":
        return dataclasses.replace(self, **kw)


# The five workloads: four SSD problems and one selective scan.
TINY_SISO_F32 = SSDConfig("tiny_siso_f32", 1, 256, 2, 16, 16, 64, 1, 2, "f32")
MAMBA2_SISO_BF16 = SSDConfig("mamba2_siso_bf16", 4, 4096, 32, 64, 128, 256, 1, 1, "bf16")
MAMBA3_MIMO_BF16 = SSDConfig("mamba3_mimo_bf16", 2, 8192, 32, 64, 128, 64, 4, 32, "bf16",
                             bc_scale=1.0 / math.sqrt(128))
LONG_ROT_F32 = SSDConfig("long_rotation_f32", 1, 131072, 24, 64, 64, 256, 1, 24, "f32",
                         theta=True)
SELECTIVE_SCAN_F32 = SelectiveScanConfig("selective_scan_f32", 4, 4096, 512, 16)
# Rotation variant: the long-rotation shape (24 heads, P = N = 64) at T = 32768 with half of the
# state rotated and the split-halves pairing; a measured shape, not one of the five workloads.
ROT_VARIANT_F32 = SSDConfig("rotation_halves_rope32_f32", 1, 32768, 24, 64, 64, 256, 1, 24,
                            "f32", theta=True, rope_dim=32, halves=True)
# Trapezoidal Mamba-3 (T = 16384, 16 heads, P = N = 64, R = 2, rotation); a measured shape, not
# one of the five workloads.
TRAP_MIMO_ROT_F32 = SSDConfig("mamba3_trapezoidal_f32", 1, 16384, 16, 64, 64, 64, 2, 16, "f32",
                              theta=True, trapezoidal=True)

# Backward of the unrotated SSD on the Mamba-2 SISO shape (4 x 4096 steps, 32 heads, P = 64,
# N = 128, bf16 inputs).
MAMBA2_BWD_BF16 = SSDConfig("mamba2_backward_bf16", 4, 4096, 32, 64, 128, 64, 1, 1, "bf16",
                            backward=True)
# Trapezoidal backward on the trapezoidal forward's shape above.
TRAP_BWD_F32 = SSDConfig("mamba3_trapezoidal_backward_f32", 1, 16384, 16, 64, 64, 64, 2, 16,
                         "f32", theta=True, trapezoidal=True, backward=True)
# Rotated backward on the long-rotation shape (T = 131072, 24 heads, P = N = 64, f32).
LONG_ROT_BWD_F32 = SSDConfig("long_rotation_backward_f32", 1, 131072, 24, 64, 64, 256, 1, 24,
                             "f32", theta=True, backward=True)

SSD_CONFIGS = [TINY_SISO_F32, MAMBA2_SISO_BF16, MAMBA3_MIMO_BF16, LONG_ROT_F32]


def make_ssd_inputs(cfg: SSDConfig, seed: int = 0, *, slow_decay: bool = False,
                    init_state: bool = False, device: Optional[str] = None) -> dict:
    """Draw one problem for ``cfg`` on the CPU (then optionally move it to ``device``)."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    b, T, R, H, P, N, G = (cfg.batch, cfg.seqlen, cfg.mimo_rank, cfg.nheads, cfg.headdim,
                           cfg.dstate, cfg.ngroups)
    f32 = torch.float32
    x = torch.randn((b, T, R, H, P), generator=g, dtype=f32)
    if cfg.x_scale != 1.0:
        x.mul_(cfg.x_scale)
    B = torch.randn((b, T, R, G, N), generator=g, dtype=f32)
    C = torch.randn((b, T, R, G, N), generator=g, dtype=f32)
    if cfg.bc_scale != 1.0:
        B.mul_(cfg.bc_scale)
        C.mul_(cfg.bc_scale)
    dt = torch.nn.functional.softplus(torch.randn((b, T, H), generator=g, dtype=f32) - 2.0)
    A_h = -torch.exp(torch.rand((H,), generator=g, dtype=f32) * math.log(16.0))
    if slow_decay:
        dA = -torch.rand((b, T, H), generator=g, dtype=f32) * 0.01
    else:
        dA = dt * A_h
    theta = None
    if cfg.theta:
        theta = (torch.rand((b, T, H, (cfg.rope_dim or N) // 2), generator=g, dtype=f32) * 0.2
                 - 0.1)
    init = torch.randn((b, H, P, N), generator=g, dtype=f32) if init_state else None
    out = {
        "x": x.to(cfg.torch_dtype),
        "dA": dA.contiguous(),
        "B": B.to(cfg.torch_dtype),
        "C": C.to(cfg.torch_dtype),
        "theta": theta,
        "init_state": init,
    }
    if device is not None:
        out = {k: (v.to(device) if v is not None else None) for k, v in out.items()}
    return out


def make_quaternions(batch: int, T: int, H: int, N: int, seed: int = 0,
                     step: float = 0.05) -> torch.Tensor:
    """Cumulative unit quaternions [batch, T, H, N/4, 4] (w, x, y, z) for the quaternion
    rotation: a normalised random walk in R^4 started at the identity, so consecutive steps
    differ by small turns (the per-step turn of a step is a few times `step` radians)."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    u = torch.randn((batch, T, H, N // 4, 4), generator=g, dtype=torch.float64) * step
    u = torch.cumsum(u, dim=1)
    u[..., 0] += 1.0
    return (u / torch.linalg.vector_norm(u, dim=-1, keepdim=True)).to(torch.float32).contiguous()


def make_trap_inputs(cfg: SSDConfig, seed: int = 0, *, slow_decay: bool = False,
                     init_state: bool = False, prev: bool = True,
                     device: Optional[str] = None) -> dict:
    """make_ssd_inputs plus gamma, beta and (optionally) the previous step's x and B."""
    out = make_ssd_inputs(cfg, seed, slow_decay=slow_decay, init_state=init_state)
    g = torch.Generator(device="cpu")
    g.manual_seed(seed + 104729)
    b, T, R, H, P, N, G = (cfg.batch, cfg.seqlen, cfg.mimo_rank, cfg.nheads, cfg.headdim,
                           cfg.dstate, cfg.ngroups)
    f32 = torch.float32
    lam = torch.sigmoid(torch.randn((b, T, H), generator=g, dtype=f32))
    sc = torch.nn.functional.softplus(torch.randn((b, T, H), generator=g, dtype=f32) - 2.0)
    out["gamma"] = (lam * sc).contiguous()
    out["beta"] = ((1.0 - lam) * sc * torch.exp(out["dA"])).contiguous()
    out["prev_x"] = out["prev_B"] = None
    if prev:
        out["prev_x"] = (torch.randn((b, R, H, P), generator=g, dtype=f32) * cfg.x_scale
                         ).to(cfg.torch_dtype)
        out["prev_B"] = (torch.randn((b, R, G, N), generator=g, dtype=f32) * cfg.bc_scale
                         ).to(cfg.torch_dtype)
    if device is not None:
        out = {k: (v.to(device) if v is not None else None) for k, v in out.items()}
    return out


def make_trap_bwd_inputs(cfg: SSDConfig, seed: int = 0, *,
                         device: Optional[str] = None) -> dict:
    """A trapezoidal forward problem (initial state, previous write) plus the cotangents dy and
    dfinal (standard normal f32, from a third generator) for its backward."""
    out = make_trap_inputs(cfg, seed, init_state=True, prev=True)
    g = torch.Generator(device="cpu")
    g.manual_seed(seed + 7919)
    b, T, R, H, P, N = cfg.batch, cfg.seqlen, cfg.mimo_rank, cfg.nheads, cfg.headdim, cfg.dstate
    out["dy"] = torch.randn((b, T, R, H, P), generator=g, dtype=torch.float32)
    out["dfinal"] = torch.randn((b, H, P, N), generator=g, dtype=torch.float32)
    if device is not None:
        out = {k: (v.to(device) if v is not None else None) for k, v in out.items()}
    return out


def make_bwd_inputs(cfg: SSDConfig, seed: int = 0, *, device: Optional[str] = None) -> dict:
    """A forward problem (with an initial state) plus the cotangents dy [b,T,R,H,P] and dfinal
    [b,H,P,N] (standard normal f32, from a second generator) for the backward."""
    out = make_ssd_inputs(cfg, seed, init_state=True)
    g = torch.Generator(device="cpu")
    g.manual_seed(seed + 7919)
    b, T, R, H, P, N = cfg.batch, cfg.seqlen, cfg.mimo_rank, cfg.nheads, cfg.headdim, cfg.dstate
    out["dy"] = torch.randn((b, T, R, H, P), generator=g, dtype=torch.float32)
    out["dfinal"] = torch.randn((b, H, P, N), generator=g, dtype=torch.float32)
    if device is not None:
        out = {k: (v.to(device) if v is not None else None) for k, v in out.items()}
    return out


def make_selective_scan_inputs(cfg: SelectiveScanConfig, seed: int = 0,
                               device: Optional[str] = None) -> dict:
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    b, T, D, N = cfg.batch, cfg.seqlen, cfg.d_model, cfg.d_state
    f32 = torch.float32
    u = torch.randn((b, T, D), generator=g, dtype=f32)
    delta = torch.nn.functional.softplus(torch.randn((b, T, D), generator=g, dtype=f32))
    A = -(torch.rand((D, N), generator=g, dtype=f32) * 1.5 + 0.5)
    B = torch.randn((b, T, N), generator=g, dtype=f32)
    C = torch.randn((b, T, N), generator=g, dtype=f32)
    skip = torch.randn((D,), generator=g, dtype=f32)
    out = {"u": u, "delta": delta, "A": A, "B": B, "C": C, "skip": skip}
    if device is not None:
        out = {k: v.to(device) for k, v in out.items()}
    return out

"""numpy fp64 restatement of the pages' chunked algorithm (TEST INFRASTRUCTURE ONLY).

This is the algebra the GPU kernels are built on, written step by step in the pages' order so
that the pin tests can check the sequential oracle (``oracle.ssd``) against it:

- ``segsum``: the segsum.rs page (burn_mamba modules/misc/segsum.rs), ``segsum`` doc comment:
  out[..., i, j] = cumsum(x)[i] - cumsum(x)[j] for i >= j, -inf above the diagonal, so that
  exp(segsum) is the causal 1-semiseparable decay mask.
- ``k1_chunk_cumsum`` .. ``k5_chunk_scan``: the serial.rs page (burn_mamba mamba3/ssd/serial.rs),
  functions k1_ssd_chunk_cumsum, k2_ssd_bmm, k3_ssd_chunk_state, k4_ssd_state_passing,
  k5_ssd_chunk_scan, on rank-fused tensors (fused index i = t*R + r, time-major).
- ``rotate_pairs`` / cumulative angles: the scan.py page (steertts mamba3/scan.py),
  cumulative_angles and rotate_by; the rotation is absorbed as B~ = R(-Phi_t) B, C~ = R(-Phi_t) C
  and the final state is turned back by R(Phi_{T-1}) (module docstring, "THE TRICK").
- Ragged T: zero padding with dA = 0 and x = 0 (moments.rs page, module header: pads are
  identity decay and zero write, so the carried state passes through unchanged).
- ``chunked_backward`` / ``chunked_backward_rotated`` / ``trapezoidal_backward_expanded``: the
  chain rule through that decomposition (and through the trapezoid's 2R-channel expansion) (the pages ask for a trainable scan but print no backward formulas), per chunk,
  plain and in chunk-local rotation frames, so the pins can check the sequential reverse mode
  (``oracle.ssd_backward``) against the chunked algebra the GPU backward is built on.

It is deliberately unfused and unblocked: every intermediate of the pages is materialised.
"""
from __future__ import annotations

import numpy as np


def segsum(x: np.ndarray) -> np.ndarray:
    """[..., T] -> [..., T, T]; lower triangle = sum_{k=j+1..i} x_k, strict upper = -inf."""
    T = x.shape[-1]
    cs = np.cumsum(x, axis=-1)
    out = cs[..., :, None] - cs[..., None, :]
    upper = np.triu(np.ones((T, T), dtype=bool), k=1)
    out = np.where(upper, -np.inf, out)
    return out


def rotate_pairs(v: np.ndarray, ang: np.ndarray) -> np.ndarray:
    """Turn interleaved pairs (v[...,2k], v[...,2k+1]) of the last axis by +ang[...,k]."""
    a, b = v[..., 0::2], v[..., 1::2]
    c, s = np.cos(ang), np.sin(ang)
    out = np.empty_like(v)
    out[..., 0::2] = c * a - s * b
    out[..., 1::2] = s * a + c * b
    return out


def k1_chunk_cumsum(da_bnlh: np.ndarray):
    """K1: intra-chunk prefix sums [b,H,n,l] and the per-chunk totals [b,H,n]."""
    cum = np.cumsum(np.transpose(da_bnlh, (0, 3, 1, 2)), axis=3)
    return cum, cum[..., -1]


def k2_bmm(c_bnLhn: np.ndarray, b_bnLhn: np.ndarray) -> np.ndarray:
    """K2: CB[b,n,h,i,j] = sum_s C[i,s] B[j,s] on rank-fused tensors."""
    return np.einsum("bnihs,bnjhs->bnhij", c_bnLhn, b_bnLhn)


def k3_chunk_state(v_bnLhp, b_bnLhn, cum_fused_bhnL):
    """K3: chunk-end state from zero: sum_i exp(cum_last - cum[i//R]) V[i,:]^T B[i,:] -> [b,n,h,p,s]."""
    last = cum_fused_bhnL[..., -1:]
    decay = np.exp(last - cum_fused_bhnL)                        # [b,h,n,L]
    dv = v_bnLhp * np.transpose(decay, (0, 2, 3, 1))[..., None]  # [b,n,L,h,p]
    return np.einsum("bnihp,bnihs->bnhps", dv, b_bnLhn)


def k4_state_passing(states_bnhps, chunk_end_bhn, init_bhps):
    """K4: sequential h <- exp(chunk_end[c]) h + S[c]; returns per-chunk input states and final."""
    nch = states_bnhps.shape[1]
    h = init_bhps.copy()
    ins = []
    for c in range(nch):
        ins.append(h.copy())
        h = np.exp(chunk_end_bhn[:, :, c])[:, :, None, None] * h + states_bnhps[:, c]
    return np.stack(ins, axis=1), h


def k5_chunk_scan(cum_fused_bhnL, da_bhnl, v_bnLhp, c_bnLhn, cb_bnhLL, hin_bnhps, R):
    """K5: y = (L_mimo o CB) V + exp(cum[i//R]) C[i] h_in.

    L_mimo is exp(segsum(dA)) of the unfused chunk, expanded so that
    L[i, j] = exp(cum[i//R] - cum[j//R]) when i//R >= j//R and 0 otherwise.
    """
    b, n, L, H, P = v_bnLhp.shape
    l = L // R
    cum = np.transpose(cum_fused_bhnL, (0, 2, 1, 3))               # [b,n,h,L]
    # off-diagonal ("blue") part: exp(cum_i) * C_i . h_in
    blue = np.exp(cum)[..., None] * np.einsum("bnihs,bnhps->bnhip", c_bnLhn, hin_bnhps)
    # diagonal ("orange") part
    seg = segsum(np.transpose(da_bhnl, (0, 2, 1, 3)))             # [b,n,h,l,l]
    seg_f = np.repeat(np.repeat(seg, R, axis=-2), R, axis=-1)      # [b,n,h,L,L]
    orange = np.einsum("bnhij,bnjhp->bnhip", np.exp(seg_f) * cb_bnhLL, v_bnLhp)
    y = blue + orange                                              # [b,n,h,L,p]
    return np.transpose(y, (0, 1, 3, 2, 4)).reshape(b, n, l, R, H, P)


def chunked_forward(x, dA, B, C, theta=None, init_state=None, chunk_len=64):
    """K1..K5 on [b,T,R,H,P] inputs; returns (y [b,T,R,H,P], final [b,H,P,N])."""
    x = np.asarray(x, np.float64)
    dA = np.asarray(dA, np.float64)
    B = np.asarray(B, np.float64)
    C = np.asarray(C, np.float64)
    b, T, R, H, P = x.shape
    G, N = B.shape[3], B.shape[4]
    hpg = H // G
    # per-head B/C (expand groups)
    Bh = np.repeat(B, hpg, axis=3)
    Ch = np.repeat(C, hpg, axis=3)
    phi = None
    if theta is not None:
        phi = np.cumsum(np.asarray(theta, np.float64), axis=1)     # [b,T,H,N/2]
        Bh = rotate_pairs(Bh, -phi[:, :, None, :, :])
        Ch = rotate_pairs(Ch, -phi[:, :, None, :, :])
    init = np.zeros((b, H, P, N)) if init_state is None else np.asarray(init_state, np.float64)
    if T == 0:
        return np.zeros((b, 0, R, H, P)), init.copy()
    l = int(chunk_len)
    nch = -(-T // l)
    pad = nch * l - T
    if pad:
        x = np.concatenate([x, np.zeros((b, pad, R, H, P))], axis=1)
        dA = np.concatenate([dA, np.zeros((b, pad, H))], axis=1)
        Bh = np.concatenate([Bh, np.zeros((b, pad, R, H, N))], axis=1)
        Ch = np.concatenate([Ch, np.zeros((b, pad, R, H, N))], axis=1)
    L = l * R
    v = x.reshape(b, nch, L, H, P)
    bf = Bh.reshape(b, nch, L, H, N)
    cf = Ch.reshape(b, nch, L, H, N)
    da_bnlh = dA.reshape(b, nch, l, H)
    cum, chunk_end = k1_chunk_cumsum(da_bnlh)
    cum_fused = np.repeat(cum, R, axis=3)                          # [b,h,n,L]
    cb = k2_bmm(cf, bf)
    states = k3_chunk_state(v, bf, cum_fused)
    hin, final = k4_state_passing(states, chunk_end, init)
    y = k5_chunk_scan(cum_fused, np.transpose(da_bnlh, (0, 3, 1, 2)), v, cf, cb, hin, R).reshape(b, nch * l, R, H, P)[:, :T]
    if phi is not None:
        final = rotate_pairs(final, phi[:, T - 1][:, :, None, :])
    return y, final


def trapezoidal_absorbed(x, dA, B, C, gamma, beta, theta=None, init_state=None, prev_x=None,
                         prev_B=None):
    """The scan.py page's trapezoidal forward in its absorbed frame: per step the write
    S_t = sum_r x_{t,r} (outer) B_{t,r}; the beta stream is S shifted one step (S_{-1} from
    prev_x/prev_B); w_t = gamma_t R(-Phi_t) S_t + beta_t R(-Phi_{t-1}) S_{t-1} with Phi_{-1} = 0;
    g_t = exp(dA_t) g_{t-1} + w_t from g_{-1} = h_{-1}; h_t = R(Phi_t) g_t; y_t = C_t . h_t.
    Returns (y [b,T,R,H,P], final [b,H,P,N])."""
    x, dA, B, C, gamma, beta = (np.asarray(v, np.float64) for v in (x, dA, B, C, gamma, beta))
    b, T, R, H, P = x.shape
    G, N = B.shape[3], B.shape[4]
    Bh = np.repeat(B, H // G, axis=3)                        # [b,T,R,H,N]
    Ch = np.repeat(C, H // G, axis=3)
    S = np.einsum("btrhp,btrhn->bthpn", x, Bh)               # [b,T,H,P,N]
    if prev_x is not None:
        s0 = np.einsum("brhp,brhn->bhpn", np.asarray(prev_x, np.float64),
                       np.repeat(np.asarray(prev_B, np.float64), H // G, axis=2))
    else:
        s0 = np.zeros((b, H, P, N))
    Sprev = np.concatenate([s0[:, None], S[:, :-1]], axis=1)
    if theta is not None:
        phi = np.cumsum(np.asarray(theta, np.float64), axis=1)   # [b,T,H,N/2]
    else:
        phi = np.zeros((b, T, H, N // 2))
    phi_prev = np.concatenate([np.zeros_like(phi[:, :1]), phi[:, :-1]], axis=1)
    w = (gamma[..., None, None] * rotate_pairs(S, -phi[:, :, :, None, :])
         + beta[..., None, None] * rotate_pairs(Sprev, -phi_prev[:, :, :, None, :]))
    g = np.zeros((b, H, P, N)) if init_state is None else np.asarray(init_state, np.float64).copy()
    y = np.zeros((b, T, R, H, P))
    for t in range(T):
        g = np.exp(dA[:, t])[:, :, None, None] * g + w[:, t]
        h = rotate_pairs(g, phi[:, t][:, :, None, :])
        y[:, t] = np.einsum("brhn,bhpn->brhp", Ch[:, t], h)
    final = rotate_pairs(g, phi[:, T - 1][:, :, None, :]) if T else g
    return y, final


def chunked_backward(x, dA, B, C, dy, init_state=None, dfinal=None, chunk_len=64):
    """Reverse mode of the unrotated SSD in the chunked form the GPU backward uses, fp64, for
    the loss <dy, y> + <dfinal, final> (the pages give no backward formulas: this is the chain
    rule through the K1..K5 decomposition, written out per chunk).  Per chunk c, with fused
    rows i (step s(i) = i // R), cum the in-chunk prefix of dA, L_ij = exp(cum_s(i) - cum_s(j))
    for s(j) <= s(i), CB = C B^T, DX = dy x^T, M = L o CB, A = L o DX, W = M o DX,
    el_j = exp(cum_end - cum_s(j)), e_i = exp(cum_s(i)), h_in the chunk-input state and
    G = dL/dh_out the gradient carried back from the later chunks (D_c = sum_i e_i dy_i C_i^T):
      dx = M^T dy + diag(el) B G^T        dB = A^T C + diag(el) x G       dC = A B + diag(e) dy h_in
      dL/dcum_s = sum over the step's rows of (rowsum W - colsum W + E_i - Q_i), with
      E_i = e_i C_i . (h_in^T dy_i), Q_j = el_j x_j . (G B_j), plus at the chunk's last step
      sum_j Q_j + exp(cum_end) <G, h_in>;  ddA_t = sum_{s >= t in the chunk} dL/dcum_s.
    Returns dict dx, ddA, dB, dC, dinit."""
    x, dA, B, C, dy = (np.asarray(v, np.float64) for v in (x, dA, B, C, dy))
    b, T, R, H, P = x.shape
    G, N = B.shape[3], B.shape[4]
    l = int(chunk_len)
    nch = -(-T // l)
    Tp = nch * l
    pad = Tp - T

    def padt(v):
        if pad == 0:
            return v
        w = [(0, 0)] * v.ndim
        w[1] = (0, pad)
        return np.pad(v, w)

    xp, dAp, Bp, Cp, dyp = (padt(v) for v in (x, dA, B, C, dy))
    L = l * R
    step = np.arange(L) // R
    out = {"dx": np.zeros_like(x), "ddA": np.zeros_like(dA), "dB": np.zeros_like(B),
           "dC": np.zeros_like(C), "dinit": np.zeros((b, H, P, N))}
    dBp = np.zeros_like(Bp)
    dCp = np.zeros_like(Cp)
    for bi in range(b):
        for hi in range(H):
            g = hi // (H // G)
            X = xp[bi, :, :, hi, :].reshape(nch, L, P)
            Bm = Bp[bi, :, :, g, :].reshape(nch, L, N)
            Cm = Cp[bi, :, :, g, :].reshape(nch, L, N)
            DY = dyp[bi, :, :, hi, :].reshape(nch, L, P)
            cum = np.cumsum(dAp[bi, :, hi].reshape(nch, l), axis=1)
            cumr = cum[:, step]
            cend = cum[:, -1]
            S = [(np.exp(cend[c] - cumr[c])[:, None] * X[c]).T @ Bm[c] for c in range(nch)]
            D = [(np.exp(cumr[c])[:, None] * DY[c]).T @ Cm[c] for c in range(nch)]
            hin = []
            h = (np.zeros((P, N)) if init_state is None
                 else np.asarray(init_state, np.float64)[bi, hi])
            for c in range(nch):
                hin.append(h)
                h = np.exp(cend[c]) * h + S[c]
            Gc = [None] * nch
            gcur = (np.zeros((P, N)) if dfinal is None
                    else np.asarray(dfinal, np.float64)[bi, hi])
            for c in range(nch - 1, -1, -1):
                Gc[c] = gcur
                gcur = np.exp(cend[c]) * gcur + D[c]
            out["dinit"][bi, hi] = gcur
            for c in range(nch):
                causal = step[:, None] >= step[None, :]
                Lm = np.where(causal, np.exp(np.where(causal, cumr[c][:, None] - cumr[c][None, :],
                                                      0.0)), 0.0)
                CB = Cm[c] @ Bm[c].T
                DX = DY[c] @ X[c].T
                M, A = Lm * CB, Lm * DX
                W = M * DX
                el, e = np.exp(cend[c] - cumr[c]), np.exp(cumr[c])
                U = el[:, None] * (Bm[c] @ Gc[c].T)            # [L, P]
                V = DY[c] @ hin[c]                              # [L, N]
                dxc = M.T @ DY[c] + U
                dBc = A.T @ Cm[c] + el[:, None] * (X[c] @ Gc[c])
                dCc = A @ Bm[c] + e[:, None] * V
                E = e * np.sum(Cm[c] * V, axis=1)
                Q = np.sum(X[c] * U, axis=1)
                rows = W.sum(axis=1) - W.sum(axis=0) + E - Q
                dcum = rows.reshape(l, R).sum(axis=1)
                dcum[-1] += Q.sum() + np.exp(cend[c]) * np.sum(Gc[c] * hin[c])
                ddA_c = np.cumsum(dcum[::-1])[::-1]
                t0 = c * l
                nv = min(l, T - t0)
                out["dx"][bi, t0:t0 + nv, :, hi, :] = dxc.reshape(l, R, P)[:nv]
                out["ddA"][bi, t0:t0 + nv, hi] = ddA_c[:nv]
                dBp[bi, t0:t0 + l, :, g, :] += dBc.reshape(l, R, N)
                dCp[bi, t0:t0 + l, :, g, :] += dCc.reshape(l, R, N)
    out["dB"] = dBp[:, :T]
    out["dC"] = dCp[:, :T]
    return out


def chunked_backward_rotated(x, dA, B, C, theta, dy, init_state=None, dfinal=None, chunk_len=64):
    """Reverse mode of the rotated SSD in chunk-local frames, fp64 (the form the GPU backward
    uses).  Inside chunk c, phi_t is the angle accumulated since the chunk's start; the chunk is
    the plain problem on B^ = R(-phi)B, C^ = R(-phi)C entered with the physical h_in(c) and left
    through h_in(c+1) = R(phi_end) g_end.  The plain per-chunk gradients (chunked_backward's
    formulas) on B^, C^ with G^_c = R(-phi_end) dL/dh_in(c+1) then give dB = R(phi) dB^,
    dC = R(phi) dC^ and dL/dphi_t = sum over the step's rows of (dB^_0 B^_1 - dB^_1 B^_0 +
    dC^_0 C^_1 - dC^_1 C^_0) plus, at the chunk's end, sum_p (G^_1 g_0 - G^_0 g_1) with
    g = g_end; dtheta_t sums dL/dphi over the steps t .. chunk end.  Returns dict dx, ddA, dB,
    dC, dtheta, dinit."""
    x, dA, B, C, theta, dy = (np.asarray(v, np.float64) for v in (x, dA, B, C, theta, dy))
    b, T, R, H, P = x.shape
    G, N = B.shape[3], B.shape[4]
    K = N // 2
    l = int(chunk_len)
    nch = -(-T // l)
    pad = nch * l - T

    def padt(v):
        if pad == 0:
            return v
        w = [(0, 0)] * v.ndim
        w[1] = (0, pad)
        return np.pad(v, w)

    xp, dAp, Bp, Cp, dyp, thp = (padt(v) for v in (x, dA, B, C, dy, theta))
    L = l * R
    step = np.arange(L) // R
    out = {"dx": np.zeros_like(x), "ddA": np.zeros_like(dA), "dtheta": np.zeros_like(theta),
           "dinit": np.zeros((b, H, P, N))}
    dBp = np.zeros_like(Bp)
    dCp = np.zeros_like(Cp)
    cross = lambda d, v: d[..., 0::2] * v[..., 1::2] - d[..., 1::2] * v[..., 0::2]
    for bi in range(b):
        for hi in range(H):
            g = hi // (H // G)
            X = xp[bi, :, :, hi, :].reshape(nch, L, P)
            DY = dyp[bi, :, :, hi, :].reshape(nch, L, P)
            cum = np.cumsum(dAp[bi, :, hi].reshape(nch, l), axis=1)
            cumr = cum[:, step]
            cend = cum[:, -1]
            phi = np.cumsum(thp[bi, :, hi, :].reshape(nch, l, K), axis=1)   # local angles
            phir = phi[:, step, :]                                           # [nch, L, K]
            Bh = rotate_pairs(Bp[bi, :, :, g, :].reshape(nch, L, N), -phir)
            Ch = rotate_pairs(Cp[bi, :, :, g, :].reshape(nch, L, N), -phir)
            pend = phi[:, -1, :]                                             # [nch, K]
            S = [(np.exp(cend[c] - cumr[c])[:, None] * X[c]).T @ Bh[c] for c in range(nch)]
            D = [(np.exp(cumr[c])[:, None] * DY[c]).T @ Ch[c] for c in range(nch)]
            hin, gend = [], []
            h = (np.zeros((P, N)) if init_state is None
                 else np.asarray(init_state, np.float64)[bi, hi])
            for c in range(nch):
                hin.append(h)
                ge = np.exp(cend[c]) * h + S[c]
                gend.append(ge)
                h = rotate_pairs(ge, np.broadcast_to(pend[c], (P, K)))
            Gh = [None] * nch
            v = (np.zeros((P, N)) if dfinal is None
                 else np.asarray(dfinal, np.float64)[bi, hi])
            for c in range(nch - 1, -1, -1):
                Gh[c] = rotate_pairs(v, np.broadcast_to(-pend[c], (P, K)))
                v = np.exp(cend[c]) * Gh[c] + D[c]
            out["dinit"][bi, hi] = v
            for c in range(nch):
                causal = step[:, None] >= step[None, :]
                Lm = np.where(causal, np.exp(np.where(causal, cumr[c][:, None] - cumr[c][None, :],
                                                      0.0)), 0.0)
                CB = Ch[c] @ Bh[c].T
                DX = DY[c] @ X[c].T
                M, A = Lm * CB, Lm * DX
                W = M * DX
                el, e = np.exp(cend[c] - cumr[c]), np.exp(cumr[c])
                U = el[:, None] * (Bh[c] @ Gh[c].T)
                V = DY[c] @ hin[c]
                dxc = M.T @ DY[c] + U
                dBh = A.T @ Ch[c] + el[:, None] * (X[c] @ Gh[c])
                dCh = A @ Bh[c] + e[:, None] * V
                E = e * np.sum(Ch[c] * V, axis=1)
                Q = np.sum(X[c] * U, axis=1)
                rows = W.sum(axis=1) - W.sum(axis=0) + E - Q
                dcum = rows.reshape(l, R).sum(axis=1)
                dcum[-1] += Q.sum() + np.exp(cend[c]) * np.sum(Gh[c] * hin[c])
                ddA_c = np.cumsum(dcum[::-1])[::-1]
                dphi = (cross(dBh, Bh[c]) + cross(dCh, Ch[c])).reshape(l, R, K).sum(axis=1)
                dphi[-1] += cross(gend[c], Gh[c]).sum(axis=0)   # sum_p (G^_1 g_0 - G^_0 g_1)
                dth = np.cumsum(dphi[::-1], axis=0)[::-1]
                t0 = c * l
                nv = min(l, T - t0)
                out["dx"][bi, t0:t0 + nv, :, hi, :] = dxc.reshape(l, R, P)[:nv]
                out["ddA"][bi, t0:t0 + nv, hi] = ddA_c[:nv]
                out["dtheta"][bi, t0:t0 + nv, hi, :] = dth[:nv]
                dBp[bi, t0:t0 + l, :, g, :] += rotate_pairs(dBh, phir[c]).reshape(l, R, N)
                dCp[bi, t0:t0 + l, :, g, :] += rotate_pairs(dCh, phir[c]).reshape(l, R, N)
    out["dB"] = dBp[:, :T]
    out["dC"] = dCp[:, :T]
    return out


def trapezoidal_backward_expanded(x, dA, B, C, gamma, beta, dy, theta=None, init_state=None,
                                  prev_x=None, prev_B=None, dfinal=None, chunk_len=64):
    """Reverse mode of the trapezoidal SSD through its 2R-channel expansion (the form the GPU
    uses), fp64: x^ = [gamma_t x_t, beta_t x_{t-1}], B^ = [B_t, R(theta_t) B_{t-1}] (per head
    with theta), C^ = [C_t, 0], dy^ = [dy, 0]; the chunked backward of that plain (or rotated)
    problem, then the chain rule back through the expansion:
      dx_t = gamma_t dx^[t, r] + beta_{t+1} dx^[t+1, R+r],  dprev_x = beta_0 dx^[0, R+r]
      dgamma_t = <dx^[t, :R], x_t>,  dbeta_t = <dx^[t, R:], x_{t-1}>
      dB_t = sum_heads dB^[t, r] + R(theta_{t+1})^T dB^[t+1, R+r],  dprev_B likewise at t = 0
      dC_t = sum_heads dC^[t, r],  dtheta_t = dtheta^_t + sum_r (dB^_1 B^_0 - dB^_0 B^_1)[t, R+r].
    Returns the same dict as oracle.ssd_trap_backward."""
    x, dA, B, C, gamma, beta, dy = (np.asarray(v, np.float64)
                                    for v in (x, dA, B, C, gamma, beta, dy))
    b, T, R, H, P = x.shape
    G, N = B.shape[3], B.shape[4]
    rot = theta is not None
    th = np.asarray(theta, np.float64) if rot else None
    G2 = H if rot else G
    hof = (np.arange(H) // (H // G)) if rot else np.arange(G)   # group of each expanded row
    xprev = np.zeros_like(x)
    xprev[:, 1:] = x[:, :-1]
    Bprev = np.zeros_like(B)
    Bprev[:, 1:] = B[:, :-1]
    if prev_x is not None:
        xprev[:, 0] = np.asarray(prev_x, np.float64)
        Bprev[:, 0] = np.asarray(prev_B, np.float64)
    xh = np.concatenate([gamma[:, :, None, :, None] * x, beta[:, :, None, :, None] * xprev], axis=2)
    Bcur, Bsh = B[:, :, :, hof, :], Bprev[:, :, :, hof, :]          # [b, T, R, G2, N]
    if rot:
        Bsh = rotate_pairs(Bsh, th[:, :, None, :, :])
    Bh = np.concatenate([Bcur, Bsh], axis=2)
    Ch = np.concatenate([C[:, :, :, hof, :], np.zeros_like(Bsh)], axis=2)
    dyh = np.concatenate([dy, np.zeros_like(dy)], axis=2)
    if rot:
        g = chunked_backward_rotated(xh, dA, Bh, Ch, th, dyh, init_state, dfinal, chunk_len)
    else:
        g = chunked_backward(xh, dA, Bh, Ch, dyh, init_state, dfinal, chunk_len)
    dxh, dBh, dCh = g["dx"], g["dB"], g["dC"]
    out = {"ddA": g["ddA"], "dinit": g["dinit"]}
    dx = gamma[:, :, None, :, None] * dxh[:, :, :R]
    dx[:, :-1] += beta[:, 1:, None, :, None] * dxh[:, 1:, R:]
    out["dx"] = dx
    out["dgamma"] = np.sum(dxh[:, :, :R] * x, axis=(2, 4))
    out["dbeta"] = np.sum(dxh[:, :, R:] * xprev, axis=(2, 4))
    back = dBh[:, :, R:]                                             # shifted channels
    if rot:
        back = rotate_pairs(back, -th[:, :, None, :, :])             # R(theta_t)^T
    dB = np.zeros_like(B)
    dC = np.zeros_like(C)
    dpB = np.zeros((b, R, G, N))
    for j in range(G2):
        gi = hof[j]
        dB[:, :, :, gi] += dBh[:, :, :R, j]
        dB[:, :-1, :, gi] += back[:, 1:, :, j]
        dC[:, :, :, gi] += dCh[:, :, :R, j]
        dpB[:, :, gi] += back[:, 0, :, j]
    out["dB"], out["dC"] = dB, dC
    if rot:
        sh, dsh = Bh[:, :, R:], dBh[:, :, R:]
        extra = dsh[..., 1::2] * sh[..., 0::2] - dsh[..., 0::2] * sh[..., 1::2]
        out["dtheta"] = g["dtheta"] + extra.sum(axis=2)
    if prev_x is not None:
        out["dprev_x"] = beta[:, 0, None, :, None] * dxh[:, 0, R:]
        out["dprev_B"] = dpB
    return out

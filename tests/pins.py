"""Checks that tie the fp64 oracle to facts fixed by the pages and by plain mathematics.

Each ``pin_*`` function runs the oracle (optionally with one planted mistake, ``mutation``) on
small seeded inputs and returns a list of ``(check name, error, tolerance)``.  With
``mutation=0`` every error must be within tolerance; with each planted mistake at least one
check must fail, which shows that the pins would notice that kind of error.

None of these checks re-types the oracle's own loop: they compare it with printed values, closed
forms, a differently organised computation (the pages' chunked algebra in
``oracle.chunked_ref``), superposition identities, or exact invariants.
"""
from __future__ import annotations

import math
import os

import numpy as np

import oracle
from oracle import chunked_ref

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _rng(seed):
    return np.random.default_rng(seed)


def _problem(seed, b, T, R, H, G, P, N, *, theta=False, init=False, decay=(0.0, 0.5)):
    r = _rng(seed)
    x = r.standard_normal((b, T, R, H, P))
    dA = -r.uniform(decay[0], decay[1], (b, T, H))
    B = r.standard_normal((b, T, R, G, N))
    C = r.standard_normal((b, T, R, G, N))
    th = r.uniform(-0.4, 0.4, (b, T, H, N // 2)) if theta else None
    h0 = r.standard_normal((b, H, P, N)) if init else None
    return x, dA, B, C, th, h0


def _maxerr(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    if a.size == 0 and b.size == 0:
        return 0.0
    return float(np.max(np.abs(a - b)))


def load_golden(name):
    vals = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            k, v = line.split(":", 1)
            vals[k.strip()] = [float(t) for t in v.split()]
    return vals


# --------------------------------------------------------------------------------------------
# Selective scan
# --------------------------------------------------------------------------------------------

def pin_worked_example(mutation=0):
    """The SSM Selective Scan page's worked example (section 示例), to its 3 printed decimals."""
    g = load_golden("selective_scan_worked_example.txt")
    b, T, D, N = (int(g[k][0]) for k in ("batch", "seq_len", "d_model", "d_state"))
    u = np.array(g["u"]).reshape(b, T, D)
    delta = np.array(g["delta"]).reshape(b, T, D)
    A = np.array(g["A"]).reshape(D, N)
    B = np.array(g["B"]).reshape(b, T, N)
    C = np.array(g["C"]).reshape(b, T, N)
    skip = np.array(g["skip"])
    tol = g["tolerance"][0] + 1e-9
    y = oracle.selective_scan(u, delta, A, B, C, skip, mutation=mutation)
    # A_bar is printed for delta = 1: exp(1 * A).  A single step from h = e_n isolates it.
    abar = []
    for d in range(D):
        for n in range(N):
            uu = np.zeros((1, 2, D)); uu[0, 0, d] = 1.0
            dd = np.ones((1, 2, D))
            BB = np.zeros((1, 2, N)); BB[0, 0, n] = 1.0
            CC = np.zeros((1, 2, N)); CC[0, 1, n] = 1.0
            yy = oracle.selective_scan(uu, dd, A, BB, CC, None, mutation=mutation)
            abar.append(yy[0, 1, d])
    return [
        ("worked_example_y", _maxerr(y.reshape(-1), g["y"]), tol),
        ("worked_example_A_bar", _maxerr(abar, g["A_bar"]), tol),
    ]


def pin_selective_scan_superposition(mutation=0):
    """A diagonal-A selective scan is N independent scalar recurrences per channel, each of them
    an SSD problem with one state (heads = channels, P = N = 1, x = delta*u, dA = delta*A[:,n]),
    plus the skip term: y = sum_n SSD_n + skip*u."""
    r = _rng(11)
    b, T, D, N = 2, 23, 5, 4
    u = r.standard_normal((b, T, D))
    delta = np.log1p(np.exp(r.standard_normal((b, T, D))))
    A = -r.uniform(0.5, 2.0, (D, N))
    B = r.standard_normal((b, T, N))
    C = r.standard_normal((b, T, N))
    skip = r.standard_normal((D,))
    y = oracle.selective_scan(u, delta, A, B, C, skip, mutation=mutation)
    ref = skip[None, None, :] * u
    for n in range(N):
        x = (delta * u)[:, :, None, :, None]                     # [b,T,1,D,1]
        dA = delta * A[None, None, :, n]                          # [b,T,D]
        Bn = np.broadcast_to(B[:, :, None, None, n:n + 1], (b, T, 1, 1, 1))
        Cn = np.broadcast_to(C[:, :, None, None, n:n + 1], (b, T, 1, 1, 1))
        yn, _ = oracle.ssd(x, dA, Bn, Cn)
        ref = ref + yn[:, :, 0, :, 0]
    return [("selective_scan_vs_scalar_ssd_sum", _maxerr(y, ref), 1e-11)]


# --------------------------------------------------------------------------------------------
# SSD
# --------------------------------------------------------------------------------------------

def pin_closed_form(mutation=0):
    """scan.py page, module docstring "THE SCAN": g_t = A_t * (g_-1 + sum_{s<=t} w_s / A_s) with
    A_t = prod_{r<=t} alpha_r, evaluated by brute force on tiny inputs (alpha in [0.5, 1))."""
    out = []
    for seed, T in ((1, 1), (2, 7), (3, 16)):
        r = _rng(seed)
        alpha = r.uniform(0.5, 1.0, T)
        w = r.standard_normal(T)
        g0 = r.standard_normal()
        ref = []
        for t in range(T):
            At = math.prod(alpha[: t + 1])
            ref.append(At * (g0 + sum(w[s] / math.prod(alpha[: s + 1]) for s in range(t + 1))))
        x = w.reshape(1, T, 1, 1, 1)
        dA = np.log(alpha).reshape(1, T, 1)
        one = np.ones((1, T, 1, 1, 1))
        y, fin = oracle.ssd(x, dA, one, one, init_state=np.full((1, 1, 1, 1), g0),
                            mutation=mutation)
        out.append((f"closed_form_T{T}", _maxerr(y.reshape(-1), ref), 1e-12))
        out.append((f"closed_form_final_T{T}", _maxerr(fin.reshape(-1), ref[-1:]), 1e-12))
    return out


def pin_special_cases(mutation=0):
    """Cases that reduce to textbook forms: no decay (dA = 0) with one state and one channel is a
    prefix sum y_t = C_t * sum_{s<=t} x_s B_s; a single step is y = C . (exp(dA) h0 + x (x) B)."""
    r = _rng(5)
    T = 19
    x, B, C = r.standard_normal(T), r.standard_normal(T), r.standard_normal(T)
    y, _ = oracle.ssd(x.reshape(1, T, 1, 1, 1), np.zeros((1, T, 1)), B.reshape(1, T, 1, 1, 1),
                      C.reshape(1, T, 1, 1, 1), mutation=mutation)
    res = [("prefix_sum", _maxerr(y.reshape(-1), C * np.cumsum(x * B)), 1e-12)]
    P, N = 3, 4
    x1 = r.standard_normal((1, 1, 1, 1, P))
    B1 = r.standard_normal((1, 1, 1, 1, N))
    C1 = r.standard_normal((1, 1, 1, 1, N))
    dA1 = np.array([[[-0.3]]])
    h0 = r.standard_normal((1, 1, P, N))
    y1, f1 = oracle.ssd(x1, dA1, B1, C1, init_state=h0, mutation=mutation)
    h1 = math.exp(-0.3) * h0[0, 0] + np.outer(x1.reshape(P), B1.reshape(N))
    res.append(("single_step_y", _maxerr(y1.reshape(P), h1 @ C1.reshape(N)), 1e-13))
    res.append(("single_step_final", _maxerr(f1[0, 0], h1), 1e-13))
    return res


def pin_chunk_invariance(mutation=0):
    """The serial.rs page's K1..K5 decomposition (restated in oracle.chunked_ref) computed at
    chunk lengths 1, 8, 16, 64 and T must equal the sequential recurrence: chunking is exact.
    Same pattern as the scan.py page's verify() (chunks 8/16/64, a ragged length 37)."""
    res = []
    cases = [
        dict(seed=21, b=2, T=64, R=1, H=2, G=2, P=4, N=6, init=False),
        dict(seed=22, b=1, T=37, R=1, H=4, G=2, P=3, N=4, init=True),      # ragged, groups
        dict(seed=23, b=2, T=40, R=3, H=2, G=1, P=3, N=4, init=True),      # MIMO, shared B/C
    ]
    for c in cases:
        x, dA, B, C, th, h0 = _problem(c["seed"], c["b"], c["T"], c["R"], c["H"], c["G"], c["P"],
                                       c["N"], init=c["init"])
        y, fin = oracle.ssd(x, dA, B, C, init_state=h0, mutation=mutation)
        for l in (1, 8, 16, 64, c["T"]):
            y2, f2 = chunked_ref.chunked_forward(x, dA, B, C, None, h0, l)
            res.append((f"chunk{l}_seed{c['seed']}_y", _maxerr(y, y2), 1e-10))
            res.append((f"chunk{l}_seed{c['seed']}_final", _maxerr(fin, f2), 1e-10))
    return res


def pin_rotation(mutation=0):
    """The scan.py page's rotation identity (module docstring "THE TRICK"): the rotated
    recurrence equals the plain scan with B~ = R(-Phi_t) B, C~ = R(-Phi_t) C and the state turned
    back by R(Phi_{T-1}).  Plus two exact facts: theta = 0 changes nothing, and with no writes
    and no decay the state is the initial state turned by the summed angle (rotate_by's
    convention: (a, b) -> (c a - s b, s a + c b))."""
    res = []
    x, dA, B, C, th, h0 = _problem(31, 2, 45, 2, 2, 1, 3, 6, theta=True, init=True)
    y, fin = oracle.ssd(x, dA, B, C, th, h0, mutation=mutation)
    for l in (1, 16, 45):
        y2, f2 = chunked_ref.chunked_forward(x, dA, B, C, th, h0, l)
        res.append((f"rotation_absorbed_chunk{l}_y", _maxerr(y, y2), 1e-10))
        res.append((f"rotation_absorbed_chunk{l}_final", _maxerr(fin, f2), 1e-10))
    y0, f0 = oracle.ssd(x, dA, B, C, np.zeros_like(th), h0, mutation=mutation)
    yn, fn = oracle.ssd(x, dA, B, C, None, h0, mutation=mutation)
    res.append(("theta_zero_is_identity", max(_maxerr(y0, yn), _maxerr(f0, fn)), 0.0))
    T = 9
    r = _rng(32)
    ang = r.uniform(-0.5, 0.5, (1, T, 1, 1))
    h0 = np.array([1.0, 0.0]).reshape(1, 1, 1, 2)
    _, f = oracle.ssd(np.zeros((1, T, 1, 1, 1)), np.zeros((1, T, 1)), np.zeros((1, T, 1, 1, 2)),
                      np.zeros((1, T, 1, 1, 2)), ang, h0, mutation=mutation)
    tot = float(ang.sum())
    res.append(("pure_rotation", _maxerr(f.reshape(2), [math.cos(tot), math.sin(tot)]), 1e-13))
    return res


def pin_mimo_superposition(mutation=0):
    """MIMO: every rank's write of step t lands before y_{t,r} is read (the serial.rs page's K5
    mask i//R >= j//R).  By linearity the rank-R output is the sum over writing ranks r' of
    rank-1 runs: y[:, :, r] = sum_{r'} SSD(x_{r'}, B_{r'}, C_r), the initial state counted once."""
    b, T, R, H, G, P, N = 2, 21, 3, 2, 2, 3, 4
    x, dA, B, C, th, h0 = _problem(41, b, T, R, H, G, P, N, theta=True, init=True)
    y, fin = oracle.ssd(x, dA, B, C, th, h0, mutation=mutation)
    yref = np.zeros_like(y)
    fref = np.zeros_like(fin)
    for rp in range(R):
        for r in range(R):
            ys, fs = oracle.ssd(x[:, :, rp:rp + 1], dA, B[:, :, rp:rp + 1], C[:, :, r:r + 1], th,
                                h0 if rp == 0 else None)
            yref[:, :, r] += ys[:, :, 0]
            if r == 0:
                fref += fs
    return [("mimo_superposition_y", _maxerr(y, yref), 1e-11),
            ("mimo_superposition_final", _maxerr(fin, fref), 1e-11)]


def pin_causality_and_continuation(mutation=0):
    """Causality (scan.py page, verify(): appended large noise must not change earlier outputs)
    and continuation (the serial.rs page's initial_state / final_state hand-off): two calls
    chained through the final state equal one call."""
    b, T, R, H, G, P, N = 2, 40, 2, 2, 1, 3, 4
    x, dA, B, C, th, h0 = _problem(51, b, T + 9, R, H, G, P, N, theta=True, init=True)
    x2 = x.copy()
    x2[:, T:] *= 50.0
    ya, _ = oracle.ssd(x[:, :T], dA[:, :T], B[:, :T], C[:, :T], th[:, :T], h0, mutation=mutation)
    yb, _ = oracle.ssd(x2, dA, B, C, th, h0, mutation=mutation)
    res = [("causality", _maxerr(ya, yb[:, :T]), 0.0)]
    yf, ff = oracle.ssd(x, dA, B, C, th, h0, mutation=mutation)
    y1, f1 = oracle.ssd(x[:, :T], dA[:, :T], B[:, :T], C[:, :T], th[:, :T], h0, mutation=mutation)
    y2, f2 = oracle.ssd(x[:, T:], dA[:, T:], B[:, T:], C[:, T:], th[:, T:], f1, mutation=mutation)
    res.append(("continuation_y", _maxerr(yf, np.concatenate([y1, y2], axis=1)), 1e-12))
    res.append(("continuation_final", _maxerr(ff, f2), 1e-12))
    return res


SSD_PINS = [pin_closed_form, pin_special_cases, pin_chunk_invariance, pin_rotation,
            pin_mimo_superposition, pin_causality_and_continuation]
SS_PINS = [pin_worked_example, pin_selective_scan_superposition]


# ------------------------------------------------------------------------------ trapezoidal
def _trap_problem(seed, b, T, R, H, G, P, N, *, theta=False, prev=True):
    x, dA, B, C, th, h0 = _problem(seed, b, T, R, H, G, P, N, theta=theta, init=True)
    r = _rng(seed + 1000)
    gamma = r.uniform(0.2, 1.0, (b, T, H))
    beta = r.uniform(0.2, 1.0, (b, T, H))
    px = r.standard_normal((b, R, H, P)) if prev else None
    pb = r.standard_normal((b, R, G, N)) if prev else None
    return x, dA, B, C, gamma, beta, th, h0, px, pb


def pin_trapezoidal_rule(mutation=0):
    """With no decay (dA = 0) and gamma = beta = 1/2 the state is the trapezoidal-rule sum of the
    writes; for a write that is linear in time, s_t = t, with s_{-1} = -1 from the previous
    step, that sum is exact: h_t = integral of s from -1 to t = (t^2 - 1)/2."""
    T = 12
    t = np.arange(T, dtype=np.float64)
    x = t.reshape(1, T, 1, 1, 1)
    one = np.ones((1, T, 1, 1, 1))
    half = np.full((1, T, 1), 0.5)
    y, f = oracle.ssd_trapezoidal(x, np.zeros((1, T, 1)), one, one, half, half,
                                  prev_x=np.full((1, 1, 1, 1), -1.0),
                                  prev_B=np.ones((1, 1, 1, 1)), mutation=mutation)
    ref = (t * t - 1.0) / 2.0
    return [("trapezoid_of_linear_write", _maxerr(y.reshape(T), ref), 1e-12),
            ("trapezoid_final", _maxerr(f.reshape(1), ref[-1:]), 1e-12)]


def pin_trapezoidal_absorbed_frame(mutation=0):
    """The scan.py page's own trapezoidal algebra (absorbed frame: the gamma write turned by
    -Phi_t, the beta write by -Phi_{t-1}, one step less; chunked_ref.trapezoidal_absorbed)
    against the oracle's physical-frame recurrence, with MIMO ranks, groups, an initial state
    and a previous write."""
    res = []
    x, dA, B, C, gm, bt, th, h0, px, pb = _trap_problem(41, 2, 23, 2, 4, 2, 3, 6, theta=True)
    y, f = oracle.ssd_trapezoidal(x, dA, B, C, gm, bt, th, h0, px, pb, mutation=mutation)
    y2, f2 = chunked_ref.trapezoidal_absorbed(x, dA, B, C, gm, bt, th, h0, px, pb)
    res.append(("trap_absorbed_y", _maxerr(y, y2), 1e-10))
    res.append(("trap_absorbed_final", _maxerr(f, f2), 1e-10))
    return res


def pin_trapezoidal_combined_injection(mutation=0):
    """The moments.rs page's combined injections: the trapezoid is one scalar-decay system with
    2R write channels, x^ = [gamma_t x_t, beta_t x_{t-1}] and b^ = [B_t, R(theta_t) B_{t-1}]
    (the previous write turned by this step's angle), read by the R output channels -- checked
    against the plain oracle with zero C on the extra channels.  Also: beta = 0 and gamma = 1
    is the plain recurrence, and a stream cut in two continues exactly through final_state and
    the last step's (x, B) as the next call's previous write."""
    res = []
    b, T, R, H, G, P, N = 2, 19, 2, 2, 2, 3, 4
    x, dA, B, C, gm, bt, th, h0, px, pb = _trap_problem(43, b, T, R, H, G, P, N, theta=True)
    y, f = oracle.ssd_trapezoidal(x, dA, B, C, gm, bt, th, h0, px, pb, mutation=mutation)
    xp = np.concatenate([px[:, None], x[:, :-1]], axis=1)          # x_{t-1}
    bp = np.concatenate([pb[:, None], B[:, :-1]], axis=1)          # B_{t-1}
    xh = np.concatenate([gm[:, :, None, :, None] * x, bt[:, :, None, :, None] * xp], axis=2)
    # b^ turned by theta_t of each head: expand the groups to heads first
    bph = np.repeat(bp, H // G, axis=3)
    bh = np.concatenate([np.repeat(B, H // G, axis=3),
                         chunked_ref.rotate_pairs(bph, th[:, :, None, :, :])], axis=2)
    ch = np.concatenate([np.repeat(C, H // G, axis=3), np.zeros((b, T, R, H, N))], axis=2)
    y2, f2 = oracle.ssd(xh, dA, bh, ch, th, h0)
    res.append(("combined_injection_y", _maxerr(y, y2[:, :, :R]), 1e-10))
    res.append(("combined_injection_final", _maxerr(f, f2), 1e-10))
    ones, zeros = np.ones_like(gm), np.zeros_like(bt)
    y3, f3 = oracle.ssd_trapezoidal(x, dA, B, C, ones, zeros, th, h0, px, pb, mutation=mutation)
    y4, f4 = oracle.ssd(x, dA, B, C, th, h0)
    res.append(("beta0_gamma1_is_plain", max(_maxerr(y3, y4), _maxerr(f3, f4)), 1e-12))
    k = 8
    sl = lambda a, lo, hi: None if a is None else a[:, lo:hi]
    ya, fa = oracle.ssd_trapezoidal(sl(x, 0, k), sl(dA, 0, k), sl(B, 0, k), sl(C, 0, k),
                                    sl(gm, 0, k), sl(bt, 0, k), sl(th, 0, k), h0, px, pb,
                                    mutation=mutation)
    yb, fb = oracle.ssd_trapezoidal(sl(x, k, T), sl(dA, k, T), sl(B, k, T), sl(C, k, T),
                                    sl(gm, k, T), sl(bt, k, T), sl(th, k, T), fa,
                                    x[:, k - 1], B[:, k - 1], mutation=mutation)
    res.append(("stream_continuation",
                max(_maxerr(np.concatenate([ya, yb], axis=1), y), _maxerr(fb, f)), 1e-12))
    return res


TRAP_PINS = [pin_trapezoidal_rule, pin_trapezoidal_absorbed_frame,
             pin_trapezoidal_combined_injection]


# ------------------------------------------------------------------------- rotation variants
def pin_rotation_variant_reductions(mutation=0):
    """rope_dim = N with interleaved pairs is the plain rotated recurrence (exactly), and the
    split-halves pairing is the interleaved one on a permuted state axis: with the state
    dimensions reordered so that k -> 2k and k + N/2 -> 2k+1, B, C and the initial state
    reordered alike, y is unchanged and the final state is the reordered one."""
    res = []
    x, dA, B, C, th, h0 = _problem(51, 2, 29, 2, 2, 1, 3, 8, theta=True, init=True)
    y, f = oracle.ssd_rotation_variant(x, dA, B, C, th, h0, rope_dim=8, halves=False,
                                       mutation=mutation)
    y0, f0 = oracle.ssd(x, dA, B, C, th, h0)
    res.append(("full_interleaved_is_plain", max(_maxerr(y, y0), _maxerr(f, f0)), 0.0))
    N = 8
    perm = np.empty(N, dtype=int)        # new position of old dimension d
    perm[:N // 2] = 2 * np.arange(N // 2)
    perm[N // 2:] = 2 * np.arange(N // 2) + 1
    inv = np.argsort(perm)               # old dimension at new position
    yh, fh = oracle.ssd_rotation_variant(x, dA, B, C, th, h0, rope_dim=8, halves=True,
                                         mutation=mutation)
    yp, fp = oracle.ssd(x, dA, B[..., inv], C[..., inv], th, h0[..., inv])
    res.append(("halves_is_permuted_interleaved_y", _maxerr(yh, yp), 1e-12))
    res.append(("halves_is_permuted_interleaved_final", _maxerr(fh[..., inv], fp), 1e-12))
    return res


def pin_rope_dim_superposition(mutation=0):
    """With rope_dim < N the state splits into two independent blocks: the first rope_dim
    dimensions turn, the rest follow the unrotated recurrence; y is the sum of the two blocks'
    outputs (C . h splits over the state axis) -- for both pairings."""
    res = []
    Dr = 4
    x, dA, B, C, th, h0 = _problem(53, 1, 31, 2, 2, 2, 3, 10, theta=False, init=True)
    th = _rng(54).uniform(-0.4, 0.4, (1, 31, 2, Dr // 2))
    for halves in (False, True):
        y, f = oracle.ssd_rotation_variant(x, dA, B, C, th, h0, rope_dim=Dr, halves=halves,
                                           mutation=mutation)
        ya, fa = oracle.ssd_rotation_variant(x, dA, B[..., :Dr], C[..., :Dr], th,
                                             h0[..., :Dr], rope_dim=Dr, halves=halves)
        yb, fb = oracle.ssd(x, dA, B[..., Dr:], C[..., Dr:], None, h0[..., Dr:])
        tag = "halves" if halves else "interleaved"
        res.append((f"rope_{tag}_y", _maxerr(y, ya + yb), 1e-12))
        res.append((f"rope_{tag}_final",
                    _maxerr(f, np.concatenate([fa, fb], axis=-1)), 1e-12))
    return res


ROT_PINS = [pin_rotation_variant_reductions, pin_rope_dim_superposition]


# ------------------------------------------------------------------------ quaternion rotation
def _quat_left_matrix(q):
    """4 x 4 matrix of v -> q v (Hamilton product, components (w, x, y, z)), for q [..., 4]."""
    w, x, y, z = (q[..., k] for k in range(4))
    return np.stack([np.stack([w, -x, -y, -z], -1), np.stack([x, w, -z, y], -1),
                     np.stack([y, z, w, -x], -1), np.stack([z, -y, x, w], -1)], -2)


def _unit_quat_walk(seed, shape, step=0.15):
    """Smooth cumulative unit quaternions: a normalised random walk in R^4 (no products)."""
    r = _rng(seed)
    u = np.cumsum(r.normal(0.0, step, shape + (4,)), axis=1)
    u[..., 0] += 1.0
    return u / np.linalg.norm(u, axis=-1, keepdims=True)


def pin_quaternion_reductions(mutation=0):
    """The quaternion form against closed forms: (1) cumulative quaternions cos Phi + i sin Phi
    (Phi the cumulative angle) turn both pairs of each 4-block by the step angle, exactly the
    interleaved angle rotation with each block's angle on its two pairs; (2) with no writes and
    no decay the final state is Q_{T-1} h0 blockwise (the step turns compose to the cumulative
    one), and for Q = cos phi + j sin phi that turns (h0, h2) by +phi and (h1, h3) by -phi (left
    multiplication; on the right the second pair would turn by +phi); the norm of every block
    is preserved."""
    res = []
    x, dA, B, C, _, h0 = _problem(61, 2, 27, 2, 2, 1, 3, 8, init=True)
    th = _rng(62).uniform(-0.4, 0.4, (2, 27, 2, 2))
    Phi = np.cumsum(th, axis=1)
    Q = np.zeros((2, 27, 2, 2, 4))
    Q[..., 0], Q[..., 1] = np.cos(Phi), np.sin(Phi)
    yq, fq = oracle.ssd_quaternion(x, dA, B, C, Q, h0, mutation=mutation)
    ya, fa = oracle.ssd(x, dA, B, C, np.repeat(th, 2, axis=3), h0)
    res.append(("quat_i_axis_is_pairwise_angles", max(_maxerr(yq, ya), _maxerr(fq, fa)), 1e-12))
    T = 11
    z5 = lambda *s: np.zeros(s)
    Qw = _unit_quat_walk(63, (1, T, 1, 2))
    h0 = _rng(64).standard_normal((1, 1, 2, 8))
    _, f = oracle.ssd_quaternion(z5(1, T, 1, 1, 2), z5(1, T, 1), z5(1, T, 1, 1, 8),
                                 z5(1, T, 1, 1, 8), Qw, h0, mutation=mutation)
    L = _quat_left_matrix(Qw[0, T - 1, 0])                     # [2 blocks, 4, 4]
    want = np.einsum("kab,pkb->pka", L, h0[0, 0].reshape(2, 2, 4)).reshape(2, 8)
    res.append(("quat_pure_turn_composes_to_cumulative", _maxerr(f[0, 0], want), 1e-12))
    res.append(("quat_block_norms_preserved",
                _maxerr(np.linalg.norm(f[0, 0].reshape(2, 2, 4), axis=-1),
                        np.linalg.norm(h0[0, 0].reshape(2, 2, 4), axis=-1)), 1e-12))
    phi = 0.7
    Qj = np.zeros((1, 3, 1, 1, 4))
    Qj[..., 0], Qj[..., 2] = math.cos(phi), math.sin(phi)      # constant: one turn at step 0
    hv = np.array([1.0, 2.0, 3.0, 4.0]).reshape(1, 1, 1, 4)
    _, f = oracle.ssd_quaternion(z5(1, 3, 1, 1, 1), z5(1, 3, 1), z5(1, 3, 1, 1, 4),
                                 z5(1, 3, 1, 1, 4), Qj, hv, mutation=mutation)
    c, s = math.cos(phi), math.sin(phi)
    want = [c * 1 - s * 3, c * 2 + s * 4, s * 1 + c * 3, c * 4 - s * 2]
    res.append(("quat_j_axis_left_multiplication", _maxerr(f.reshape(4), want), 1e-13))
    return res


def pin_quaternion_absorbed_frame(mutation=0):
    """The rotation absorbed into B and C (left multiplication is orthogonal, so
    C . (Q g) = (Q^* C) . g): the plain recurrence on B~ = Q_t^* B_t, C~ = Q_t^* C_t per head,
    with the final state turned back by Q_{T-1}, equals the quaternion recurrence (MIMO, a group
    shared by two heads, an initial state)."""
    res = []
    b, T, R, H, G, P, N = 1, 33, 2, 2, 1, 3, 8
    x, dA, B, C, _, h0 = _problem(65, b, T, R, H, G, P, N, init=True, decay=(0.0, 0.2))
    Q = _unit_quat_walk(66, (b, T, H, N // 4))
    y, f = oracle.ssd_quaternion(x, dA, B, C, Q, h0, mutation=mutation)
    Qc = Q * np.array([1.0, -1.0, -1.0, -1.0])
    Lc = _quat_left_matrix(Qc)                                   # [b, T, H, N/4, 4, 4]
    turn = lambda V: np.einsum("bthkij,btrhkj->btrhki", Lc,
                               np.repeat(V, H // G, axis=3).reshape(b, T, R, H, N // 4, 4)
                               ).reshape(b, T, R, H, N)
    yp, g = oracle.ssd(x, dA, turn(B), turn(C), None, h0)
    Lf = _quat_left_matrix(Q[:, T - 1])                          # [b, H, N/4, 4, 4]
    fp = np.einsum("bhkij,bhpkj->bhpki", Lf, g.reshape(b, H, P, N // 4, 4)).reshape(b, H, P, N)
    res.append(("quat_absorbed_frame_y", _maxerr(y, yp), 1e-10))
    res.append(("quat_absorbed_frame_final", _maxerr(f, fp), 1e-10))
    return res


QUAT_PINS = [pin_quaternion_reductions, pin_quaternion_absorbed_frame]


# ------------------------------------------------------------------------------------ backward
def pin_backward_finite_differences(mutation=0):
    """The backward oracle against central differences of the forward oracle: for the loss
    L = <dy, y> + <dfinal, final> and a random direction v of each input, (L(X + eps v) -
    L(X - eps v)) / (2 eps) must equal <dL/dX, v>.  MIMO ranks, a group shared by two heads
    (dB, dC summed over them), an initial state and a length that crosses the oracle's
    64-step recompute checkpoint; once without and once with the rotation (dtheta too)."""
    res = []
    for rot in (False, True):
        x, dA, B, C, th, h0 = _problem(61 + rot, 2, 70, 2, 2, 1, 3, 4, theta=rot, init=True)
        r = _rng(62 + rot)
        dy = r.standard_normal(x.shape)
        dfin = r.standard_normal(h0.shape)
        g = oracle.ssd_backward(x, dA, B, C, dy, h0, dfin, theta=th, mutation=mutation)

        def loss(xx, aa, bb, cc, hh, tt):
            y, f = oracle.ssd(xx, aa, bb, cc, tt, hh)
            return float((dy * y).sum() + (dfin * f).sum())

        args = {"x": x, "ddA": dA, "dB": B, "dC": C, "dinit": h0, "dtheta": th}
        order = ["x", "ddA", "dB", "dC", "dinit", "dtheta"]
        eps = 1e-5
        for name in order:
            if args[name] is None:
                continue
            v = r.standard_normal(args[name].shape)
            plus = [None if args[k] is None else args[k] + (eps * v if k == name else 0)
                    for k in order]
            minus = [None if args[k] is None else args[k] - (eps * v if k == name else 0)
                     for k in order]
            fd = (loss(*plus) - loss(*minus)) / (2 * eps)
            gk = "dx" if name == "x" else name
            an = float((g[gk] * v).sum())
            tag = "rot_" if rot else ""
            res.append((f"fd_{tag}{gk}", abs(fd - an) / (1.0 + abs(fd)), 1e-7))
    return res


def pin_trapezoidal_backward_finite_differences(mutation=0):
    """The trapezoidal backward oracle against central differences of the trapezoidal forward
    oracle along a random direction of each input (x, dA, B, C, gamma, beta, theta, init,
    prev_x, prev_B): MIMO ranks, a group shared by two heads, the rotation, a previous write and
    a length that crosses the 64-step recompute checkpoint."""
    res = []
    x, dA, B, C, gm, bt, th, h0, px, pb = _trap_problem(71, 2, 70, 2, 2, 1, 3, 4, theta=True)
    r = _rng(72)
    dy = r.standard_normal(x.shape)
    dfin = r.standard_normal(h0.shape)
    g = oracle.ssd_trap_backward(x, dA, B, C, gm, bt, dy, theta=th, init_state=h0, prev_x=px,
                                 prev_B=pb, dfinal=dfin, mutation=mutation)

    def loss(xx, aa, bb, cc, gg, be, tt, hh, pxx, pbb):
        y, f = oracle.ssd_trapezoidal(xx, aa, bb, cc, gg, be, tt, hh, pxx, pbb)
        return float((dy * y).sum() + (dfin * f).sum())

    names = ["dx", "ddA", "dB", "dC", "dgamma", "dbeta", "dtheta", "dinit", "dprev_x", "dprev_B"]
    vals = [x, dA, B, C, gm, bt, th, h0, px, pb]
    eps = 1e-5
    for i, name in enumerate(names):
        v = r.standard_normal(vals[i].shape)
        plus = [vals[k] + (eps * v if k == i else 0) for k in range(len(vals))]
        minus = [vals[k] - (eps * v if k == i else 0) for k in range(len(vals))]
        fd = (loss(*plus) - loss(*minus)) / (2 * eps)
        an = float((g[name] * v).sum())
        res.append((f"fd_trap_{name}", abs(fd - an) / (1.0 + abs(fd)), 1e-7))
    return res


def pin_trapezoidal_backward_reduces_to_plain(mutation=0):
    """beta = 0, gamma = 1 and no previous write make the trapezoidal recurrence the plain
    rotated one, so its reverse mode must give the plain reverse mode's gradients (two
    separately written reverse modes agreeing), with and without the rotation."""
    res = []
    for rot in (False, True):
        x, dA, B, C, _, bt, th, h0, _, _ = _trap_problem(81 + rot, 2, 70, 2, 2, 1, 3, 4,
                                                         theta=rot, prev=False)
        gm, bt = np.ones_like(bt), np.zeros_like(bt)
        r = _rng(83 + rot)
        dy = r.standard_normal(x.shape)
        dfin = r.standard_normal(h0.shape)
        gt = oracle.ssd_trap_backward(x, dA, B, C, gm, bt, dy, theta=th, init_state=h0,
                                      dfinal=dfin, mutation=mutation)
        gp = oracle.ssd_backward(x, dA, B, C, dy, h0, dfin, theta=th)
        for k in ("dx", "ddA", "dB", "dC", "dinit") + (("dtheta",) if rot else ()):
            tag = "rot_" if rot else ""
            res.append((f"trap_as_plain_{tag}{k}", _maxerr(gt[k], gp[k]), 1e-10))
    return res


def pin_backward_chunked_algebra(mutation=0):
    """The sequential reverse mode against the chunked backward algebra (the per-chunk formulas
    the GPU kernels use, restated in numpy fp64 in chunked_ref): ragged T, MIMO ranks, a group
    shared by two heads, an initial state and dfinal, at several chunk lengths."""
    res = []
    x, dA, B, C, _, h0 = _problem(91, 2, 37, 2, 4, 2, 3, 4, init=True)
    r = _rng(92)
    dy = r.standard_normal(x.shape)
    dfin = r.standard_normal(h0.shape)
    g = oracle.ssd_backward(x, dA, B, C, dy, h0, dfin, mutation=mutation)
    for l in (1, 8, 16, 37):
        ref = chunked_ref.chunked_backward(x, dA, B, C, dy, h0, dfin, chunk_len=l)
        for k in ("dx", "ddA", "dB", "dC", "dinit"):
            res.append((f"chunked_bwd_l{l}_{k}", _maxerr(g[k], ref[k]), 1e-9))
    return res


def pin_rotated_backward_chunk_local_frames(mutation=0):
    """The sequential rotated reverse mode against the chunk-local-frame restatement
    (chunked_ref.chunked_backward_rotated, the form the GPU uses): ragged T, MIMO ranks, a
    group shared by two differently turned heads, at several chunk lengths."""
    res = []
    x, dA, B, C, th, h0 = _problem(93, 2, 37, 2, 4, 2, 3, 4, theta=True, init=True)
    r = _rng(94)
    dy = r.standard_normal(x.shape)
    dfin = r.standard_normal(h0.shape)
    g = oracle.ssd_backward(x, dA, B, C, dy, h0, dfin, theta=th, mutation=mutation)
    for l in (1, 8, 16, 37):
        ref = chunked_ref.chunked_backward_rotated(x, dA, B, C, th, dy, h0, dfin, chunk_len=l)
        for k in ("dx", "ddA", "dB", "dC", "dtheta", "dinit"):
            res.append((f"rot_chunked_bwd_l{l}_{k}", _maxerr(g[k], ref[k]), 1e-9))
    return res


BWD_PINS = [pin_backward_finite_differences, pin_backward_chunked_algebra,
            pin_rotated_backward_chunk_local_frames]
def pin_trapezoidal_backward_expansion(mutation=0):
    """The sequential trapezoidal reverse mode against the 2R-channel expansion, its chunked
    backward and the chain rule back through it (chunked_ref.trapezoidal_backward_expanded, the
    form the GPU uses), with and without the rotation, with a previous write."""
    res = []
    for rot in (False, True):
        x, dA, B, C, gm, bt, th, h0, px, pb = _trap_problem(95 + rot, 2, 37, 2, 4, 2, 3, 4,
                                                            theta=rot)
        r = _rng(97 + rot)
        dy = r.standard_normal(x.shape)
        dfin = r.standard_normal(h0.shape)
        g = oracle.ssd_trap_backward(x, dA, B, C, gm, bt, dy, theta=th, init_state=h0,
                                     prev_x=px, prev_B=pb, dfinal=dfin, mutation=mutation)
        for l in (8, 37):
            ref = chunked_ref.trapezoidal_backward_expanded(x, dA, B, C, gm, bt, dy, theta=th,
                                                            init_state=h0, prev_x=px, prev_B=pb,
                                                            dfinal=dfin, chunk_len=l)
            for k in sorted(g):
                tag = "rot_" if rot else ""
                res.append((f"trap_expanded_{tag}l{l}_{k}", _maxerr(g[k], ref[k]), 1e-9))
    return res


TRAP_BWD_PINS = [pin_trapezoidal_backward_finite_differences,
                 pin_trapezoidal_backward_reduces_to_plain,
                 pin_trapezoidal_backward_expansion]

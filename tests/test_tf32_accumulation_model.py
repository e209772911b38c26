"""Would the fp32 path meet its 1e-4 gate on the tensor core?  A CPU model, checked against the
fp64 oracle.

The fp32-input chunk products (CB = C B^T, (L o CB) x, B^T (dec o x), C h^T) can run as
tcgen05 kind::tf32 MMAs with each fp32 operand split into a tf32 high part and a tf32 remainder
(three products: hi*hi + hi*lo + lo*hi).  A chain of kind::tf32 MMAs measured on the GPU against
fp64 put nearly all of its errors toward zero, so the model here adds each group of exact
products into an fp32 accumulator rounded toward zero.  The chunked algorithm (scan.py page: the
rotation absorbed into B and C; serial.rs page: K1..K5 with the state passed between chunks in
fp32) is run with every product under that model, and y and the final state are compared with
the oracle under the fp32 gate |got - ref| <= 1e-4 (1 + |ref|).

Findings pinned here, on the slow-decay inputs with an initial state (long memory, the hard case):
  * plain tf32 (one product) misses the gate by orders of magnitude;
  * three products into one accumulator over the whole K (256 rows of a chunk) miss it too;
  * three products with a fresh accumulator per 32-deep K block, the block sums added in fp32
    round-to-nearest, meet it;
  * the order of the three products matters: with the two small correction products issued
    first the accumulator truncates at their magnitude, and only the hi*hi steps truncate at the
    block's own, which leaves a clearly smaller error than hi*hi first (the library's tf32 chunk
    scan, ssd_chunked_forward_tf32, issues them in that order).
"""
import numpy as np

import oracle
from chunked_ssd_scan_gb300 import workloads as wl

TOL = 1e-4


def _tf32(a):
    """Round fp32 to the 10 explicit mantissa bits of tf32 (to nearest, ties away from zero)."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    return ((u + np.uint32(0x1000)) & np.uint32(0xFFFFE000)).view(np.float32)


def _to_f32_toward_zero(v):
    f = v.astype(np.float32)
    over = np.abs(f.astype(np.float64)) > np.abs(v)
    f[over] = np.nextafter(f[over], np.float32(0))
    return f


def _matmul(a, b, products, kblock, small_first=False, group=8):
    """a [M, K] @ b [K, N] of fp32 operands: `products` tf32 products per pair of `group`-deep K
    groups (1: hi*hi; 3: + hi*lo + lo*hi, with small_first the two corrections before hi*hi),
    accumulated toward zero in fp32; a fresh accumulator per `kblock` of K (0: the whole K), the
    block sums added in fp32 round-to-nearest."""
    a = a.astype(np.float32)
    b = b.astype(np.float32)
    ah, bh = _tf32(a), _tf32(b)
    al, bl = _tf32(a - ah), _tf32(b - bh)
    terms = [(ah, bh)] if products == 1 else [(ah, bh), (ah, bl), (al, bh)]
    if small_first and products == 3:
        terms = terms[1:] + terms[:1]
    k = a.shape[1]
    kblock = kblock or k
    out = np.zeros((a.shape[0], b.shape[1]), np.float32)
    for k0 in range(0, k, kblock):
        acc = np.zeros_like(out)
        for x, y in terms:
            for ks in range(k0, min(k0 + kblock, k), group):
                s = x[:, ks:ks + group].astype(np.float64) @ y[ks:ks + group, :].astype(np.float64)
                acc = _to_f32_toward_zero(acc.astype(np.float64) + s)
        out = (out + acc).astype(np.float32)
    return out


def _chunked_forward(inp, chunk, products, kblock, **kw):
    """One head, batch 1, rank 1: the chunked forward with every product under the model."""
    x = inp["x"].numpy()[0, :, 0, 0].astype(np.float32)
    dA = inp["dA"].numpy()[0, :, 0].astype(np.float64)
    B = inp["B"].numpy()[0, :, 0, 0].astype(np.float32)
    C = inp["C"].numpy()[0, :, 0, 0].astype(np.float32)
    phi = np.cumsum(inp["theta"].numpy()[0, :, 0].astype(np.float64), axis=0)
    T, P = x.shape
    cs, sn = np.cos(phi), np.sin(phi)

    def turn(v):   # each pair (2k, 2k+1) turned by -Phi_t
        v = v.astype(np.float64)
        o = np.empty_like(v)
        o[:, 0::2] = cs * v[:, 0::2] + sn * v[:, 1::2]
        o[:, 1::2] = -sn * v[:, 0::2] + cs * v[:, 1::2]
        return o.astype(np.float32)

    Bt, Ct = turn(B), turn(C)
    g = inp["init_state"].numpy()[0, 0].astype(np.float32)
    mm = lambda a, b: _matmul(a, b, products, kblock, **kw)
    y = np.zeros((T, P), np.float32)
    for c0 in range(0, T, chunk):
        c1 = min(T, c0 + chunk)
        cum = np.cumsum(dA[c0:c1])
        Bc, Cc, xc = Bt[c0:c1], Ct[c0:c1], x[c0:c1]
        mask = np.tril(np.exp(cum[:, None] - cum[None, :])).astype(np.float32)
        M = (mask * mm(Cc, Bc.T)).astype(np.float32)
        y_off = np.exp(cum)[:, None].astype(np.float32) * mm(Cc, g.T)
        y[c0:c1] = (mm(M, xc) + y_off).astype(np.float32)
        dec = np.exp(cum[-1] - cum).astype(np.float32)
        g = (np.float32(np.exp(cum[-1])) * g + mm((dec[:, None] * xc).T, Bc)).astype(np.float32)
    c, s = np.cos(phi[-1]), np.sin(phi[-1])
    g64 = g.astype(np.float64)
    fin = np.empty_like(g64)
    fin[:, 0::2] = c * g64[:, 0::2] - s * g64[:, 1::2]
    fin[:, 1::2] = s * g64[:, 0::2] + c * g64[:, 1::2]
    return y, fin


def _worst_over_bound(got, ref):
    return float((np.abs(got - ref) / (TOL * (1.0 + np.abs(ref)))).max())


def test_three_tf32_products_need_short_k_blocks():
    cfg = wl.SSDConfig("tf32_model", 1, 2048, 1, 64, 64, 256, 1, 1, "f32", theta=True)
    inp = wl.make_ssd_inputs(cfg, seed=0, slow_decay=True, init_state=True)
    yr, fr = oracle.ssd(*(None if inp[k] is None else inp[k].numpy()
                          for k in ("x", "dA", "B", "C", "theta", "init_state")))
    yr, fr = yr[0, :, 0, 0], fr[0, 0]
    worst = {}
    for name, products, kblock in (("tf32", 1, 0), ("3xtf32_fullK", 3, 0), ("3xtf32_K32", 3, 32)):
        y, fin = _chunked_forward(inp, cfg.chunk_len, products, kblock)
        worst[name] = max(_worst_over_bound(y, yr), _worst_over_bound(fin, fr))
    assert worst["tf32"] > 50.0, worst
    assert worst["3xtf32_fullK"] > 1.0, worst
    assert worst["3xtf32_K32"] < 0.8, worst


def test_correction_products_first_shrink_the_truncation_error():
    """The same 3 x tf32, 32-deep-block arithmetic with the accumulator truncating after every
    two products (a pessimistic reading of the hardware's grouping): issuing hi*lo and lo*hi
    before hi*hi leaves a clearly smaller worst error than hi*hi first."""
    cfg = wl.SSDConfig("tf32_order", 1, 1024, 1, 64, 64, 256, 1, 1, "f32", theta=True)
    inp = wl.make_ssd_inputs(cfg, seed=3, slow_decay=True, init_state=True)
    yr, fr = oracle.ssd(*(None if inp[k] is None else inp[k].numpy()
                          for k in ("x", "dA", "B", "C", "theta", "init_state")))
    yr, fr = yr[0, :, 0, 0], fr[0, 0]
    worst = {}
    for name, first in (("hi_first", False), ("small_first", True)):
        y, fin = _chunked_forward(inp, 128, 3, 32, small_first=first, group=2)
        worst[name] = max(_worst_over_bound(y, yr), _worst_over_bound(fin, fr))
    assert worst["small_first"] < 0.7 * worst["hi_first"], worst

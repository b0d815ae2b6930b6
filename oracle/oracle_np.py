"""Independent NumPy oracle for low-bit KV-cache quantization and decode attention.

TEST INFRASTRUCTURE ONLY: imported by the tests, the smoke check and the
benchmark's CPU baseline, never by the product package. It is written
separately from the C++ oracle (``kvq_oracle.cpp``) so that the two can check
each other; they share nothing but the definitions below.

Definitions (KV Cache量化技术介绍, developer.horizon.auto/blog/13163):
  * KVQuant, "Per-Channel Key Quantization": keys get one scale and zero-point
    per channel, here over each completed block of ``Bk`` tokens.
  * KVQuant, "Pre-RoPE Key Quantization": keys are quantized before RoPE;
    RoPE is applied to the dequantized keys when attention reads them.
  * KVQuant, "Per-Vector Dense-and-Sparse Quantization": the largest-|x|
    elements of each token vector are kept as fp16 (index, value) pairs and
    left out of the dense statistics.
  * Quanto, steps 1-2: block-wise quantization; every block keeps a scale and a
    zero_point to restore its values (the formula image is lost on the page).
  * KVQuant, "Non-Uniform KV Cache Quantization": codes index a calibrated
    table of levels instead of a uniform grid.
Readings taken where the page is silent (they match the C++ oracle):
  q = clamp(rint_half_even(fp32(fp32(x - z) / s)), 0, 2^b - 1), z = block min
  (fp16, -0 stored as +0), s = fp16_round_up(fp32(fp32(max - min) / (2^b - 1))),
  x_hat = q*s + z; s = 0 gives codes 0; an all-outlier group has s = z = 0.
  With a level table 0 = l_0 < ... < l_L = 1: r = fp16_round_up(fp32(max) -
  fp32(min)) in the scale's slot, u = fp32(fp32(x - z) / r), q = the number of
  binary32 midpoints fp32(0.5 (l_k + l_k+1)) below u (nearest level, ties to
  the lower), x_hat = z + r * l_q. Tables come from 1-D k-means (Lloyd) on
  normalized calibration values, end levels held at 0 and 1.
"""
from __future__ import annotations

import numpy as np

__all__ = [
    "half_up", "select_outliers", "group_params", "quantize", "pack_rows",
    "unpack_rows", "encode", "dequant", "rope", "attention",
    "group_params_levels", "quantize_levels", "fit_levels",
]


def half_up(x):
    """Round binary32 values toward +infinity to binary16 (x >= 0, finite)."""
    x = np.asarray(x, dtype=np.float32)
    h = x.astype(np.float16)                       # round to nearest
    low = h.astype(np.float32) < x
    with np.errstate(over="ignore"):
        h = np.where(low, np.nextafter(h, np.float16(np.inf)), h)
    return h.astype(np.float16)


def select_outliers(x, n_out):
    """Per row of ``x`` (fp16, [..., D]): indices of the n_out largest |x|.

    Ties go to the lower index; slots are in descending |x| then ascending
    index (a stable sort on -|x|).
    """
    x = np.asarray(x, dtype=np.float16)
    mag = np.abs(x.astype(np.float64))
    order = np.argsort(-mag, axis=-1, kind="stable")[..., :n_out]
    vals = np.take_along_axis(x, order, axis=-1)
    return order.astype(np.uint16), vals


def group_params(x, excluded, bits, axis):
    """Scale and zero of the groups of ``x`` along ``axis`` (fp16 in/out).

    ``excluded`` marks outlier elements, which the statistics skip.
    """
    L = (1 << bits) - 1
    xf = x.astype(np.float32)
    big = np.float32(np.inf)
    mn = np.where(excluded, big, xf).min(axis=axis)
    mx = np.where(excluded, -big, xf).max(axis=axis)
    empty = np.all(excluded, axis=axis)
    with np.errstate(invalid="ignore"):
        rng = (mx - mn).astype(np.float32)
        s = half_up(np.where(empty, np.float32(0), rng / np.float32(L)))
    z = np.where(empty, np.float32(0), mn).astype(np.float16)
    z = np.where(z == 0, np.float16(0), z)          # -0 -> +0
    return s, z


def quantize(x, s, z, bits):
    """Codes clamp(rint((x - z)/s), 0, L) with binary32 steps; s == 0 -> 0."""
    L = (1 << bits) - 1
    xf = np.asarray(x, dtype=np.float16).astype(np.float32)
    sf = np.asarray(s, dtype=np.float16).astype(np.float32)
    zf = np.asarray(z, dtype=np.float16).astype(np.float32)
    with np.errstate(invalid="ignore", divide="ignore"):
        d = (xf - zf).astype(np.float32)
        r = (d / sf).astype(np.float32)
        q = np.clip(np.rint(r), 0, L)
    q = np.where(sf == 0, 0, q)
    return q.astype(np.uint8)


def group_params_levels(x, excluded, axis):
    """Range r = fp16_round_up(fp32(max - min)) and zero z of the groups of
    ``x`` along ``axis``, for a level table (fp16 in/out)."""
    xf = x.astype(np.float32)
    big = np.float32(np.inf)
    mn = np.where(excluded, big, xf).min(axis=axis)
    mx = np.where(excluded, -big, xf).max(axis=axis)
    empty = np.all(excluded, axis=axis)
    with np.errstate(invalid="ignore"):
        r = half_up(np.where(empty, np.float32(0), (mx - mn).astype(np.float32)))
    z = np.where(empty, np.float32(0), mn).astype(np.float16)
    z = np.where(z == 0, np.float16(0), z)
    return r, z


def quantize_levels(x, r, z, levels):
    """Nearest level of u = fp32(fp32(x - z) / r): the count of binary32
    midpoints below u; r == 0 -> 0."""
    lv = np.asarray(levels, dtype=np.float32)
    mids = ((lv[:-1] + lv[1:]) * np.float32(0.5)).astype(np.float32)
    xf = np.asarray(x, dtype=np.float16).astype(np.float32)
    rf = np.asarray(r, dtype=np.float16).astype(np.float32)
    zf = np.asarray(z, dtype=np.float16).astype(np.float32)
    with np.errstate(invalid="ignore", divide="ignore"):
        u = ((xf - zf).astype(np.float32) / rf).astype(np.float32)
    q = (u[..., None] > mids).sum(axis=-1)
    return np.where(rf == 0, 0, q).astype(np.uint8)


def fit_levels(u, bits, iters=100):
    """1-D k-means of samples u in [0, 1] into 2^bits levels: start at k / L,
    hold l_0 = 0 and l_L = 1, move each interior level to the mean of the
    samples nearest to it (ties to the lower level; a level without samples
    stays); binary64, returned as binary32."""
    u = np.asarray(u, dtype=np.float64).ravel()
    L = (1 << bits) - 1
    lv = np.arange(L + 1, dtype=np.float64) / L
    for _ in range(iters):
        mids = 0.5 * (lv[:-1] + lv[1:])
        cell = np.searchsorted(mids, u, side="left")          # number of midpoints strictly below u
        cnt = np.bincount(cell, minlength=L + 1)
        tot = np.bincount(cell, weights=u, minlength=L + 1)
        inner = np.arange(1, L)
        has = cnt[inner] > 0
        lv[inner[has]] = tot[inner[has]] / cnt[inner[has]]
    return lv.astype(np.float32)


def pack_rows(codes, bits):
    """LSB-first bitstream per row: element d at bits [b*d, b*d + b)."""
    codes = np.asarray(codes, dtype=np.uint8)
    shp = codes.shape
    planes = (codes[..., None] >> np.arange(bits, dtype=np.uint8)) & 1   # [..., D, b]
    stream = planes.reshape(*shp[:-1], shp[-1] * bits)
    return np.packbits(stream, axis=-1, bitorder="little")


def unpack_rows(rows, D, bits):
    stream = np.unpackbits(np.asarray(rows, dtype=np.uint8), axis=-1, bitorder="little")
    stream = stream[..., : D * bits].reshape(*rows.shape[:-1], D, bits).astype(np.uint8)
    return (stream << np.arange(bits, dtype=np.uint8)).sum(axis=-1).astype(np.uint8)


def _outlier_mask(idx, D):
    mask = np.zeros(idx.shape[:-1] + (D,), dtype=bool)
    if idx.shape[-1]:
        np.put_along_axis(mask, idx.astype(np.int64), True, axis=-1)
    return mask


def encode(K, V, bits, Bk, Gv, n_out, levels=None, window=None):
    """Encode streams K, V of shape [P, T, D] (fp16). Returns a dict of arrays
    laid out like the C++ oracle's outputs. ``levels``: a level table
    (non-uniform codes) or None (uniform grid). ``window``: sliding-window
    key statistics (page mlqm.cn/news/1064729 §3.2, "滑动窗口统计": the scale
    and zero come from the most recent `window` tokens only): the (s, z) of
    key block b and channel c are those of the dense elements of channel c in
    tokens [max(0, (b + 1) Bk - window), (b + 1) Bk); the block's codes use
    them. None (or window = Bk) is the per-block statistics."""
    K = np.asarray(K, dtype=np.float16)
    V = np.asarray(V, dtype=np.float16)
    P, T, D = K.shape
    ng = D // Gv
    nb = T // Bk

    # Values: outliers per token, then one (s, z) per token and group.
    vi, vv = select_outliers(V, n_out)
    vmask = _outlier_mask(vi, D)
    Vg = V.reshape(P, T, ng, Gv)
    if levels is None:
        vs, vz = group_params(Vg, vmask.reshape(P, T, ng, Gv), bits, axis=-1)
        vq = quantize(Vg, vs[..., None], vz[..., None], bits).reshape(P, T, D)
    else:
        vs, vz = group_params_levels(Vg, vmask.reshape(P, T, ng, Gv), axis=-1)
        vq = quantize_levels(Vg, vs[..., None], vz[..., None], levels).reshape(P, T, D)

    # Keys: completed blocks only; one (s, z) per block and channel.
    Kb = K[:, : nb * Bk].reshape(P, nb, Bk, D)
    ki, kv = select_outliers(Kb, n_out)
    kmask = _outlier_mask(ki, D)
    if levels is not None and window is not None and window != Bk:
        raise ValueError("window statistics are defined for the uniform grid")
    if levels is None and window is not None and window != Bk:
        if window % Bk or window < Bk:
            raise ValueError("window: a positive multiple of the key block")
        Kt = K[:, : nb * Bk]
        tmask = kmask.reshape(P, nb * Bk, D)
        ks = np.zeros((P, nb, D), np.float16)
        kz = np.zeros((P, nb, D), np.float16)
        for b in range(nb):                                          # the window ending with block b
            lo = max(0, (b + 1) * Bk - window)
            ks[:, b], kz[:, b] = group_params(Kt[:, lo:(b + 1) * Bk], tmask[:, lo:(b + 1) * Bk], bits, axis=1)
        kq = quantize(Kb, ks[:, :, None, :], kz[:, :, None, :], bits).reshape(P, nb * Bk, D)
    elif levels is None:
        ks, kz = group_params(Kb, kmask, bits, axis=2)              # [P, nb, D]
        kq = quantize(Kb, ks[:, :, None, :], kz[:, :, None, :], bits).reshape(P, nb * Bk, D)
    else:
        ks, kz = group_params_levels(Kb, kmask, axis=2)
        kq = quantize_levels(Kb, ks[:, :, None, :], kz[:, :, None, :], levels).reshape(P, nb * Bk, D)

    rb = D * bits // 8
    k_codes = np.zeros((P, T, rb), dtype=np.uint8)
    k_codes[:, : nb * Bk] = pack_rows(kq, bits)
    k_outl = np.zeros((P, T, n_out, 2), dtype=np.uint16)
    k_outl[:, : nb * Bk, :, 0] = ki.reshape(P, nb * Bk, n_out)
    k_outl[:, : nb * Bk, :, 1] = kv.reshape(P, nb * Bk, n_out).view(np.uint16)
    k_tail = np.zeros((P, Bk, D), dtype=np.float16)
    k_tail[:, : T - nb * Bk] = K[:, nb * Bk:]
    v_outl = np.stack([vi, vv.view(np.uint16)], axis=-1)
    return {
        "k_codes": k_codes,
        "k_meta": np.stack([ks.view(np.uint16), kz.view(np.uint16)], axis=-1),
        "k_tail": k_tail,
        "k_outl": k_outl,
        "v_codes": pack_rows(vq, bits),
        "v_meta": np.stack([vs.view(np.uint16), vz.view(np.uint16)], axis=-1),
        "v_outl": v_outl,
    }


def dequant(enc, T, D, bits, Bk, Gv, n_out, levels=None):
    """x_hat = q*s + z (with a level table: z + r * l_q) in float64, outliers
    restored, tail keys as fp16."""
    P = enc["v_codes"].shape[0]
    ng = D // Gv
    nb = T // Bk
    step = (lambda q: q.astype(np.float64)) if levels is None else (
        lambda q: np.asarray(levels, dtype=np.float32).astype(np.float64)[q])
    vq = step(unpack_rows(enc["v_codes"], D, bits)).reshape(P, T, ng, Gv)
    vmeta = enc["v_meta"].view(np.float16).astype(np.float64)
    Vh = (vq * vmeta[..., 0:1] + vmeta[..., 1:2]).reshape(P, T, D)
    Kh = np.empty((P, T, D), dtype=np.float64)
    kq = step(unpack_rows(enc["k_codes"][:, : nb * Bk], D, bits)).reshape(P, nb, Bk, D)
    kmeta = enc["k_meta"].view(np.float16).astype(np.float64)          # [P, nb, D, 2]
    Kh[:, : nb * Bk] = (kq * kmeta[:, :, None, :, 0] + kmeta[:, :, None, :, 1]).reshape(P, nb * Bk, D)
    Kh[:, nb * Bk:] = enc["k_tail"][:, : T - nb * Bk].astype(np.float64)
    for arr, outl, upto in ((Vh, enc["v_outl"], T), (Kh, enc["k_outl"], nb * Bk)):
        if n_out and upto:
            idx = outl[:, :upto, :, 0].astype(np.int64)
            val = outl[:, :upto, :, 1].view(np.float16).astype(np.float64)
            np.put_along_axis(arr[:, :upto], idx, val, axis=-1)
    return Kh, Vh


def rope(x, pos, theta):
    """Rotate-half RoPE: pairs (i, i + D/2), angle pos * theta^(-2i/D), float64."""
    x = np.asarray(x, dtype=np.float64)
    D = x.shape[-1]
    h = D // 2
    inv = theta ** (-2.0 * np.arange(h, dtype=np.float64) / D)
    phi = np.asarray(pos, dtype=np.float64)[..., None] * inv
    c, s = np.cos(phi), np.sin(phi)
    a, b = x[..., :h], x[..., h:]
    return np.concatenate([a * c - b * s, b * c + a * s], axis=-1)


def attention(Kh, Vh, q, q_pos, theta, sm_scale, pos_offset=0.0):
    """Exact softmax attention: Kh, Vh [P, T, D] float64, q [P, G, D] fp16."""
    P, T, D = Kh.shape
    qd = np.asarray(q, dtype=np.float16).astype(np.float64)
    pos = np.arange(T, dtype=np.float64) + pos_offset
    if theta > 0:
        Kr = rope(Kh, pos[None, :], theta)
        qr = rope(qd, np.full(qd.shape[:-1], q_pos + pos_offset), theta)
    else:
        Kr, qr = Kh, qd
    sc = sm_scale * np.einsum("pgd,ptd->pgt", qr, Kr)
    sc = sc - sc.max(axis=-1, keepdims=True)
    p = np.exp(sc)
    return np.einsum("pgt,ptd->pgd", p, Vh) / p.sum(axis=-1)[..., None]

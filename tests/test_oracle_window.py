"""Pins of the oracle's sliding-window key statistics (no GPU).

Page mlqm.cn/news/1064729 ("UltraQuant ..."), §3.2 "时空自适应量化", names
sliding-window statistics: the scale and zero come from a recent fixed-size
window of tokens (for example the last 1024) instead of the whole sequence.
The oracle's reading: the (s, z) of key block b and channel c are the group
parameters of that channel's dense elements in tokens
[max(0, (b + 1) Bk - W), (b + 1) Bk). These tests check that reading against
a brute-force search written from it (outlier sets by a plain sort, window
min and max by a loop, the scale against the fp16 value table, the codes
against all levels), against its special cases (W = Bk is the per-block rule,
values on one grid round-trip exactly) and the error bound, for both oracles.
"""
from fractions import Fraction

import numpy as np
import pytest

from oracle import oracle_cpp as oc
from oracle import oracle_np as on
import kvq_inputs as ki

ALL_HALF = np.arange(0, 0x7C00, dtype=np.uint16).view(np.float16)
ALL_HALF_F64 = ALL_HALF.astype(np.float64)


def _streams(T, seed, bits=4, Bk=64, Gv=64, frac=0.01):
    w = ki.Workload("win", 1, 8, 2, 128, T, bits, Bk, Gv, frac, 5e5, seed)
    K, V = ki.streams_np(w, [(0, 0), (0, 1)], T)
    return w, K, V


def _encode_both(K, V, bits, Bk, Gv, n_out, window):
    a = oc.encode(K, V, bits, Bk, Gv, n_out, window=window)
    b = on.encode(K, V, bits, Bk, Gv, n_out, window=window)
    for name in a:
        assert np.array_equal(np.asarray(a[name]).view(np.uint8), np.asarray(b[name]).view(np.uint8)), name
    return a


@pytest.mark.parametrize("bits,Bk", [(4, 64), (3, 128), (2, 64)])
def test_window_of_one_block_is_the_block_rule(bits, Bk):
    w, K, V = _streams(3 * Bk + 17, 41, bits, Bk, 32)
    plain = oc.encode(K, V, bits, Bk, 32, 1)
    win = _encode_both(K, V, bits, Bk, 32, 1, Bk)
    for name in plain:
        assert np.array_equal(np.asarray(plain[name]).view(np.uint8), np.asarray(win[name]).view(np.uint8)), name


def _outlier_channels(x, n_out):
    """Brute force: the n_out channels of largest |x| (ties to the lower channel)."""
    mags = [(-abs(float(v)), c) for c, v in enumerate(x)]
    return {c for _, c in sorted(mags)[:n_out]}


@pytest.mark.parametrize("bits,Bk,W", [(4, 64, 256), (3, 64, 1024), (2, 128, 384), (8, 64, 192)])
def test_window_params_and_codes_brute_force(bits, Bk, W):
    L = (1 << bits) - 1
    n_out = 1
    T = 6 * Bk + 9
    w, K, V = _streams(T, 50 + bits, bits, Bk, 64)
    # a drifting channel: the window statistics differ from the block's
    K[:, :, 5] += np.linspace(0, 40, T).astype(np.float16)
    enc = _encode_both(K, V, bits, Bk, 64, n_out, W)
    nb = T // Bk
    meta = enc["k_meta"].view(np.float16).astype(np.float64)          # [P, nb, D, 2]
    codes = on.unpack_rows(enc["k_codes"][:, : nb * Bk], 128, bits)
    rng = np.random.default_rng(bits)
    for p in range(2):
        outl = [_outlier_channels(K[p, t], n_out) for t in range(nb * Bk)]
        for b in range(nb):
            lo = max(0, (b + 1) * Bk - W)
            for c in list(rng.choice(128, 12, replace=False)) + [5]:
                dense = [float(K[p, t, c]) for t in range(lo, (b + 1) * Bk) if c not in outl[t]]
                if not dense:
                    assert meta[p, b, c, 0] == 0 and meta[p, b, c, 1] == 0
                    continue
                m, M = min(dense), max(dense)
                assert meta[p, b, c, 1] == (m if m != 0 else 0.0)
                q = np.float32(np.float32(np.float32(M) - np.float32(m)) / np.float32(L))
                s_want = ALL_HALF_F64[np.searchsorted(ALL_HALF_F64, float(q), side="left")]
                assert meta[p, b, c, 0] == s_want
                S, Z = Fraction(s_want), Fraction(meta[p, b, c, 1])
                for t in range(b * Bk, (b + 1) * Bk):
                    if c in outl[t] or S == 0:
                        continue
                    X = Fraction(float(K[p, t, c]))
                    ratio = (X - Z) / S
                    assert 0 <= ratio <= L * (1 + Fraction(1, 2 ** 20))    # inside the window's range
                    dist = [abs(X - (k * S + Z)) for k in range(L + 1)]
                    best = min(dist)
                    if abs(ratio - (int(ratio) + Fraction(1, 2))) > Fraction(1, 2 ** 18):
                        assert codes[p, t, c] == dist.index(best), (p, b, c, t)


def test_window_grid_round_trip():
    """Every key of a channel on one grid z + q s, with 0 and L in the first
    block: the window statistics are that grid's, and x_hat == x."""
    bits, Bk, W, L = 4, 64, 256, 15
    T = 8 * Bk
    rng = np.random.default_rng(3)
    s = 2.0 ** -rng.integers(2, 6, size=128)
    z = -s * rng.integers(0, 64, size=128)
    q = rng.integers(0, L + 1, size=(1, T, 128))
    q[0, 0], q[0, 1] = 0, L
    K = (z + q * s).astype(np.float16)
    assert np.array_equal(K.astype(np.float64), z + q * s)                    # exact fp16 values
    V = rng.standard_normal((1, T, 128)).astype(np.float16)
    enc = _encode_both(K, V, bits, Bk, 64, 0, W)
    Kh, _ = oc.dequant(enc, T, 128, bits, Bk, 64, 0)
    assert np.array_equal(Kh, K.astype(np.float64))
    meta = enc["k_meta"].view(np.float16).astype(np.float64)
    assert np.all(meta[0, :, :, 0] == s) and np.all(meta[0, :, :, 1] == z)


@pytest.mark.parametrize("W", [128, 1024])
def test_window_error_bound_and_outliers(W):
    bits, Bk = 3, 64
    T = 10 * Bk + 3
    w, K, V = _streams(T, 60, bits, Bk, 32)
    enc = _encode_both(K, V, bits, Bk, 32, 1, W)
    Kh, _ = oc.dequant(enc, T, 128, bits, Bk, 32, 1)
    nb = T // Bk
    s = np.repeat(enc["k_meta"].view(np.float16).astype(np.float64)[..., 0], Bk, axis=1)   # [P, nb*Bk, D]
    err = np.abs(Kh[:, : nb * Bk] - K[:, : nb * Bk].astype(np.float64))
    outl = np.zeros(err.shape, bool)
    np.put_along_axis(outl, enc["k_outl"][:, : nb * Bk, :, 0].astype(np.int64), True, axis=-1)
    assert np.all(err[outl] == 0)                                             # outliers restored exactly
    assert np.all(err[~outl] <= s[~outl] * (0.5 + 2.0 ** -20))
    # a wider window never gives a smaller scale than the block's own
    plain = oc.encode(K, V, bits, Bk, 32, 1)
    sp = plain["k_meta"].view(np.float16).astype(np.float64)[..., 0]
    sw = enc["k_meta"].view(np.float16).astype(np.float64)[..., 0]
    assert np.all(sw >= sp)

"""Pins of the oracle's non-uniform codes (KVQuant "Non-Uniform KV Cache
Quantization"): a calibrated table of 2^b levels on each group's normalized
range replaces the uniform grid (no GPU needed).

The level fit is checked against planted clusters and against the k-means
fixed-point property; the codes against a brute-force nearest-level search;
dequantization against values placed exactly on the levels and against the
half-gap error bound; and the C++ and NumPy oracles against each other.
"""
import numpy as np
import pytest

from fractions import Fraction

from oracle import oracle_cpp as oc
from oracle import oracle_np as on
import kvq_inputs as ki

ALL_HALF = np.arange(0, 0x7C00, dtype=np.uint16).view(np.float16)   # every finite fp16 >= 0
ALL_HALF_F64 = ALL_HALF.astype(np.float64)


def _nearest_level(u, levels):
    """Brute force: index of the level closest to u (float64), ties to the lower."""
    lv = np.asarray(levels, dtype=np.float64)
    d = np.abs(np.asarray(u, dtype=np.float64)[..., None] - lv)
    return np.argmin(d, axis=-1)       # argmin returns the first (lower) index on ties


def _range_pin_holds(x, r, z):
    """The stored range of a level-table group: r is the smallest binary16
    value at or above fp32(max) - fp32(min) (found in the table of all fp16
    values), and the levels span the group: z + r >= max, exactly."""
    d32 = np.float32(np.float32(x.max()) - np.float32(x.min()))
    want = ALL_HALF[np.searchsorted(ALL_HALF_F64, float(d32), side="left")]
    if r.view(np.uint16) != want.view(np.uint16):
        return False
    return Fraction(float(z)) + Fraction(float(r)) >= Fraction(float(x.max()))


def test_range_rounds_up_against_value_table():
    """Range r of a level-table group (KVQuant "Non-Uniform KV Cache
    Quantization": the levels sit on the group's normalized range, so the top
    level must reach the maximum)."""
    rng = np.random.default_rng(31)
    rn_would_fail = 0
    for trial in range(400):
        n = int(rng.integers(2, 80))
        x = (rng.standard_normal(n) * np.exp(rng.uniform(-8, 6))).astype(np.float16)
        if trial % 4 == 0:                       # a spread that is not an fp16 value
            x[0] = np.float16(np.float16(1.0) + np.float16(2.0 ** -10) * rng.integers(1, 9))
            x[1] = np.float16(-np.float16(2.0 ** -rng.integers(3, 12)))
        r, z = oc.group_params_levels(x)
        r2, z2 = on.group_params_levels(x[None], np.zeros((1, n), bool), axis=-1)
        assert r.view(np.uint16) == r2[0].view(np.uint16) and z.view(np.uint16) == z2[0].view(np.uint16)
        assert z.view(np.uint16) == (x.min() if x.min() != 0 else np.float16(0)).view(np.uint16)
        assert _range_pin_holds(x, r, z), (x, r, z)
        # the same pin rejects a range rounded to nearest wherever that rounds down
        d32 = np.float32(np.float32(x.max()) - np.float32(x.min()))
        r_rn = d32.astype(np.float16)
        if float(r_rn) < float(d32):
            rn_would_fail += 1
            assert not _range_pin_holds(x, r_rn, z)
    assert rn_would_fail > 50


@pytest.mark.parametrize("bits", [2, 3, 4])
def test_fit_recovers_planted_clusters(bits):
    L = (1 << bits) - 1
    rng = np.random.default_rng(bits)
    # interior centres moved off the uniform grid but inside their starting cells
    centres = (np.arange(1, L) + rng.uniform(-0.3, 0.3, L - 1)) / L
    u = np.concatenate([c + rng.normal(0, 2e-4, 4000) for c in centres] + [np.zeros(500), np.ones(500)])
    for fit in (oc.fit_levels, on.fit_levels):
        lv = fit(np.clip(u, 0, 1), bits, 50)
        assert lv[0] == 0 and lv[-1] == 1
        np.testing.assert_allclose(lv[1:-1], centres, atol=2e-5)


@pytest.mark.parametrize("bits", [2, 3, 4])
def test_fit_is_a_kmeans_fixed_point(bits):
    u = np.random.default_rng(10 + bits).beta(2.0, 5.0, 20000)
    lv = oc.fit_levels(u, bits, 400).astype(np.float64)
    assert np.all(np.diff(lv) > 0)
    cell = _nearest_level(u, lv)
    for k in range(1, len(lv) - 1):
        members = u[cell == k]
        assert len(members) > 0
        assert abs(members.mean() - lv[k]) < 1e-6          # binary32 rounding of the level


@pytest.mark.parametrize("bits", [2, 3, 4, 8])
def test_codes_are_the_nearest_level(bits):
    rng = np.random.default_rng(20 + bits)
    lv = oc.fit_levels(rng.beta(2.0, 3.0, 5000), bits, 60)
    mids = ((lv[:-1] + lv[1:]) * np.float32(0.5)).astype(np.float32)
    for trial in range(40):
        x = (rng.standard_normal(64) * rng.uniform(0.1, 30)).astype(np.float16)
        r, z = oc.group_params_levels(x)
        r2, z2 = on.group_params_levels(x[None], np.zeros((1, 64), bool), axis=-1)
        assert r.view(np.uint16) == r2[0].view(np.uint16) and z.view(np.uint16) == z2[0].view(np.uint16)
        u = ((x.astype(np.float32) - np.float32(z)).astype(np.float32) / np.float32(r)).astype(np.float32)
        codes = oc.quantize_levels(x, r, z, bits, lv)
        assert np.array_equal(codes, on.quantize_levels(x, r, z, lv).astype(np.int32))
        # away from the binary32-rounded midpoints the nearest level is unambiguous
        clear = np.min(np.abs(u.astype(np.float64)[:, None] - mids.astype(np.float64)), axis=1) > 1e-6
        assert np.array_equal(codes[clear], _nearest_level(u[clear], lv))
        assert codes.min() >= 0 and codes.max() <= (1 << bits) - 1


def test_values_on_the_levels_round_trip_exactly():
    # dyadic levels and a power-of-two range: x = z + r * l_k is an fp16 value
    # and u = l_k exactly, so every code is k and x_hat == x
    lv = np.array([0, 1 / 16, 3 / 16, 5 / 16, 1 / 2, 11 / 16, 7 / 8, 1], dtype=np.float32)
    z, r = -1.0, 2.0
    x = (z + r * lv.astype(np.float64)[np.arange(64) % 8]).astype(np.float16)
    rr, zz = oc.group_params_levels(x)
    assert float(rr) == r and float(zz) == z
    assert np.array_equal(oc.quantize_levels(x, rr, zz, 3, lv), np.arange(64) % 8)
    K = np.tile(x[None, :, None], (1, 1, 64)).astype(np.float16)[:, :64, :]   # each channel: the 64 values
    V = np.tile(x[None, None, :], (1, 64, 1)).astype(np.float16)
    enc = oc.encode(K, V, 3, 64, 64, 0, levels=lv)
    Kh, Vh = oc.dequant(enc, 64, 64, 3, 64, 64, 0, levels=lv)
    assert np.array_equal(Vh, np.broadcast_to(x.astype(np.float64), Vh.shape))
    assert np.array_equal(Kh, K.astype(np.float64))


@pytest.mark.parametrize("bits,Bk,Gv,n_out", [(4, 64, 64, 1), (3, 128, 32, 1), (2, 64, 32, 2)])
def test_error_bound_outliers_and_oracles_agree(bits, Bk, Gv, n_out):
    w = ki.WORKLOADS["gqa8b"].replace(B=1, H_kv=2, H_q=8)
    K, V = ki.streams_np(w, [(0, 0), (0, 1)], 2 * Bk + 7)
    T, D = K.shape[1], K.shape[2]
    # calibration: normalized dense values of a uniform encoding of other tokens
    Kc, Vc = ki.streams_np(w, [(0, 0)], 512, layer=1)
    u = (Vc - Vc.min(axis=-1, keepdims=True)) / (Vc.max(axis=-1, keepdims=True) - Vc.min(axis=-1, keepdims=True))
    lv = oc.fit_levels(u.astype(np.float64).ravel(), bits, 80)
    enc = oc.encode(K, V, bits, Bk, Gv, n_out, levels=lv)
    enc_np = on.encode(K, V, bits, Bk, Gv, n_out, levels=lv)
    for name in enc:
        assert np.array_equal(np.asarray(enc[name]).view(np.uint8), np.asarray(enc_np[name]).view(np.uint8)), name
    Kh, Vh = oc.dequant(enc, T, D, bits, Bk, Gv, n_out, levels=lv)
    Kh2, Vh2 = on.dequant(enc_np, T, D, bits, Bk, Gv, n_out, levels=lv)
    assert np.array_equal(Kh, Kh2) and np.array_equal(Vh, Vh2)
    half_gap = float(np.max(np.diff(lv.astype(np.float64)))) / 2
    vmeta = enc["v_meta"].view(np.float16).astype(np.float64)                 # [P, T, ng, 2]
    r = np.repeat(vmeta[..., 0], Gv, axis=-1)                                  # per element
    outl = np.zeros(V.shape, bool)
    np.put_along_axis(outl, enc["v_outl"][..., 0].astype(np.int64), True, axis=-1)
    err = np.abs(Vh - V.astype(np.float64))
    assert np.all(err[~outl] <= r[~outl] * (half_gap + 1e-6) + 1e-12)
    assert np.all(err[outl] == 0)                                              # outliers restored exactly

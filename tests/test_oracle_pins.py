"""Pins of the CPU oracle to facts outside itself (no GPU needed).

Each test checks one oracle step against something the method or mathematics
fixes: values on the quantization grid, the rounding error bound, brute force
over all levels, a brute-force sort, the IEEE binary16 value table, the
textbook 2-D rotation, the textbook softmax, and closed-form special cases of
attention. Both oracles (C++ and NumPy) are checked, and they are checked
against each other.
"""
from fractions import Fraction
import os

import numpy as np
import pytest

from oracle import oracle_cpp as oc
from oracle import oracle_np as on
import kvq_inputs as ki

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
ALL_HALF = np.arange(0, 0x7C00, dtype=np.uint16).view(np.float16)   # every finite fp16 >= 0
ALL_HALF_F64 = ALL_HALF.astype(np.float64)


def _brute_half_up(x32: np.float32) -> np.float16:
    """Smallest binary16 value >= x, by search in the table of all values."""
    i = np.searchsorted(ALL_HALF_F64, float(x32), side="left")
    return ALL_HALF[i]


# -------------------------------------------------------------- binary16 steps
def test_half_up_against_value_table():
    rng = np.random.default_rng(7)
    xs = np.concatenate([
        rng.uniform(0, 4, 3000), np.exp(rng.uniform(-20, 10, 3000)),
        ALL_HALF_F64[rng.integers(1, len(ALL_HALF), 500)],            # exact fp16 values
        [0.0, 2.0 ** -24, 2.0 ** -25, 2.0 ** -14, 65504.0, 1.0 + 2.0 ** -23],
    ]).astype(np.float32)
    for x in xs:
        want = _brute_half_up(x)
        assert oc.half_up(x).view(np.uint16) == want.view(np.uint16), x
        assert on.half_up(x).view(np.uint16) == want.view(np.uint16), x


def test_half_decode_exact():
    # every finite binary16 pattern decodes to numpy's value (numpy's float16
    # is the IEEE binary16 type)
    pats = np.concatenate([np.arange(0, 0x7C00), np.arange(0x8000, 0xFC00)]).astype(np.uint16)
    for p in pats[:: 37]:
        assert oc.half_to_double(p.view(np.float16)) == float(p.view(np.float16))


# -------------------------------------------------------------- grid round trip
@pytest.mark.parametrize("bits", [2, 3, 4, 8])
def test_grid_round_trip_values_and_keys(bits):
    """Values already on the grid z + q*s come back exactly (codes, s, z, x)."""
    L = (1 << bits) - 1
    rng = np.random.default_rng(bits)
    P, T, D, Bk, Gv = 2, 128, 64, 64, 32
    # s = 2^-e, z a multiple of s with small magnitude, so z + q*s is exact in fp16
    Qv = rng.integers(0, L + 1, size=(P, T, D))
    for g in range(D // Gv):                          # each value group sees 0 and L
        Qv[:, :, g * Gv] = 0
        Qv[:, :, g * Gv + 1] = L
    Qk = rng.integers(0, L + 1, size=(P, T, D))
    for blk in range(T // Bk):                        # each key block/channel too
        Qk[:, blk * Bk, :] = 0
        Qk[:, blk * Bk + 1, :] = L
    s_v = 2.0 ** -rng.integers(2, 6, size=(P, T, D // Gv))
    z_v = rng.integers(-8, 8, size=(P, T, D // Gv)) * s_v
    V = (z_v.repeat(Gv, -1) + Qv * s_v.repeat(Gv, -1)).astype(np.float16)
    assert np.array_equal(V.astype(np.float64), z_v.repeat(Gv, -1) + Qv * s_v.repeat(Gv, -1))
    s_k = 2.0 ** -rng.integers(2, 6, size=(P, T // Bk, 1, D))
    z_k = rng.integers(-8, 8, size=(P, T // Bk, 1, D)) * s_k
    K = (z_k + Qk.reshape(P, T // Bk, Bk, D) * s_k).reshape(P, T, D).astype(np.float16)
    for orc in (oc, on):
        enc = orc.encode(K, V, bits, Bk, Gv, 0)
        vm = enc["v_meta"].view(np.float16).astype(np.float64)
        assert np.array_equal(vm[..., 0], s_v)
        assert np.array_equal(vm[..., 1], z_v)
        km = enc["k_meta"].view(np.float16).astype(np.float64)
        assert np.array_equal(km[..., 0], s_k[:, :, 0])
        assert np.array_equal(km[..., 1], z_k[:, :, 0])
        assert np.array_equal(on.unpack_rows(enc["v_codes"], D, bits), Qv)
        assert np.array_equal(on.unpack_rows(enc["k_codes"], D, bits), Qk)
        Kh, Vh = orc.dequant(enc, T, D, bits, Bk, Gv, 0)
        assert np.array_equal(Kh, K.astype(np.float64))
        assert np.array_equal(Vh, V.astype(np.float64))


# -------------------------------------------------------------- error bound
@pytest.mark.parametrize("bits,Bk,Gv,n_out", [(4, 64, 64, 1), (3, 128, 32, 1), (2, 128, 32, 2), (4, 64, 32, 0),
                                             (8, 64, 64, 1)])
def test_error_bound_and_outliers_exact(bits, Bk, Gv, n_out):
    """|x - x_hat| <= s/2 + 2^-20 (M - m) on dense elements; outliers exact."""
    w = ki.WORKLOADS["gqa8b"]
    T, D = 2 * Bk + 17, 128
    K = np.stack([ki.keys_np(w, 0, 0, h, 0, T) for h in range(2)])
    V = np.stack([ki.values_np(w, 0, 0, h, 0, T) for h in range(2)])
    for orc in (oc, on):
        enc = orc.encode(K, V, bits, Bk, Gv, n_out)
        Kh, Vh = orc.dequant(enc, T, D, bits, Bk, Gv, n_out)
        # values
        vm = enc["v_meta"].view(np.float16).astype(np.float64)
        s = vm[..., 0].repeat(Gv, -1)
        outm = np.zeros(V.shape, bool)
        if n_out:
            np.put_along_axis(outm, enc["v_outl"][..., 0].astype(np.int64), True, -1)
        Vg = np.where(outm, np.nan, V.astype(np.float64)).reshape(2, T, D // Gv, Gv)
        rng_ = (np.nanmax(Vg, -1) - np.nanmin(Vg, -1)).repeat(Gv, -1)
        err = np.abs(Vh - V.astype(np.float64))
        assert np.all(err[~outm] <= (s / 2 + 2.0 ** -20 * rng_)[~outm])
        assert np.all(err[outm] == 0)
        # keys (completed blocks)
        nb = T // Bk
        km = enc["k_meta"].view(np.float16).astype(np.float64)
        sk = np.repeat(km[..., 0], Bk, axis=1)
        koutm = np.zeros((2, nb * Bk, D), bool)
        if n_out:
            np.put_along_axis(koutm, enc["k_outl"][:, : nb * Bk, :, 0].astype(np.int64), True, -1)
        Kb = np.where(koutm, np.nan, K[:, : nb * Bk].astype(np.float64)).reshape(2, nb, Bk, D)
        krng = np.repeat(np.nanmax(Kb, 2) - np.nanmin(Kb, 2), Bk, axis=1)
        kerr = np.abs(Kh[:, : nb * Bk] - K[:, : nb * Bk].astype(np.float64))
        assert np.all(kerr[~koutm] <= (sk / 2 + 2.0 ** -20 * krng)[~koutm])
        assert np.all(kerr[koutm] == 0)
        # tail keys are the fp16 inputs
        assert np.array_equal(Kh[:, nb * Bk:], K[:, nb * Bk:].astype(np.float64))


# -------------------------------------------------------------- brute force codes
@pytest.mark.parametrize("bits", [2, 3, 4, 8])
def test_codes_brute_force(bits):
    """The code is the nearest level (ties to even), unless fp32 rounding sits on a tie."""
    L = (1 << bits) - 1
    rng = np.random.default_rng(100 + bits)
    checked = 0
    for trial in range(60):
        n = int(rng.integers(2, 40))
        x = (rng.standard_normal(n) * np.exp(rng.uniform(-6, 3))).astype(np.float16)
        s, z = oc.group_params(x, bits)
        s2, z2 = on.group_params(x[None], np.zeros((1, n), bool), bits, axis=-1)
        assert s.view(np.uint16) == s2[0].view(np.uint16) and z.view(np.uint16) == z2[0].view(np.uint16)
        assert z == x.min() or (x.min() == 0 and z == 0)
        Mx = Fraction(float(x.max()))
        # s rounds (M - z)/L up: the top level covers the maximum, within one fp32 rounding
        assert Fraction(float(z)) + L * Fraction(float(s)) >= Mx * (1 - Fraction(1, 2 ** 22)) - Fraction(1, 2 ** 40)
        codes = oc.quantize(x, s, z, bits)
        assert np.array_equal(codes, on.quantize(x, s, z, bits).astype(np.int32))
        if s == 0:
            assert np.all(codes == 0)
            continue
        S, Z = Fraction(float(s)), Fraction(float(z))
        for xi, qi in zip(x, codes):
            X = Fraction(float(xi))
            dist = [abs(X - (k * S + Z)) for k in range(L + 1)]
            best = min(dist)
            cands = [k for k in range(L + 1) if dist[k] == best]
            want = cands[0] if len(cands) == 1 else [k for k in cands if k % 2 == 0][0]
            ratio = (X - Z) / S
            near_tie = abs(ratio - (int(ratio) + Fraction(1, 2))) <= Fraction(1, 2 ** 18)
            if near_tie:
                assert qi in cands or abs(qi - want) == 1
            else:
                assert qi == want, (xi, s, z, qi, want)
            checked += 1
    assert checked > 500


def test_constant_group_and_all_outlier_group():
    x = np.full(16, 0.375, np.float16)
    for bits in (2, 3, 4):
        s, z = oc.group_params(x, bits)
        assert s == 0 and z == np.float16(0.375)
        assert np.all(oc.quantize(x, s, z, bits) == 0)
        s, z = oc.group_params(x, bits, excluded=np.ones(16, np.uint8))
        assert s == 0 and z == 0 and z.view(np.uint16) == 0
    # -0 and +0 minimum store +0
    s, z = oc.group_params(np.array([-0.0, 1.0, 0.0], np.float16), 4)
    assert z.view(np.uint16) == 0
    # a key channel that is the outlier of every token of its block
    T, D, Bk = 64, 64, 64
    K = np.ones((1, T, D), np.float16)
    K[0, :, 5] = 100.0
    V = np.ones((1, T, D), np.float16)
    for orc in (oc, on):
        enc = orc.encode(K, V, 4, Bk, 64, 1)
        km = enc["k_meta"].view(np.uint16)
        assert km[0, 0, 5, 0] == 0 and km[0, 0, 5, 1] == 0
        Kh, _ = orc.dequant(enc, T, D, 4, Bk, 64, 1)
        assert np.array_equal(Kh, K.astype(np.float64))


# -------------------------------------------------------------- outliers
def test_outlier_selection_brute_force():
    rng = np.random.default_rng(3)
    for trial in range(200):
        D = int(rng.choice([8, 64, 128]))
        x = rng.integers(-6, 7, size=D).astype(np.float16) * np.float16(0.5)   # many ties, +-0
        n_out = int(rng.integers(0, 4))
        mags = [abs(float(v)) for v in x]
        want = sorted(range(D), key=lambda i: (-mags[i], i))[:n_out]
        idx, val = oc.select_outliers(x, n_out)
        assert list(idx) == want
        assert np.array_equal(val.view(np.uint16), x[want].view(np.uint16))
        idx2, val2 = on.select_outliers(x[None], n_out)
        assert list(idx2[0]) == want
        assert np.array_equal(val2[0].view(np.uint16), x[want].view(np.uint16))


def test_no_outliers_is_plain_group_quantization():
    rng = np.random.default_rng(11)
    V = rng.standard_normal((1, 64, 64)).astype(np.float16)
    enc = oc.encode(V, V, 4, 64, 32, 0)
    for t in range(64):
        for g in range(2):
            s, z = oc.group_params(V[0, t, 32 * g: 32 * g + 32], 4)
            assert enc["v_meta"][0, t, g, 0] == s.view(np.uint16)
            assert enc["v_meta"][0, t, g, 1] == z.view(np.uint16)


# -------------------------------------------------------------- packing
def _golden_pack():
    rows = []
    with open(os.path.join(GOLDEN, "pack_lsb_first.txt")) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                b, codes, want = (p.strip() for p in line.split("|"))
                rows.append((int(b), [int(c) for c in codes.split()], bytes.fromhex(want.replace(" ", ""))))
    return rows


@pytest.mark.parametrize("bits,codes,want", _golden_pack())
def test_pack_golden(bits, codes, want):
    assert bytes(oc.pack_row(np.array(codes), bits)) == want
    assert bytes(on.pack_rows(np.array([codes], np.uint8), bits)[0]) == want
    assert list(on.unpack_rows(np.frombuffer(want, np.uint8)[None], len(codes), bits)[0]) == codes


# -------------------------------------------------------------- RoPE
def test_rope_is_the_textbook_rotation():
    rng = np.random.default_rng(5)
    for _ in range(20):
        x = rng.standard_normal(2)
        pos = float(rng.integers(0, 10 ** 6))
        # D = 2: one pair, frequency theta^0 = 1, angle = pos
        R = np.array([[np.cos(pos), -np.sin(pos)], [np.sin(pos), np.cos(pos)]])
        for y in (oc.rope(x, pos, 1e4), on.rope(x, pos, 1e4)):
            np.testing.assert_allclose(y, R @ x, rtol=0, atol=1e-12)
    # D = 4, theta = 1e4: pairs (0, 2) at angle pos and (1, 3) at pos / 100
    x = np.array([1.0, 2.0, 3.0, 4.0])
    pos = 7.0
    a, b = pos, pos / 100.0
    want = np.array([1 * np.cos(a) - 3 * np.sin(a), 2 * np.cos(b) - 4 * np.sin(b),
                     3 * np.cos(a) + 1 * np.sin(a), 4 * np.cos(b) + 2 * np.sin(b)])
    np.testing.assert_allclose(oc.rope(x, pos, 1e4), want, atol=1e-14)
    np.testing.assert_allclose(on.rope(x, pos, 1e4), want, atol=1e-14)


def test_rope_norm_and_composition():
    rng = np.random.default_rng(6)
    x = rng.standard_normal(128)
    y = oc.rope(x, 1234.0, 5e5)
    assert abs(np.linalg.norm(y) - np.linalg.norm(x)) < 1e-12
    np.testing.assert_allclose(oc.rope(oc.rope(x, 1000.0, 5e5), 234.0, 5e5), y, atol=1e-11)


# -------------------------------------------------------------- attention
def _rand_cache(rng, P, T, D):
    return rng.standard_normal((P, T, D)), rng.standard_normal((P, T, D))


def test_attention_theta0_is_textbook_softmax():
    from scipy.special import softmax
    rng = np.random.default_rng(8)
    P, T, D, G = 2, 37, 16, 3
    Kh, Vh = _rand_cache(rng, P, T, D)
    q = rng.standard_normal((P, G, D)).astype(np.float16)
    sc = 0.3
    want = np.einsum("pgt,ptd->pgd", softmax(sc * np.einsum("pgd,ptd->pgt", q.astype(np.float64), Kh), axis=-1), Vh)
    np.testing.assert_allclose(oc.attention(Kh, Vh, q, T - 1, 0.0, sc), want, atol=1e-12)
    np.testing.assert_allclose(on.attention(Kh, Vh, q, T - 1, 0.0, sc), want, atol=1e-12)


def test_attention_special_cases():
    rng = np.random.default_rng(9)
    P, T, D, G = 2, 50, 32, 2
    Kh, Vh = _rand_cache(rng, P, T, D)
    q = rng.standard_normal((P, G, D)).astype(np.float16)
    for orc in (oc, on):
        # one token: the output is that token's value
        out = orc.attention(Kh[:, :1], Vh[:, :1], q, 0, 1e4, 0.2)
        np.testing.assert_allclose(out, np.repeat(Vh[:, :1], G, 1), atol=1e-15)
        # q = 0: uniform weights, the output is the mean of the values
        out = orc.attention(Kh, Vh, np.zeros_like(q), T - 1, 1e4, 0.2)
        np.testing.assert_allclose(out, np.repeat(Vh.mean(1, keepdims=True), G, 1), atol=1e-13)
        # values all one: softmax rows sum to one
        out = orc.attention(Kh, np.ones_like(Vh), q, T - 1, 1e4, 0.2)
        np.testing.assert_allclose(out, 1.0, atol=1e-12)
        # RoPE depends only on relative position: shift every position by 1000
        a = orc.attention(Kh, Vh, q, T - 1, 1e4, 0.2)
        b = orc.attention(Kh, Vh, q, T - 1, 1e4, 0.2, pos_offset=1000.0)
        np.testing.assert_allclose(a, b, atol=1e-9)


# -------------------------------------------------------------- two oracles agree
@pytest.mark.parametrize("name", ["tiny_mha", "gqa8b", "int3", "int2"])
def test_cpp_and_numpy_oracles_agree(name):
    w = ki.WORKLOADS[name]
    T = min(w.T, 3 * w.key_block + 21)
    n_out = 0 if w.outlier_frac == 0 else max(1, int(w.outlier_frac * w.D))
    P = min(w.H_kv, 3)
    K = np.stack([ki.keys_np(w, 0, 0, h, 0, T) for h in range(P)])
    V = np.stack([ki.values_np(w, 0, 0, h, 0, T) for h in range(P)])
    e1 = oc.encode(K, V, w.bits, w.key_block, w.value_group, n_out)
    e2 = on.encode(K, V, w.bits, w.key_block, w.value_group, n_out)
    for k in e1:
        assert np.array_equal(np.asarray(e1[k]).view(np.uint8), np.asarray(e2[k]).view(np.uint8)), k
    Kh, Vh = oc.dequant(e1, T, w.D, w.bits, w.key_block, w.value_group, n_out)
    Kh2, Vh2 = on.dequant(e2, T, w.D, w.bits, w.key_block, w.value_group, n_out)
    assert np.array_equal(Kh, Kh2) and np.array_equal(Vh, Vh2)
    q = ki.queries_np(w, 0, 0)[0, : P * w.G].reshape(P, w.G, w.D)
    a = oc.attention(Kh, Vh, q, T - 1, w.rope_theta, 1 / np.sqrt(w.D))
    b = on.attention(Kh, Vh, q, T - 1, w.rope_theta, 1 / np.sqrt(w.D))
    np.testing.assert_allclose(a, b, atol=1e-12)


def test_generator_numpy_and_torch_agree():
    torch = pytest.importorskip("torch")
    w = ki.WORKLOADS["gqa8b"].replace(B=2, H_kv=2, H_q=8, T=200)
    K, V = ki.kv_torch(w, 1, 100, 50, "cpu")
    for b in range(2):
        for h in range(2):
            assert np.array_equal(K[b, h].numpy().view(np.uint16), ki.keys_np(w, 1, b, h, 100, 50).view(np.uint16))
            assert np.array_equal(V[b, h].numpy().view(np.uint16), ki.values_np(w, 1, b, h, 100, 50).view(np.uint16))
    assert np.array_equal(ki.queries_torch(w, 0, 3, "cpu").numpy().view(np.uint16), ki.queries_np(w, 0, 3).view(np.uint16))

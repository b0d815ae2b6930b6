"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle.

Codes, scales, zeros, tails and outlier lists must match bit for bit; decode
attention must be within 2e-3 max-abs and 1e-2 relative (2-norm) of the
oracle's float64 attention on its own encoding of the same fp16 inputs.
"""
import math

import numpy as np
import pytest
import torch

import bit_quantized_kv_append_gb300 as kvq
from bit_quantized_kv_append_gb300 import build as kbuild
import kvq_inputs as ki
import kvq_testlib as tl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available(), "the gpu tests need a CUDA device"
    kbuild.build()
    kvq.lib()


W = ki.Workload
SMALL = {
    # name: (workload, T, append pieces)
    "tiny_mha": (ki.WORKLOADS["tiny_mha"], 512, [512]),
    "tiny_mha_pieces": (ki.WORKLOADS["tiny_mha"], 505, [1, 62, 1, 64, 65, 130, 1, 1, 100, 80]),
    "mha_rope_tail": (W("mha", 2, 4, 4, 128, 1000, 4, 64, 64, 0.0, 1e4, 2), 1000, [1000]),
    "gqa_outliers_deferred_tail": (W("gqa", 2, 8, 2, 128, 777, 4, 64, 64, 0.01, 5e5, 3), 777,
                                   [100, 300, 1, 376]),
    "int3_bk128_gv32": (W("int3", 1, 8, 2, 128, 700, 3, 128, 32, 0.01, 5e5, 4), 700, [700]),
    "int2_pieces": (W("int2", 1, 8, 2, 128, 700, 2, 128, 32, 0.01, 5e5, 4), 700, [129, 127, 1, 443]),
    "d64_g2_two_outliers": (W("d64", 2, 4, 2, 64, 333, 3, 64, 32, 0.04, 1e4, 6), 333, [333]),
    "g8_gv128": (W("g8", 1, 16, 2, 128, 300, 4, 64, 128, 0.01, 5e5, 7), 300, [300]),
    "g1_d64_int2_norope": (W("g1", 3, 2, 2, 64, 200, 2, 128, 64, 0.0, 0.0, 8), 200, [200]),
    # 8-bit codes (decode on the CUDA-core kernel at both head dims)
    "int8_gqa_outliers": (W("int8", 2, 8, 2, 128, 300, 8, 64, 64, 0.01, 5e5, 41), 300, [130, 1, 169]),
    "int8_d64_bk128_gv32": (W("int8d64", 1, 4, 2, 64, 260, 8, 128, 32, 0.0, 1e4, 42), 260, [260]),
}


def _run_small(w, T, pieces, q_positions=None):
    T_max = (T // w.key_block + 1) * w.key_block
    cache = tl.make_cache(w, T_max)
    K, V = ki.kv_torch(w, 0, 0, T, "cuda")
    tl.append_pieces(cache, K, V, pieces)
    assert cache.T_cur == T
    streams = [(b, h) for b in range(w.B) for h in range(w.H_kv)]
    Kh, Vh = tl.host_streams(w, streams, T)
    assert np.array_equal(Kh.view(np.uint16), K.cpu().numpy().reshape(-1, T, w.D).view(np.uint16))
    enc = tl.oracle_encode(w, Kh, Vh)
    tl.sync()
    tl.compare_streams(cache, streams, enc, T)
    q = ki.queries_torch(w, 0, 0, "cuda")
    qn = q.cpu().numpy()
    for q_pos in (q_positions or [T - 1]):
        out = cache.decode(q, q_pos=q_pos).cpu().numpy()
        ref = tl.oracle_decode(w, enc, T, tl.q_of_streams(qn, w, streams), q_pos)
        got = tl.q_of_streams(out, w, streams)
        tl.check_decode(got, ref, f"q_pos={q_pos}")


@pytest.mark.parametrize("name", list(SMALL))
def test_small_parity(name):
    w, T, pieces = SMALL[name]
    _run_small(w, T, pieces, q_positions=[T - 1, T // 3, 0])


def test_generator_on_device_matches_host():
    w = ki.WORKLOADS["gqa8b"].replace(B=2, H_kv=2, H_q=8)
    K, V = ki.kv_torch(w, 3, 1000, 300, "cuda")
    for b in range(2):
        for h in range(2):
            assert np.array_equal(K[b, h].cpu().numpy().view(np.uint16), ki.keys_np(w, 3, b, h, 1000, 300).view(np.uint16))
            assert np.array_equal(V[b, h].cpu().numpy().view(np.uint16), ki.values_np(w, 3, b, h, 1000, 300).view(np.uint16))
    assert np.array_equal(ki.queries_torch(w, 0, 5, "cuda").cpu().numpy().view(np.uint16),
                          ki.queries_np(w, 0, 5).view(np.uint16))


@pytest.mark.parametrize("T", [1, 63, 64, 65, 127, 128, 129])
def test_token_by_token_block_edges(T):
    w = W("edge", 1, 4, 2, 128, T, 4, 64, 64, 0.01, 1e4, 11)
    _run_small(w, T, [1] * T, q_positions=[T - 1])


def test_single_token_returns_its_value():
    w = W("one", 1, 2, 2, 128, 1, 4, 64, 64, 0.0, 1e4, 12)
    cache = tl.make_cache(w, 64)
    K, V = ki.kv_torch(w, 0, 0, 1, "cuda")
    cache.append(K, V)
    out = cache.decode(ki.queries_torch(w, 0, 0, "cuda")).float().cpu().numpy()
    v_hat = tl.oracle_decode(w, tl.oracle_encode(w, *tl.host_streams(w, [(0, 0), (0, 1)], 1)), 1,
                             np.zeros((2, 1, 128), np.float16), 0)
    np.testing.assert_allclose(out[0], v_hat[:, 0], atol=1e-3)


def _planted_inputs(w, T):
    rng = np.random.default_rng(5)
    K = rng.standard_normal((w.B, w.H_kv, T, w.D)).astype(np.float16)
    V = rng.standard_normal((w.B, w.H_kv, T, w.D)).astype(np.float16)
    K[0, 0, :64, 7] = 300.0                     # channel 7: the outlier of every token of block 0
    V[0, 0, 5, :] = 0.5                         # constant value vector: s = 0 in both groups
    V[0, 0, 6, :32] = -0.0                      # -0 minimum
    V[0, 1, 7, :] = np.float16(2.0 ** -20)      # subnormal
    V[0, 1, 8, :] = np.float16(6e-5) * np.arange(w.D)
    K[0, 1, 64:128, 3] = 60000.0                # huge magnitudes
    K[0, 1, 64:128, 4] = -60000.0
    V[0, 0, 9, 10] = 65504.0
    V[0, 0, 9, 11] = -65504.0
    K[0, 1, 130:140, :] = 0.0                   # all-zero keys
    return K, V


@pytest.mark.parametrize("bits", [4, 8])
def test_planted_degenerate_groups(bits):
    w = W("planted", 1, 4, 2, 128, 200, bits, 64, 64, 0.01, 1e4, 13)
    T = 200
    K, V = _planted_inputs(w, T)
    cache = tl.make_cache(w, 256)
    cache.append(torch.from_numpy(K).cuda(), torch.from_numpy(V).cuda())
    streams = [(0, 0), (0, 1)]
    enc = tl.oracle_encode(w, K[0], V[0])
    assert enc["k_meta"][0, 0, 7, 0] == 0 and enc["k_meta"][0, 0, 7, 1] == 0   # all-outlier channel
    tl.sync()
    tl.compare_streams(cache, streams, enc, T)
    q = ki.queries_torch(w, 0, 0, "cuda")
    out = cache.decode(q).cpu().numpy()
    ref = tl.oracle_decode(w, enc, T, tl.q_of_streams(q.cpu().numpy(), w, streams), T - 1)
    # fp16 values up to 65504 in V: compare relative to the value range
    got = tl.q_of_streams(out, w, streams).astype(np.float64)
    assert np.linalg.norm(got - ref) / np.linalg.norm(ref) < 1e-2


def test_int8_value_ties():
    """8-bit value groups whose quotients (x - z) / s are exact half-integers:
    min 0 and max 255/16 give s = 1/16 exactly, so x = (k + 1/2)/16 sits on a
    rounding tie (ties to the even code)."""
    w = W("ties8", 1, 4, 2, 128, 64, 8, 64, 64, 0.0, 0.0, 14)
    rng = np.random.default_rng(14)
    K = rng.standard_normal((1, 2, 64, 128)).astype(np.float16)
    V = rng.standard_normal((1, 2, 64, 128)).astype(np.float16)
    for t in range(64):
        ks = rng.integers(0, 255, size=62)
        V[0, 0, t, 0] = 0.0
        V[0, 0, t, 1] = 255 / 16
        V[0, 0, t, 2:64] = ((ks + 0.5) / 16).astype(np.float16)
    assert np.all(V[0, 0, :, 2:64].astype(np.float64) * 16 % 1 == 0.5)
    cache = tl.make_cache(w, 64)
    cache.append(torch.from_numpy(K).cuda(), torch.from_numpy(V).cuda())
    enc = tl.oracle_encode(w, K[0], V[0])
    tl.sync()
    tl.compare_streams(cache, [(0, 0), (0, 1)], enc, 64)


@pytest.mark.parametrize("bits,Bk,Gv,frac", [(4, 64, 64, 0.0), (3, 128, 32, 0.0), (2, 128, 32, 0.0),
                                             (4, 64, 32, 0.01), (3, 64, 64, 0.01), (2, 64, 64, 0.01)])
def test_low_bit_ties_values_and_keys(bits, Bk, Gv, frac):
    """Exact rounding ties at 2, 3 and 4 bits (Quanto steps 1-2: the codes
    round the quotient (x - z) / s to the nearest integer, ties to even). Every
    value group and every key channel of a full block holds 0 and L/16, so
    s = 1/16 exactly and z = 0, and its other elements are (k + 1/2)/16: each
    quotient is an exact half-integer. With outliers, channel 127 of every
    token carries the vector's largest |x| (the outlier), outside the ties."""
    L = (1 << bits) - 1
    w = W("ties", 1, 4, 2, 128, 2 * Bk + 5, bits, Bk, Gv, frac, 5e5, 15 + bits)
    T = w.T
    rng = np.random.default_rng(100 + bits)
    K = ((rng.integers(0, L, size=(1, 2, T, 128)) + 0.5) / 16).astype(np.float16)
    V = ((rng.integers(0, L, size=(1, 2, T, 128)) + 0.5) / 16).astype(np.float16)
    for blk in range(T // Bk):                      # key channels: 0 and L/16 in every full block
        K[0, :, blk * Bk, :] = 0.0
        K[0, :, blk * Bk + 1, :] = L / 16
    for g in range(128 // Gv):                      # value groups: 0 and L/16 in every token
        V[0, :, :, g * Gv] = 0.0
        V[0, :, :, g * Gv + 1] = L / 16
    if frac > 0:
        K[0, :, :, 127] = 100.0 + np.arange(T)[None, :] / 64
        V[0, :, :, 127] = -100.0
    cache = tl.make_cache(w, (T // Bk + 1) * Bk)
    cache.append(torch.from_numpy(K).cuda(), torch.from_numpy(V).cuda())
    enc = tl.oracle_encode(w, K[0], V[0])
    vmeta = enc["v_meta"].view(np.float16).astype(np.float64)
    kmeta = enc["k_meta"].view(np.float16).astype(np.float64)
    assert np.all(vmeta[..., 0] == 1 / 16) and np.all(vmeta[..., 1] == 0)    # s = 1/16, z = 0: exact ties
    tie_channels = kmeta[..., :127, 0] if frac > 0 else kmeta[..., 0]
    assert np.all(tie_channels == 1 / 16)
    tl.sync()
    tl.compare_streams(cache, [(0, 0), (0, 1)], enc, T)
    q = ki.queries_torch(w, 0, 0, "cuda")
    out = cache.decode(q).cpu().numpy()
    ref = tl.oracle_decode(w, enc, T, tl.q_of_streams(q.cpu().numpy(), w, [(0, 0), (0, 1)]), T - 1)
    tl.check_decode(tl.q_of_streams(out, w, [(0, 0), (0, 1)]), ref, f"ties int{bits}")


def test_capacity_and_noop():
    w = W("cap", 1, 2, 2, 64, 128, 4, 64, 64, 0.0, 0.0, 14)
    cache = tl.make_cache(w, 128)
    K, V = ki.kv_torch(w, 0, 0, 129, "cuda")
    cache.append(K[:, :, :0].contiguous(), V[:, :, :0].contiguous())
    assert cache.T_cur == 0
    cache.append(K[:, :, :128].contiguous(), V[:, :, :128].contiguous())
    assert cache.T_cur == 128
    with pytest.raises(kvq.KvqError) as e:
        cache.append(K[:, :, 128:].contiguous(), V[:, :, 128:].contiguous())
    assert e.value.status == 3 and cache.T_cur == 128


FULL = ["mha7b", "gqa8b", "int3", "int2"]


@pytest.mark.parametrize("name", FULL)
def test_full_size_sampled_streams(name):
    """Full workload on the device (prefill through one append call, then decode);
    the oracle checks three sampled (b, h_kv) streams end to end: the first,
    one from the middle of the batch and heads, and the last."""
    w = ki.WORKLOADS[name]
    T = w.T
    cache = tl.make_cache(w, T + w.key_block)
    K, V = ki.kv_torch(w, 0, 0, T, "cuda")
    cache.append(K, V)
    del K, V
    q = ki.queries_torch(w, 0, 0, "cuda")
    out = cache.decode(q).cpu().numpy()
    streams = [(0, 0), (w.B // 2, w.H_kv // 2 + 1), (w.B - 1, w.H_kv - 1)]
    Kh, Vh = tl.host_streams(w, streams, T)
    enc = tl.oracle_encode(w, Kh, Vh)
    tl.compare_streams(cache, streams, enc, T)
    ref = tl.oracle_decode(w, enc, T, tl.q_of_streams(q.cpu().numpy(), w, streams), T - 1)
    tl.check_decode(tl.q_of_streams(out, w, streams), ref, name)


def test_long_context_sampled_layer():
    """1M-token cache (one of the 32 layers), one sampled stream."""
    w = ki.WORKLOADS["long1m"]
    T = w.T
    layer = 17
    cache = tl.make_cache(w, T + w.key_block)
    t0 = 0
    for chunk in (1 << 18,) * 4:                 # prefill in four appends
        K, V = ki.kv_torch(w, layer, t0, chunk, "cuda")
        cache.append(K, V)
        t0 += chunk
        del K, V
    q = ki.queries_torch(w, layer, 0, "cuda")
    out = cache.decode(q).cpu().numpy()
    streams = [(0, 5)]
    Kh, Vh = tl.host_streams(w, streams, T, layer=layer)
    enc = tl.oracle_encode(w, Kh, Vh)
    tl.compare_streams(cache, streams, enc, T)
    ref = tl.oracle_decode(w, enc, T, tl.q_of_streams(q.cpu().numpy(), w, streams), T - 1)
    tl.check_decode(tl.q_of_streams(out, w, streams), ref, "long1m")

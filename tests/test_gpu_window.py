"""GPU parity of kvq_append_window (sliding-window key statistics, page
mlqm.cn/news/1064729 §3.2) against the oracle's window encoding.

Codes, metadata, tails and outlier lists must match bit for bit; decode
(the unchanged kvq_decode_attn) must be within the decode tolerance of the
oracle's float64 attention on its own window encoding. A window of one key
block must reproduce kvq_append's cache exactly.
"""
import numpy as np
import pytest
import torch

import bit_quantized_kv_append_gb300 as kvq
from bit_quantized_kv_append_gb300 import build as kbuild
import kvq_inputs as ki
import kvq_testlib as tl
from oracle import oracle_cpp as oc

pytestmark = pytest.mark.gpu
W = ki.Workload

CASES = {
    # name: (workload, window, append pieces)
    "int4_outliers_w1024": (W("w4", 2, 8, 2, 128, 1500, 4, 64, 64, 0.01, 5e5, 71), 1024, [700, 1, 63, 600, 136]),
    "int3_bk128_w512": (W("w3", 1, 8, 2, 128, 1100, 3, 128, 32, 0.01, 5e5, 72), 512, [1100]),
    "int2_w256_no_outliers": (W("w2", 2, 4, 4, 128, 900, 2, 64, 32, 0.0, 1e4, 73), 256, [100, 300, 1, 1, 498]),
    "d64_int4_w192": (W("w64", 2, 4, 2, 64, 700, 4, 64, 32, 0.04, 1e4, 74), 192, [333, 367]),
    "int8_w256": (W("w8", 1, 4, 2, 128, 600, 8, 64, 64, 0.01, 5e5, 75), 256, [600]),
}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available(), "the gpu tests need a CUDA device"
    kbuild.build()
    kvq.lib()


def _drifting(w, T):
    K, V = ki.kv_torch(w, 0, 0, T, "cuda")
    # a channel whose range drifts over time, so window and block statistics differ
    K[:, :, :, 9] += torch.linspace(0, 30, T, device="cuda", dtype=torch.float32).half()
    return K.contiguous(), V


@pytest.mark.parametrize("name", list(CASES))
def test_window_append_parity(name):
    w, window, pieces = CASES[name]
    T = w.T
    cache = tl.make_cache(w, (T // w.key_block + 1) * w.key_block)
    K, V = _drifting(w, T)
    t = 0
    for n in pieces:
        cache.append_window(K[:, :, t:t + n].contiguous(), V[:, :, t:t + n].contiguous(), window)
        t += n
    assert t == T and cache.T_cur == T
    streams = [(b, h) for b in range(w.B) for h in range(w.H_kv)]
    Kh = K.cpu().numpy().reshape(-1, T, w.D)
    Vh = V.cpu().numpy().reshape(-1, T, w.D)
    enc = oc.encode(Kh, Vh, w.bits, w.key_block, w.value_group, tl.n_out_of(w), window=window)
    plain = tl.oracle_encode(w, Kh, Vh)
    if T // w.key_block * w.key_block > window:
        assert not np.array_equal(enc["k_meta"], plain["k_meta"])       # the window changes the statistics
    tl.sync()
    tl.compare_streams(cache, streams, enc, T)
    q = ki.queries_torch(w, 0, 0, "cuda")
    out = cache.decode(q).cpu().numpy()
    ref = tl.oracle_decode(w, enc, T, tl.q_of_streams(q.cpu().numpy(), w, streams), T - 1)
    tl.check_decode(tl.q_of_streams(out, w, streams), ref, name)


def test_window_token_by_token_across_block_edges():
    w = W("wtok", 1, 4, 2, 128, 200, 4, 64, 64, 0.01, 5e5, 76)
    T, window = w.T, 128
    cache = tl.make_cache(w, 256)
    K, V = _drifting(w, T)
    for t in range(T):
        cache.append_window(K[:, :, t:t + 1].contiguous(), V[:, :, t:t + 1].contiguous(), window)
    Kh = K.cpu().numpy().reshape(-1, T, w.D)
    Vh = V.cpu().numpy().reshape(-1, T, w.D)
    enc = oc.encode(Kh, Vh, w.bits, w.key_block, w.value_group, tl.n_out_of(w), window=window)
    tl.sync()
    tl.compare_streams(cache, [(0, 0), (0, 1)], enc, T)


def test_window_of_one_block_equals_append():
    w = W("wone", 2, 8, 2, 128, 777, 3, 64, 32, 0.01, 5e5, 77)
    T = w.T
    a = tl.make_cache(w, 832)
    b = tl.make_cache(w, 832)
    K, V = ki.kv_torch(w, 0, 0, T, "cuda")
    tl.append_pieces(a, K, V, [100, 300, 1, 376])
    t = 0
    for n in [100, 300, 1, 376]:
        b.append_window(K[:, :, t:t + n].contiguous(), V[:, :, t:t + n].contiguous(), w.key_block)
        t += n
    tl.sync()
    va, vb = a.views(), b.views()
    nb = T // w.key_block
    for name in va:
        x, y = va[name].cpu().numpy(), vb[name].cpu().numpy()
        if name in ("k_codes", "k_outl"):
            x, y = x[:, :, : nb * w.key_block], y[:, :, : nb * w.key_block]
        elif name == "k_meta":
            x, y = x[:, :, :nb], y[:, :, :nb]
        elif name == "k_tail":
            x, y = x[:, :, : T - nb * w.key_block], y[:, :, : T - nb * w.key_block]
        else:
            x, y = x[:, :, :T], y[:, :, :T]
        assert np.array_equal(x.view(np.uint8), y.view(np.uint8)), name


def test_window_argument_checks():
    w = W("wchk", 1, 2, 2, 128, 128, 4, 64, 64, 0.0, 0.0, 78)
    cache = tl.make_cache(w, 128)
    K, V = ki.kv_torch(w, 0, 0, 64, "cuda")
    for bad in (0, 32, 96):                       # not a positive multiple of the key block
        with pytest.raises(kvq.KvqError) as e:
            cache.append_window(K, V, bad)
        assert e.value.status == 2
    assert cache.T_cur == 0

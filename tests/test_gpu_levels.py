"""GPU parity of the non-uniform codes (kvq_append_levels,
kvq_decode_attn_levels) against the oracle with the same level table.

The table is fitted by the oracle's k-means on calibration values of another
layer (an input of both sides). Codes, ranges, zeros and outlier lists must
match the oracle's encoding bit for bit, and decode attention must be within
the decode tolerance of the oracle's float64 attention on its own decoding.
"""
import math

import numpy as np
import pytest
import torch

import bit_quantized_kv_append_gb300 as kvq
from bit_quantized_kv_append_gb300 import build as kbuild
from oracle import oracle_cpp as oc
import kvq_inputs as ki
import kvq_testlib as tl

pytestmark = pytest.mark.gpu

W = ki.Workload
CASES = {
    # name: (workload, T, append pieces)
    "gqa_int4_outliers_rope": (W("lv4", 2, 8, 2, 128, 256, 4, 64, 64, 0.01, 5e5, 51), 256, [128, 128]),
    "d64_int3_bk128_two_outliers": (W("lv3", 1, 4, 2, 64, 256, 3, 128, 32, 0.04, 1e4, 52), 256, [256]),
    "mha_int8_norope": (W("lv8", 1, 2, 2, 128, 128, 8, 64, 64, 0.0, 0.0, 53), 128, [64, 64]),
    "g8_int2_gv128": (W("lv2", 1, 16, 2, 128, 192, 2, 64, 128, 0.01, 5e5, 54), 192, [192]),
    # head_dim 128 runs on the tensor-core kernel (level lookups), head_dim 64 on the CUDA-core one
    "int4_bk128_mha_tc": (W("lv4b", 2, 4, 4, 128, 1024, 4, 128, 64, 0.0, 1e4, 56), 1024, [512, 512]),
    "int4_g8_gv32_long_tc": (W("lv4g", 2, 16, 2, 128, 4096, 4, 64, 32, 0.01, 5e5, 57), 4096, [4096]),
    # ragged appends ending in an unfinished key block (its keys stay fp16 in K_TAIL)
    "int4_ragged_tc": (W("lv4r", 2, 8, 2, 128, 777, 4, 64, 64, 0.01, 5e5, 58), 777, [100, 1, 63, 300, 313]),
    "int3_d64_ragged": (W("lv3r", 1, 4, 2, 64, 300, 3, 128, 32, 0.04, 1e4, 59), 300, [37, 91, 1, 171]),
    "int8_ragged_norope": (W("lv8r", 1, 2, 2, 128, 200, 8, 64, 64, 0.01, 0.0, 60), 200, [65, 70, 65]),
    "int2_g8_ragged": (W("lv2r", 1, 16, 2, 128, 250, 2, 64, 128, 0.01, 5e5, 61), 250, [1, 1, 1, 63, 184]),
    # 3-bit codes at head_dim 128 (128- and 64-token key blocks)
    "int3_bk128_gqa_tc": (W("lv3t", 2, 8, 2, 128, 700, 3, 128, 32, 0.01, 5e5, 65), 700, [300, 1, 399]),
    "int3_bk64_mha_tc": (W("lv3s", 1, 4, 4, 128, 333, 3, 64, 64, 0.01, 1e4, 66), 333, [200, 133]),
}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available(), "the gpu tests need a CUDA device"
    kbuild.build()
    kvq.lib()


def _levels(w):
    # calibration: normalized values of another layer's groups, fitted by the oracle
    Kc, Vc = ki.streams_np(w, [(0, 0)], 256, layer=7)
    x = np.concatenate([Kc.reshape(-1, w.value_group), Vc.reshape(-1, w.value_group)]).astype(np.float64)
    span = x.max(axis=1, keepdims=True) - x.min(axis=1, keepdims=True)
    u = (x - x.min(axis=1, keepdims=True)) / np.where(span > 0, span, 1.0)
    return oc.fit_levels(u.ravel(), w.bits, 60)


@pytest.mark.parametrize("precise", [False, True], ids=["default", "precise"])
@pytest.mark.parametrize("name", list(CASES))
def test_levels_parity(name, precise):
    """precise: KVQ_FLAG_PRECISE_SCORES, which keeps head_dim-128 level tables
    on the fp32 CUDA-core kernel (the default runs them on the tensor-core
    kernel)."""
    w, T, pieces = CASES[name]
    lv = _levels(w)
    T_max = (T // w.key_block + 1) * w.key_block
    cache = kvq.QuantizedKVCache(w.B, w.H_kv, w.D, T_max, w.bits, w.key_block, w.value_group,
                                 w.outlier_frac, H_q=w.H_q, rope_theta=w.rope_theta, device="cuda",
                                 precise=precise)
    K, V = ki.kv_torch(w, 0, 0, T, "cuda")
    t = 0
    for n in pieces:
        cache.append_levels(K[:, :, t:t + n].contiguous(), V[:, :, t:t + n].contiguous(), lv)
        t += n
    assert cache.T_cur == T
    streams = [(b, h) for b in range(w.B) for h in range(w.H_kv)]
    Kh, Vh = tl.host_streams(w, streams, T)
    enc = oc.encode(Kh, Vh, w.bits, w.key_block, w.value_group, tl.n_out_of(w), levels=lv)
    tl.sync()
    tl.compare_streams(cache, streams, enc, T)
    Kd, Vd = oc.dequant(enc, T, w.D, w.bits, w.key_block, w.value_group, tl.n_out_of(w), levels=lv)
    q = ki.queries_torch(w, 0, 0, "cuda")
    qs = tl.q_of_streams(q.cpu().numpy(), w, streams)
    for q_pos in (T - 1, T // 3):
        out = cache.decode_levels(q, lv, q_pos=q_pos).cpu().numpy()
        ref = oc.attention(Kd, Vd, qs, q_pos, w.rope_theta, 1.0 / math.sqrt(w.D))
        tl.check_decode(tl.q_of_streams(out, w, streams), ref, f"{name} q_pos={q_pos}")


def test_levels_token_by_token_serving():
    """The serving loop on a level-table cache: a prefill, then one token
    appended and attended per step across key-block edges (tensor-core kernel
    for these 4-bit codes; kvq_decode_step_levels on odd positions, the two
    calls on even ones), against the oracle's encoding of the same prefix."""
    w = W("lvtok", 1, 8, 2, 128, 200, 4, 64, 64, 0.01, 5e5, 62)
    lv = _levels(w)
    T0, T = 120, 200
    cache = tl.make_cache(w, 256)
    K, V = ki.kv_torch(w, 0, 0, T, "cuda")
    cache.append_levels(K[:, :, :T0].contiguous(), V[:, :, :T0].contiguous(), lv)
    streams = [(0, h) for h in range(w.H_kv)]
    Kh, Vh = tl.host_streams(w, streams, T)
    q = ki.queries_torch(w, 0, 0, "cuda")
    qs = tl.q_of_streams(q.cpu().numpy(), w, streams)
    for t in range(T0, T):
        k1, v1 = K[:, :, t:t + 1].contiguous(), V[:, :, t:t + 1].contiguous()
        if t % 2:                                        # the fused step on odd positions
            out = cache.decode_step_levels(k1, v1, q, lv)
        else:
            cache.append_levels(k1, v1, lv)
            out = cache.decode_levels(q, lv)
        if t in (T0, 127, 128, 150, T - 1):
            n = t + 1
            out = out.cpu().numpy()
            enc = oc.encode(Kh[:, :n], Vh[:, :n], w.bits, w.key_block, w.value_group, tl.n_out_of(w), levels=lv)
            Kd, Vd = oc.dequant(enc, n, w.D, w.bits, w.key_block, w.value_group, tl.n_out_of(w), levels=lv)
            ref = oc.attention(Kd, Vd, qs, n - 1, w.rope_theta, 1.0 / math.sqrt(w.D))
            tl.check_decode(tl.q_of_streams(out, w, streams), ref, f"tokens={n}")
    tl.sync()
    enc = oc.encode(Kh, Vh, w.bits, w.key_block, w.value_group, tl.n_out_of(w), levels=lv)
    tl.compare_streams(cache, streams, enc, T)


def test_decode_step_levels_matches_the_two_calls():
    """kvq_decode_step_levels is bit-identical to kvq_append_levels (one token)
    followed by kvq_decode_attn_levels, on both level kernels."""
    for w in (W("lvs4", 2, 8, 2, 128, 130, 4, 64, 64, 0.01, 5e5, 63),     # tensor-core kernel
              W("lvs3", 1, 4, 2, 64, 130, 3, 64, 32, 0.04, 1e4, 64)):     # CUDA-core kernel
        lv = _levels(w)
        a, b = tl.make_cache(w, 192), tl.make_cache(w, 192)
        K, V = ki.kv_torch(w, 0, 0, w.T + 3, "cuda")
        for c in (a, b):
            c.append_levels(K[:, :, :w.T].contiguous(), V[:, :, :w.T].contiguous(), lv)
        q = ki.queries_torch(w, 0, 0, "cuda")
        for t in range(w.T, w.T + 3):
            k1, v1 = K[:, :, t:t + 1].contiguous(), V[:, :, t:t + 1].contiguous()
            x = a.decode_step_levels(k1, v1, q, lv).clone()
            b.append_levels(k1, v1, lv)
            y = b.decode_levels(q, lv).clone()
            assert torch.equal(x, y), t
        tl.sync()
        T, Bk = a.T_cur, w.key_block
        nb = T // Bk
        va, vb = a.views(), b.views()
        for name in va:                                  # the rows written so far
            x, y = va[name].cpu().numpy(), vb[name].cpu().numpy()
            if name in ("k_codes", "k_outl"):
                x, y = x[:, :, : nb * Bk], y[:, :, : nb * Bk]
            elif name == "k_meta":
                x, y = x[:, :, :nb], y[:, :, :nb]
            elif name == "k_tail":
                x, y = x[:, :, : T - nb * Bk], y[:, :, : T - nb * Bk]
            else:
                x, y = x[:, :, :T], y[:, :, :T]
            assert np.array_equal(x.view(np.uint8), y.view(np.uint8)), name


def test_levels_exact_midpoints():
    """Quotients exactly on the midpoints (ties go to the lower level): a
    table whose levels and midpoints are fp16 values, every value group and
    key channel holding 0 and 1 (so z = 0, r = 1 and u = x), and elements
    planted on every midpoint and next to them; codes bit-exact against the
    oracle."""
    w = W("lvmid", 1, 4, 2, 128, 192, 4, 64, 64, 0.0, 1e4, 67)
    lv = np.array([k / 16 for k in range(15)] + [1.0], dtype=np.float32)
    mids = (lv[:-1].astype(np.float64) + lv[1:]) / 2
    pts = [0.0, 1.0]
    for m in mids:
        h = np.float16(m)
        assert float(h) == m                                   # the midpoints are fp16 values
        pts += [m, float(np.nextafter(h, np.float16(0))), float(np.nextafter(h, np.float16(1)))]
    grid = np.array(pts, dtype=np.float16)
    t = np.arange(w.T)[:, None]
    c = np.arange(w.D)[None, :]
    base = grid[(t + 3 * c) % len(grid)]                        # [T, D]: each token and channel meets 0 and 1
    base[:, 0], base[:, 1] = 0.0, 1.0                           # every value group holds 0 and 1
    base[0::64, :], base[1::64, :] = 0.0, 1.0                   # every key channel of a block holds 0 and 1
    Kh = np.broadcast_to(base, (w.B * w.H_kv, w.T, w.D)).copy()
    Vh = Kh[:, ::-1].copy()
    cache = tl.make_cache(w, 256)
    K = torch.from_numpy(Kh.reshape(w.B, w.H_kv, w.T, w.D)).cuda()
    V = torch.from_numpy(Vh.reshape(w.B, w.H_kv, w.T, w.D)).cuda()
    cache.append_levels(K[:, :, :100].contiguous(), V[:, :, :100].contiguous(), lv)
    cache.append_levels(K[:, :, 100:].contiguous(), V[:, :, 100:].contiguous(), lv)
    streams = [(0, h) for h in range(w.H_kv)]
    enc = oc.encode(Kh, Vh, w.bits, w.key_block, w.value_group, 0, levels=lv)
    tl.sync()
    tl.compare_streams(cache, streams, enc, w.T)

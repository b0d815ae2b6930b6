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
    # name: (workload, T, append pieces (whole key blocks))
    "gqa_int4_outliers_rope": (W("lv4", 2, 8, 2, 128, 256, 4, 64, 64, 0.01, 5e5, 51), 256, [128, 128]),
    "d64_int3_bk128_two_outliers": (W("lv3", 1, 4, 2, 64, 256, 3, 128, 32, 0.04, 1e4, 52), 256, [256]),
    "mha_int8_norope": (W("lv8", 1, 2, 2, 128, 128, 8, 64, 64, 0.0, 0.0, 53), 128, [64, 64]),
    "g8_int2_gv128": (W("lv2", 1, 16, 2, 128, 192, 2, 64, 128, 0.01, 5e5, 54), 192, [192]),
    # 4-bit codes at head_dim 128 run on the tensor-core kernel (level lookups)
    "int4_bk128_mha_tc": (W("lv4b", 2, 4, 4, 128, 1024, 4, 128, 64, 0.0, 1e4, 56), 1024, [512, 512]),
    "int4_g8_gv32_long_tc": (W("lv4g", 2, 16, 2, 128, 4096, 4, 64, 32, 0.01, 5e5, 57), 4096, [4096]),
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
    """precise: KVQ_FLAG_PRECISE_SCORES, which keeps 4-bit head_dim-128 level
    tables on the fp32 CUDA-core kernel (the default runs them on the
    tensor-core kernel)."""
    w, T, pieces = CASES[name]
    lv = _levels(w)
    cache = kvq.QuantizedKVCache(w.B, w.H_kv, w.D, T + w.key_block, w.bits, w.key_block, w.value_group,
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


def test_levels_reject_partial_blocks():
    w = W("lvp", 1, 2, 2, 128, 64, 4, 64, 64, 0.0, 0.0, 55)
    cache = tl.make_cache(w, 128)
    K, V = ki.kv_torch(w, 0, 0, 32, "cuda")
    with pytest.raises(kvq.KvqError) as e:
        cache.append_levels(K, V, np.linspace(0, 1, 16, dtype=np.float32))
    assert e.value.status == 2 and cache.T_cur == 0

"""GPU parity of kvq_decode_step, the fused decode step (append one token per
sequence, then attend its query over every cached token, in one call).

Per step: the cache it leaves matches the oracle's encoding bit for bit, the
output is within the decode tolerance of the oracle's float64 attention, and
both equal, bit for bit, kvq_append followed by kvq_decode_attn on a second
cache. The steps cross key-block edges, so a step that completes a block
(quantizing it) is covered, as is a step into an empty cache.
"""
import numpy as np
import pytest
import torch

import bit_quantized_kv_append_gb300 as kvq
from bit_quantized_kv_append_gb300 import build as kbuild
import kvq_inputs as ki
import kvq_testlib as tl

pytestmark = pytest.mark.gpu

W = ki.Workload
CASES = {
    # name: (workload, tokens appended before the first step, steps)
    "mha_rope_block_edge": (W("mha", 2, 4, 4, 128, 130, 4, 64, 64, 0.0, 1e4, 21), 126, 4),
    "gqa_outliers": (W("gqa", 2, 8, 2, 128, 195, 4, 64, 64, 0.01, 5e5, 22), 190, 5),
    "int3_bk128_gv32": (W("int3", 1, 8, 2, 128, 130, 3, 128, 32, 0.01, 5e5, 23), 125, 5),
    "d64_int2_two_outliers": (W("d64", 2, 4, 2, 64, 66, 2, 64, 32, 0.04, 1e4, 24), 62, 4),
    "from_empty": (W("one", 1, 2, 2, 128, 3, 4, 64, 64, 0.0, 1e4, 25), 0, 3),
}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available(), "the gpu tests need a CUDA device"
    kbuild.build()
    kvq.lib()


@pytest.mark.parametrize("name", list(CASES))
def test_decode_step_parity(name):
    w, T0, steps = CASES[name]
    T_end = T0 + steps
    T_max = (T_end // w.key_block + 1) * w.key_block
    fused, split = tl.make_cache(w, T_max), tl.make_cache(w, T_max)
    for c in (fused, split):                 # so that bytes no call writes compare equal too
        for buf in c.buffers.values():
            buf.zero_()
    K, V = ki.kv_torch(w, 0, 0, T_end, "cuda")
    if T0:
        for c in (fused, split):
            c.append(K[:, :, :T0].contiguous(), V[:, :, :T0].contiguous())
    streams = [(b, h) for b in range(w.B) for h in range(w.H_kv)]
    Kh, Vh = tl.host_streams(w, streams, T_end)
    for s in range(steps):
        t = T0 + s
        k1, v1 = K[:, :, t:t + 1].contiguous(), V[:, :, t:t + 1].contiguous()
        q = ki.queries_torch(w, 0, s, "cuda")
        out = fused.decode_step(k1, v1, q)
        assert fused.T_cur == t + 1
        split.append(k1, v1)
        out_split = split.decode(q, q_pos=t)
        tl.sync()
        assert torch.equal(out.view(torch.int16), out_split.view(torch.int16)), f"step {s}: fused != split"
        enc = tl.oracle_encode(w, np.ascontiguousarray(Kh[:, :t + 1]), np.ascontiguousarray(Vh[:, :t + 1]))
        tl.compare_streams(fused, streams, enc, t + 1)
        ref = tl.oracle_decode(w, enc, t + 1, tl.q_of_streams(q.cpu().numpy(), w, streams), t)
        tl.check_decode(tl.q_of_streams(out.cpu().numpy(), w, streams), ref, f"{name} step {s}")
    for key in fused.buffers:
        assert torch.equal(fused.buffers[key], split.buffers[key]), key


def test_decode_step_capacity_leaves_cache():
    w = W("cap", 1, 2, 2, 128, 64, 4, 64, 64, 0.0, 1e4, 26)
    cache = tl.make_cache(w, 64)
    K, V = ki.kv_torch(w, 0, 0, 65, "cuda")
    cache.append(K[:, :, :64].contiguous(), V[:, :, :64].contiguous())
    before = {k: v.clone() for k, v in cache.buffers.items()}
    with pytest.raises(kvq.KvqError) as e:
        cache.decode_step(K[:, :, 64:65].contiguous(), V[:, :, 64:65].contiguous(), ki.queries_torch(w, 0, 0, "cuda"))
    assert e.value.status == 3 and cache.T_cur == 64
    for k, v in cache.buffers.items():       # raw bytes: stale tail rows may hold NaN patterns
        assert torch.equal(v, before[k]), k

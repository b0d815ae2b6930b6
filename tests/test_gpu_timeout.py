"""The bounded waits of the decode kernel report an expiry on the host
(kvq_decode_attn_diag; no fault, no endless wait).

With every ring stage armed for 16 bytes more than its copies deliver, no
stage completes, so every wait runs out (after one second of the GPU's
global timer). The
kernel must then set KVQ_STATUS_TIMEOUT in the workspace's status word, write
NaN partials and return; afterwards the context, the cache and a normal decode
call must be intact. A diag call without padding must match kvq_decode_attn
bit for bit and leave the word clear.
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


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available(), "the gpu tests need a CUDA device"
    kbuild.build()
    kvq.lib()


@pytest.mark.parametrize("w", [W("to4", 2, 8, 2, 128, 700, 4, 64, 64, 0.01, 5e5, 81),
                               W("to3", 1, 8, 8, 128, 600, 3, 128, 32, 0.0, 1e4, 82)], ids=["int4", "int3_bk128"])
def test_expired_waits_are_reported_and_the_context_stays_usable(w):
    T = w.T
    cache = tl.make_cache(w, (T // w.key_block + 1) * w.key_block)
    K, V = ki.kv_torch(w, 0, 0, T, "cuda")
    cache.append(K, V)
    q = ki.queries_torch(w, 0, 0, "cuda")
    want = cache.decode(q).clone()
    assert cache.status() == 0
    # compared as bytes: unused rows (the tail past T mod Bk) hold whatever the allocation held
    before = {k: v.clone().view(torch.uint8) for k, v in cache.views().items()}

    # no padding: the diagnostic call is the ordinary one
    same = torch.empty_like(q)
    kvq.decode_attn_diag(cache.cfg, cache.ref(), q, cache.H_q, T - 1, cache.rope, 1.0 / np.sqrt(w.D), same,
                         cache.workspace, 0)
    assert torch.equal(same, want) and cache.status() == 0

    # over-armed barriers: every wait expires
    bad = torch.zeros_like(q)
    kvq.decode_attn_diag(cache.cfg, cache.ref(), q, cache.H_q, T - 1, cache.rope, 1.0 / np.sqrt(w.D), bad,
                         cache.workspace, 16)
    torch.cuda.synchronize()
    assert cache.status() & kvq.kvq.STATUS_TIMEOUT
    assert torch.isnan(bad.float()).any()                         # the outputs of the expired splits

    # the cache is untouched and the context still computes correct results
    for k, v in cache.views().items():
        assert torch.equal(v.view(torch.uint8), before[k]), k
    cache.clear_status()
    again = cache.decode(q)
    torch.cuda.synchronize()
    assert cache.status() == 0 and not torch.isnan(again.float()).any()
    assert torch.equal(again, want)

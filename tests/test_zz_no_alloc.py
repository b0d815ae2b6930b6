"""kvq_decode_attn_noalloc against kvq_decode_attn.

The allocation-free entry point serves callers that cannot hand the library a
device workspace, for instance a serving engine that reserves all device
memory at start-up and forbids later cudaMalloc calls on the decode path, or
a plain-C host that owns no device allocator. It keeps its split partials in
the library's fixed 8 MiB device array instead. Its results must match the
workspace entry point within the decode tolerance of the parity tests, on two
calls in a row (the array is reused and keeps the previous call's contents).

This file is named to be collected last, so a run that stops at the first
failure has already run every other test.
"""
import ctypes
import math

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
    "gqa_outliers_rope": W("na_gqa", 2, 8, 2, 128, 777, 4, 64, 64, 0.01, 5e5, 31),
    "int3_bk128": W("na_int3", 1, 8, 2, 128, 700, 3, 128, 32, 0.01, 5e5, 32),
    "d64_mha": W("na_d64", 2, 4, 4, 64, 300, 3, 64, 32, 0.0, 1e4, 33),
    "wide_batch": W("na_wide", 8, 32, 32, 128, 2000, 4, 64, 64, 0.0, 1e4, 34),
    # 8 MiB holds only 7 splits of B * H_q * (D + 2) floats here, against 65
    # key blocks per stream: the allocation-free call runs with fewer splits
    # than the workspace call chooses, so the split limit itself is exercised
    "split_limit_binds": W("na_cap", 32, 64, 8, 128, 4096 + 37, 4, 64, 64, 0.01, 5e5, 35),
}
SCRATCH_BYTES = 8 << 20


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available(), "the gpu tests need a CUDA device"
    kbuild.build()
    kvq.lib()


@pytest.mark.parametrize("name", list(CASES))
def test_noalloc_matches_workspace_entry(name):
    w = CASES[name]
    T = w.T
    if name == "split_limit_binds":
        fit = SCRATCH_BYTES // (w.B * w.H_q * (w.D + 2) * 4)
        assert fit < (T + w.key_block - 1) // w.key_block // 8
    cache = tl.make_cache(w, (T // w.key_block + 1) * w.key_block)
    K, V = ki.kv_torch(w, 0, 0, T, "cuda")
    cache.append(K, V)
    scale = 1.0 / math.sqrt(w.D)
    for step in (0, 1):                          # two calls in a row share the array
        q = ki.queries_torch(w, 0, step, "cuda")
        want = cache.decode(q, q_pos=T - 1, sm_scale=scale)
        got = torch.full_like(q, float("nan"))
        kvq.decode_attn_noalloc(cache.cfg, cache.ref(), q, cache.H_q, T - 1, cache.rope, scale, got)
        torch.cuda.synchronize()
        tl.check_decode(got.cpu().numpy(), want.double().cpu().numpy(), f"{name} call {step}")


def test_noalloc_rejects_shapes_beyond_its_array():
    # one split of B * H_q * (D + 2) floats would not fit in 8 MiB: refused
    # before anything touches the device (the pointers are never used)
    cfg = kvq.make_config(128, 128, 128, 64, 4, 64, 64, 0.0)
    r = kvq.CacheRef()
    for i, n in enumerate(kvq.BUFFERS):
        setattr(r, n, 0x10000 * (i + 1))
    r.T_cur = 10
    p = ctypes.c_void_p(0x10000)
    rc = kvq.lib().kvq_decode_attn_noalloc(ctypes.byref(cfg), ctypes.byref(r), p, 128, 9, None, 0.1, p, None)
    assert rc == 4

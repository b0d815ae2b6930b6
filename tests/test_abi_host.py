"""Host-side checks of the C ABI (no GPU): the library loads, exports every
entry point the header declares, sizes its buffers as documented, and rejects
bad arguments with the documented status before launching anything."""
import ctypes
import os
import re

import pytest

import bit_quantized_kv_append_gb300 as kvq
from bit_quantized_kv_append_gb300 import build as kbuild
import kvq_inputs as ki

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "kvq.h")
GOLDEN = os.path.join(ROOT, "tests", "golden")


@pytest.fixture(scope="module")
def lib():
    kbuild.build()
    return kvq.lib()


CITATION = re.compile(r"page|KVQuant|Quanto|mlqm\.cn|horizon\.auto|no passage|no counterpart")


def test_exports_every_declared_symbol(lib):
    text = open(HEADER).read()
    names = re.findall(r"KVQ_API\s+[\w\s\*]+?\b(kvq_\w+)\s*\(", text)
    assert sorted(names) == sorted(kvq.EXPORTS)
    for n in names:
        assert hasattr(lib, n), n
    assert lib.kvq_version().decode().startswith("kvq ")
    # every declaration's own comment block names the passage it implements
    # (or says that it has none)
    for m in re.finditer(r"/\*((?:(?!\*/).)*)\*/\s*KVQ_API\s+[\w\s\*]+?\b(kvq_\w+)\s*\(", text, re.S):
        assert CITATION.search(m.group(1)), f"{m.group(2)}: its comment cites no passage"
    cited = [m.group(2) for m in re.finditer(r"/\*((?:(?!\*/).)*)\*/\s*KVQ_API\s+[\w\s\*]+?\b(kvq_\w+)\s*\(",
                                             text, re.S)]
    assert sorted(cited) == sorted(names)


def test_status_strings(lib):
    for code, name in kvq.kvq.STATUS.items():
        assert lib.kvq_status_string(code).decode().startswith(name)


def _golden(name):
    vals = {}
    for line in open(os.path.join(GOLDEN, name)):
        if line.strip() and not line.startswith("#"):
            k, v = (p.strip() for p in line.split("="))
            vals[k] = int(v)
    return vals


def test_fp16_equivalent_size_matches_page_example(lib):
    g = _golden("kv_memory_example.txt")
    # one layer: H_kv * D = hidden (32 heads x 128)
    lay = kvq.layout(kvq.make_config(g["batch"], 32, 128, g["seq"]), 32)
    total = g["layers"] * lay.fp16_equiv_bytes
    assert total == g["total_bytes"]
    assert abs(total / 2 ** 30 - g["approx_gb"]) < 0.01


@pytest.mark.parametrize("name", list(ki.WORKLOADS))
def test_layout_sizes(lib, name):
    w = ki.WORKLOADS[name]
    T_max = w.T + w.key_block
    cfg = kvq.make_config(w.B, w.H_kv, w.D, T_max, w.bits, w.key_block, w.value_group, w.outlier_frac)
    lay = kvq.layout(cfg, w.H_q)
    n_out = 0 if w.outlier_frac == 0 else max(1, int(w.outlier_frac * w.D))
    S = w.B * w.H_kv
    cb = w.D * w.bits // 8
    assert lay.n_out == n_out and lay.code_row_bytes == cb
    want = [T_max * cb, T_max // w.key_block * w.D * 4, w.key_block * w.D * 2, T_max * n_out * 4,
            T_max * cb, T_max * (w.D // w.value_group) * 4, T_max * n_out * 4]
    assert list(lay.stream_bytes) == want
    assert list(lay.bytes) == [x * S for x in want]
    assert lay.cache_bytes == sum(lay.bytes)
    assert lay.fp16_equiv_bytes == 2 * S * T_max * w.D * 2
    for b in lay.stream_bytes:
        assert b % 16 == 0          # every stream starts 16-byte aligned
    # packed INT4 + metadata is ~30% of fp16; INT2 well under 25%; INT8 ~55%
    ratio = lay.cache_bytes / lay.fp16_equiv_bytes
    if w.T >= 32768:                 # the fp16 tail is a fixed cost on tiny caches
        assert ratio < {8: 0.56, 4: 0.32, 3: 0.27, 2: 0.21}[w.bits]


def _cfg(**kw):
    base = dict(B=2, H_kv=2, D=128, T_max=256, bits=4, key_block=64, value_group=64, outlier_frac=0.01)
    base.update(kw)
    return kvq.make_config(**base)


@pytest.mark.parametrize("kw", [dict(bits=1), dict(bits=5), dict(D=96), dict(key_block=32),
                                dict(value_group=48), dict(T_max=100), dict(T_max=0), dict(B=0),
                                dict(outlier_frac=0.2), dict(outlier_frac=-0.1), dict(B=70000),
                                dict(T_max=1 << 24)])
def test_layout_rejects_unsupported(lib, kw):
    out = kvq.Layout()
    assert lib.kvq_layout(ctypes.byref(_cfg(**kw)), 2, ctypes.byref(out)) == 2


def test_layout_rejects_bad_hq_and_null(lib):
    out = kvq.Layout()
    assert lib.kvq_layout(ctypes.byref(_cfg()), 3, ctypes.byref(out)) == 2
    assert lib.kvq_layout(None, 2, ctypes.byref(out)) == 1
    assert lib.kvq_layout(ctypes.byref(_cfg()), 2, None) == 1


FAKE = 0x10000  # never dereferenced: every call below must fail its host checks


def _fake_cache(T_cur, n_out=1):
    r = kvq.CacheRef()
    for i, n in enumerate(kvq.BUFFERS):
        setattr(r, n, FAKE * (i + 1) if (n_out or "outl" not in n) else None)
    r.T_cur = T_cur
    return r


def test_append_host_errors(lib):
    cfg = _cfg()
    r = _fake_cache(200)
    p = ctypes.c_void_p(FAKE)
    assert lib.kvq_append(ctypes.byref(cfg), ctypes.byref(r), p, p, 57, None) == 3   # capacity
    assert r.T_cur == 200
    assert lib.kvq_append(ctypes.byref(cfg), ctypes.byref(r), p, p, -1, None) == 1
    assert lib.kvq_append(ctypes.byref(cfg), None, p, p, 1, None) == 1
    assert lib.kvq_append(ctypes.byref(cfg), ctypes.byref(r), None, p, 1, None) == 1
    assert lib.kvq_append(ctypes.byref(cfg), ctypes.byref(r), ctypes.c_void_p(FAKE + 8), p, 1, None) == 1
    assert lib.kvq_append(ctypes.byref(cfg), ctypes.byref(r), p, p, 0, None) == 0      # no-op
    bad = _fake_cache(200)
    bad.k_meta = FAKE + 4                                                               # misaligned
    assert lib.kvq_append(ctypes.byref(cfg), ctypes.byref(bad), p, p, 1, None) == 1
    no_outl = _fake_cache(0, n_out=0)
    assert lib.kvq_append(ctypes.byref(cfg), ctypes.byref(no_outl), p, p, 1, None) == 1  # n_out=1 needs them
    assert lib.kvq_append(ctypes.byref(_cfg(bits=7)), ctypes.byref(r), p, p, 1, None) == 2
    over = _fake_cache(300)
    assert lib.kvq_append(ctypes.byref(cfg), ctypes.byref(over), p, p, 1, None) == 1   # T_cur > T_max


def test_decode_host_errors(lib):
    cfg = _cfg()
    lay = kvq.layout(cfg, 8)
    r = _fake_cache(100)
    p = ctypes.c_void_p(FAKE)
    ws = lay.workspace_bytes

    def call(cache=r, q=p, H_q=8, q_pos=99, rope=None, scale=0.1, out=p, w=p, wsb=ws, c=cfg):
        return lib.kvq_decode_attn(ctypes.byref(c), None if cache is None else ctypes.byref(cache), q, H_q,
                                   q_pos, rope, scale, out, w, wsb, None)

    assert call(wsb=ws - 1) == 4
    assert call(H_q=6) == 2                      # G = 3
    assert call(H_q=3) == 2                      # not a multiple of H_kv
    assert call(H_q=64) == 2                     # G = 32
    assert call(q_pos=-1) == 1
    assert call(q_pos=256) == 1
    assert call(cache=_fake_cache(0)) == 1       # empty cache
    assert call(cache=None) == 1
    assert call(q=None) == 1
    assert call(out=ctypes.c_void_p(FAKE + 2)) == 1
    assert call(rope=ctypes.c_void_p(FAKE + 8)) == 1
    assert call(scale=float("inf")) == 1


def test_rope_init_host_errors(lib):
    cfg = _cfg()
    lay = kvq.layout(cfg, 2)
    p = ctypes.c_void_p(FAKE)
    assert lib.kvq_rope_init(ctypes.byref(cfg), 1e4, p, lay.rope_bytes - 8, None) == 4
    assert lib.kvq_rope_init(ctypes.byref(cfg), 0.0, p, lay.rope_bytes, None) == 1
    assert lib.kvq_rope_init(ctypes.byref(cfg), 1e4, None, lay.rope_bytes, None) == 1


def test_decode_step_host_errors(lib):
    cfg = _cfg()
    lay = kvq.layout(cfg, 8)
    p = ctypes.c_void_p(FAKE)
    ws = lay.workspace_bytes
    r = _fake_cache(100)

    def call(cache=r, k=p, v=p, q=p, H_q=8, rope=None, scale=0.1, out=p, w=p, wsb=ws, c=cfg):
        return lib.kvq_decode_step(ctypes.byref(c), None if cache is None else ctypes.byref(cache), k, v, q,
                                   H_q, rope, scale, out, w, wsb, None)

    full = _fake_cache(256)
    assert call(cache=full) == 3 and full.T_cur == 256      # no room for the new token
    assert call(wsb=ws - 1) == 4
    assert call(H_q=6) == 2
    assert call(c=_cfg(bits=7)) == 2
    assert call(cache=None) == 1
    assert call(k=None) == 1
    assert call(v=ctypes.c_void_p(FAKE + 8)) == 1
    assert call(q=None) == 1
    assert call(out=ctypes.c_void_p(FAKE + 2)) == 1
    assert call(w=None) == 1
    assert call(rope=ctypes.c_void_p(FAKE + 8)) == 1
    assert call(scale=float("nan")) == 1
    no_outl = _fake_cache(10, n_out=0)
    assert call(cache=no_outl) == 1                          # n_out = 1 needs the outlier buffers
    assert r.T_cur == 100                                    # nothing changed on any error


def test_paged_layout_sizes(lib):
    cfg = _cfg(B=3, H_kv=2, D=128, T_max=256, bits=3, key_block=128, value_group=32, outlier_frac=0.01)
    lay = kvq.paged_layout(cfg, 10, 8)
    H, Bk, D, cb, ng = 2, 128, 128, 48, 4
    per_block = [H * Bk * cb, H * D * 4, H * Bk * D * 2, H * Bk * 1 * 4, H * Bk * cb, H * Bk * ng * 4, H * Bk * 4]
    assert list(lay.stream_bytes) == per_block
    assert list(lay.bytes) == [x * (3 if i == 2 else 10) for i, x in enumerate(per_block)]
    assert lay.workspace_bytes == kvq.layout(cfg, 8).workspace_bytes
    out = kvq.Layout()
    assert lib.kvq_paged_layout(ctypes.byref(cfg), 0, 8, ctypes.byref(out)) == 2
    assert lib.kvq_paged_layout(ctypes.byref(cfg), 10, 3, ctypes.byref(out)) == 2
    assert lib.kvq_paged_layout(ctypes.byref(cfg), 1 << 30, 8, ctypes.byref(out)) == 2   # blocks x heads >= 2^31


def _fake_paged(max_len=0, n_blocks=8, n_out=1):
    r = kvq.PagedCacheRef()
    for i, n in enumerate(kvq.BUFFERS):
        setattr(r, n, FAKE * (i + 1) if (n_out or "outl" not in n) else None)
    r.block_table = FAKE * 9
    r.seq_len = FAKE * 10
    r.n_blocks = n_blocks
    r.max_len = max_len
    return r


def test_paged_host_errors(lib):
    cfg = _cfg()                                     # T_max 256, Bk 64, n_out 1
    p = ctypes.c_void_p(FAKE)
    r = _fake_paged(200)
    app = lambda c=r, n=1, k=p, v=p, cf=cfg: lib.kvq_paged_append(ctypes.byref(cf), None if c is None else ctypes.byref(c),
                                                                 k, v, n, None)
    assert app(n=57) == 3 and r.max_len == 200       # 200 + 57 > 256
    assert app(n=-1) == 1
    assert app(n=0) == 0
    assert app(c=None) == 1
    assert app(k=None) == 1
    assert app(v=ctypes.c_void_p(FAKE + 4)) == 1
    assert app(cf=_cfg(bits=9)) == 2
    for field, val in (("block_table", None), ("seq_len", FAKE + 2), ("n_blocks", 0), ("max_len", -1),
                       ("max_len", 300), ("k_tail", FAKE + 8)):
        bad = _fake_paged(10)
        setattr(bad, field, val)
        assert app(c=bad) == 1, field
    assert app(c=_fake_paged(10, n_out=0)) == 1       # n_out = 1 needs the outlier pools
    lay = kvq.layout(cfg, 8)
    ws = lay.workspace_bytes
    dec = lambda c=r, q=p, H_q=8, rope=None, scale=0.1, out=p, w=p, wsb=ws: lib.kvq_paged_decode_attn(
        ctypes.byref(cfg), None if c is None else ctypes.byref(c), q, H_q, rope, scale, out, w, wsb, None)
    assert dec(wsb=ws - 1) == 4
    assert dec(H_q=6) == 2
    assert dec(c=None) == 1
    assert dec(q=None) == 1
    assert dec(out=ctypes.c_void_p(FAKE + 2)) == 1
    assert dec(rope=ctypes.c_void_p(FAKE + 8)) == 1
    assert dec(scale=float("inf")) == 1
    assert dec(c=_fake_paged(10, n_blocks=-3)) == 1


def test_fit_levels_matches_the_oracle_fit(lib):
    import numpy as np
    from oracle import oracle_cpp as oc
    rng = np.random.default_rng(31)
    for bits in (2, 3, 4, 8):
        u = rng.beta(2.0, 4.0, 5000)
        got = kvq.fit_levels(u, bits, 60)
        want = oc.fit_levels(u, bits, 60)
        assert got[0] == 0 and got[-1] == 1 and np.all(np.diff(got) > 0)
        # the two sum a cell's samples in different orders: within a binary32 ulp
        assert np.all(np.abs(got.astype(np.float64) - want.astype(np.float64)) <= np.spacing(want))
    bad = np.array([0.5, 1.2])
    with pytest.raises(kvq.KvqError):
        kvq.fit_levels(bad, 2)


def test_fit_levels_clustered_samples_stay_increasing(lib):
    """Two clusters 1e-9 apart across a starting midpoint of the 8-bit grid:
    the k-means gives them two levels that are distinct in binary64 but round
    to one binary32 value; the library's table must still increase strictly
    and be accepted by the level-table calls."""
    import numpy as np
    mid = 127.5 / 255
    u = np.concatenate([np.full(4000, mid - 5e-10), np.full(4000, mid + 5e-10)])
    got = kvq.fit_levels(u, 8, 40)
    assert got[0] == 0 and got[-1] == 1 and np.all(np.diff(got.astype(np.float64)) > 0)
    assert np.any(np.abs(got - np.float32(mid)) <= np.spacing(np.float32(mid)))   # the clusters got their levels
    cfg = kvq.make_config(1, 2, 128, 256, 8, 64, 64, 0.0)
    p = ctypes.c_void_p(FAKE)
    r = _fake_cache(64)
    # n_new = 0: every check of the table runs, nothing touches a device
    assert lib.kvq_append_levels(ctypes.byref(cfg), ctypes.byref(r), p, p, 0,
                                 got.ctypes.data_as(ctypes.c_void_p), None) == 0


def test_levels_host_errors(lib):
    import numpy as np
    cfg = _cfg()                                    # bits 4, Bk 64, T_max 256, n_out 1
    p = ctypes.c_void_p(FAKE)
    good = np.linspace(0, 1, 16).astype(np.float32)
    lv = lambda a: np.ascontiguousarray(a, dtype=np.float32).ctypes.data_as(ctypes.c_void_p)
    r = _fake_cache(64)
    app = lambda levels, n=64, c=r: lib.kvq_append_levels(ctypes.byref(cfg), ctypes.byref(c), p, p, n, levels, None)
    assert app(lv(good), n=256) == 3                     # capacity
    not_zero = good.copy(); not_zero[0] = 0.01
    not_one = good.copy(); not_one[-1] = 0.99
    flat = good.copy(); flat[5] = flat[4]
    for bad in (not_zero, not_one, flat):
        assert app(lv(bad)) == 1
    assert app(None) == 1
    assert r.T_cur == 64
    lay = kvq.layout(cfg, 8)
    dec = lambda levels, c=r: lib.kvq_decode_attn_levels(ctypes.byref(cfg), ctypes.byref(c), p, 8, 63, None, 0.1, p,
                                                         p, lay.workspace_bytes, levels, None)
    assert dec(lv(flat)) == 1

"""ctypes front end of the C++ oracle (``kvq_oracle.cpp``).

TEST INFRASTRUCTURE ONLY (tests, smoke check, the benchmark's CPU baseline).
``build()`` compiles the shared library beside this file with plain g++
(``-O2 -ffp-contract=off``, no fast-math), so each float step is one IEEE
operation rounded to nearest on both x86-64 and aarch64 hosts.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(_HERE, "kvq_oracle.cpp")
LIB = os.path.join(_HERE, "libkvq_oracle.so")
_lib = None


def build(force: bool = False) -> str:
    if force or not os.path.exists(LIB) or os.path.getmtime(LIB) < os.path.getmtime(SRC):
        tmp = LIB + f".tmp{os.getpid()}"
        subprocess.check_call([
            "g++", "-O2", "-std=c++17", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
            "-shared", "-pthread", SRC, "-o", tmp,
        ])
        os.replace(tmp, LIB)
    return LIB


def lib():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(LIB)
        P = ctypes.c_void_p
        i = ctypes.c_int
        d = ctypes.c_double
        L.kvqo_encode.argtypes = [i] * 7 + [P] * 9 + [i]
        L.kvqo_dequant.argtypes = [i] * 7 + [P] * 9 + [i]
        L.kvqo_attention.argtypes = [i, i, i, i, P, P, P, d, d, d, d, P, i]
        L.kvqo_select_outliers.argtypes = [i, P, i, P, P]
        L.kvqo_group_params.argtypes = [i, P, P, i, P, P]
        L.kvqo_quantize.argtypes = [i, P, ctypes.c_uint16, ctypes.c_uint16, i, P]
        L.kvqo_half_up.argtypes = [ctypes.c_float]
        L.kvqo_half_up.restype = ctypes.c_uint16
        L.kvqo_half_to_double.argtypes = [ctypes.c_uint16]
        L.kvqo_half_to_double.restype = ctypes.c_double
        L.kvqo_pack_row.argtypes = [i, P, i, P]
        L.kvqo_rope.argtypes = [i, P, d, d, P]
        L.kvqo_encode_levels.argtypes = [i] * 7 + [P] * 10 + [i]
        L.kvqo_encode_window.argtypes = [i] * 8 + [P] * 10 + [i]
        L.kvqo_dequant_levels.argtypes = [i] * 7 + [P] * 10 + [i]
        L.kvqo_group_params_levels.argtypes = [i, P, P, P, P]
        L.kvqo_quantize_levels.argtypes = [i, P, ctypes.c_uint16, ctypes.c_uint16, i, P, P]
        L.kvqo_fit_levels.argtypes = [ctypes.c_size_t, P, i, i, P]
        _lib = L
    return _lib


def _p(a):
    return a.ctypes.data_as(ctypes.c_void_p)


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


def encode(K, V, bits, Bk, Gv, n_out, nthreads=None, levels=None, window=None):
    """Encode streams K, V [P, T, D] fp16; same dict layout as ``oracle_np.encode``.
    ``levels``: a table of 2^bits sorted levels in [0, 1] (non-uniform codes;
    the scale slot then holds the group's range), or None (uniform grid).
    ``window``: key statistics over the most recent `window` tokens (a
    multiple of Bk; None: the block alone)."""
    K = np.ascontiguousarray(K, dtype=np.float16)
    V = np.ascontiguousarray(V, dtype=np.float16)
    P, T, D = K.shape
    nb = T // Bk
    rb = D * bits // 8
    out = {
        "k_codes": np.zeros((P, T, rb), np.uint8),
        "k_meta": np.zeros((P, nb, D, 2), np.uint16),
        "k_tail": np.zeros((P, Bk, D), np.float16),
        "k_outl": np.zeros((P, T, n_out, 2), np.uint16),
        "v_codes": np.zeros((P, T, rb), np.uint8),
        "v_meta": np.zeros((P, T, D // Gv, 2), np.uint16),
        "v_outl": np.zeros((P, T, n_out, 2), np.uint16),
    }
    lv = None if levels is None else _levels(levels, bits)
    rc = lib().kvqo_encode_window(P, T, D, bits, Bk, Gv, n_out, Bk if window is None else int(window), _p(K),
                                  _p(V), _p(out["k_codes"]), _p(out["k_meta"]), _p(out["k_tail"]),
                                  _p(out["k_outl"]), _p(out["v_codes"]), _p(out["v_meta"]), _p(out["v_outl"]),
                                  None if lv is None else _p(lv), nthreads or default_threads())
    if rc:
        raise ValueError("oracle encode: bad shape")
    return out


def _levels(levels, bits):
    lv = np.ascontiguousarray(levels, dtype=np.float32)
    if lv.shape != (1 << bits,) or np.any(np.diff(lv) <= 0):
        raise ValueError(f"levels: {1 << bits} increasing binary32 values expected")
    return lv


def dequant(enc, T, D, bits, Bk, Gv, n_out, nthreads=None, levels=None):
    P = enc["v_codes"].shape[0]
    Kh = np.zeros((P, T, D), np.float64)
    Vh = np.zeros((P, T, D), np.float64)
    e = {k: np.ascontiguousarray(v) for k, v in enc.items()}
    lv = None if levels is None else _levels(levels, bits)
    rc = lib().kvqo_dequant_levels(P, T, D, bits, Bk, Gv, n_out, _p(e["k_codes"]), _p(e["k_meta"]),
                                   _p(e["k_tail"]), _p(e["k_outl"]), _p(e["v_codes"]), _p(e["v_meta"]),
                                   _p(e["v_outl"]), _p(Kh), _p(Vh), None if lv is None else _p(lv),
                                   nthreads or default_threads())
    if rc:
        raise ValueError("oracle dequant: bad shape")
    return Kh, Vh


def attention(Kh, Vh, q, q_pos, theta, sm_scale, pos_offset=0.0, nthreads=None):
    Kh = np.ascontiguousarray(Kh, dtype=np.float64)
    Vh = np.ascontiguousarray(Vh, dtype=np.float64)
    q = np.ascontiguousarray(q, dtype=np.float16)
    P, T, D = Kh.shape
    G = q.shape[1]
    out = np.zeros((P, G, D), np.float64)
    rc = lib().kvqo_attention(P, T, D, G, _p(Kh), _p(Vh), _p(q), float(q_pos), float(pos_offset),
                              float(theta), float(sm_scale), _p(out), nthreads or default_threads())
    if rc:
        raise ValueError("oracle attention: bad shape")
    return out


def select_outliers(x, n_out):
    x = np.ascontiguousarray(x, dtype=np.float16)
    idx = np.zeros(n_out, np.uint16)
    val = np.zeros(n_out, np.uint16)
    lib().kvqo_select_outliers(x.size, _p(x), n_out, _p(idx), _p(val))
    return idx, val.view(np.float16)


def group_params(x, bits, excluded=None):
    x = np.ascontiguousarray(x, dtype=np.float16)
    ex = None if excluded is None else np.ascontiguousarray(excluded, dtype=np.uint8)
    s = np.zeros(1, np.uint16)
    z = np.zeros(1, np.uint16)
    lib().kvqo_group_params(x.size, _p(x), None if ex is None else _p(ex), bits, _p(s), _p(z))
    return s.view(np.float16)[0], z.view(np.float16)[0]


def quantize(x, s, z, bits):
    x = np.ascontiguousarray(x, dtype=np.float16)
    codes = np.zeros(x.size, np.int32)
    sb = int(np.float16(s).view(np.uint16))
    zb = int(np.float16(z).view(np.uint16))
    lib().kvqo_quantize(x.size, _p(x), sb, zb, bits, _p(codes))
    return codes


def half_up(x: float) -> np.float16:
    return np.uint16(lib().kvqo_half_up(float(np.float32(x)))).view(np.float16)


def half_to_double(h) -> float:
    return lib().kvqo_half_to_double(int(np.float16(h).view(np.uint16)))


def pack_row(codes, bits):
    codes = np.ascontiguousarray(codes, dtype=np.int32)
    out = np.zeros(codes.size * bits // 8, np.uint8)
    if lib().kvqo_pack_row(codes.size, _p(codes), bits, _p(out)):
        raise ValueError("D*bits must be a multiple of 8")
    return out


def rope(x, pos, theta):
    x = np.ascontiguousarray(x, dtype=np.float64)
    y = np.zeros_like(x)
    lib().kvqo_rope(x.size, _p(x), float(pos), float(theta), _p(y))
    return y


def group_params_levels(x, excluded=None):
    """Range r (fp16, rounded up) and zero z of one group, for a level table."""
    x = np.ascontiguousarray(x, dtype=np.float16)
    ex = None if excluded is None else np.ascontiguousarray(excluded, dtype=np.uint8)
    r = np.zeros(1, np.uint16)
    z = np.zeros(1, np.uint16)
    lib().kvqo_group_params_levels(x.size, _p(x), None if ex is None else _p(ex), _p(r), _p(z))
    return r.view(np.float16)[0], z.view(np.float16)[0]


def quantize_levels(x, r, z, bits, levels):
    x = np.ascontiguousarray(x, dtype=np.float16)
    codes = np.zeros(x.size, np.int32)
    lv = _levels(levels, bits)
    lib().kvqo_quantize_levels(x.size, _p(x), int(np.float16(r).view(np.uint16)),
                               int(np.float16(z).view(np.uint16)), bits, _p(lv), _p(codes))
    return codes


def fit_levels(u, bits, iters=100):
    """Level table of 2^bits values fitted to samples u in [0, 1] (1-D k-means)."""
    u = np.ascontiguousarray(u, dtype=np.float64)
    lv = np.zeros(1 << bits, np.float32)
    if lib().kvqo_fit_levels(u.size, _p(u), bits, int(iters), _p(lv)):
        raise ValueError("bad bits or iters")
    return lv

"""Shared helpers of the GPU parity tests: build a cache through the C ABI,
regenerate the same inputs on the host, run the oracle on them, compare.

Nothing here feeds a CUDA-path value into the oracle: the oracle encodes the
host-regenerated fp16 inputs itself; only the comparison reads GPU buffers.
"""
from __future__ import annotations

import math

import numpy as np
import torch

import bit_quantized_kv_append_gb300 as kvq
import kvq_inputs as ki
from oracle import oracle_cpp as oc

ATOL, RTOL = 2e-3, 1e-2   # decode tolerance: max-abs, and relative (2-norm)


def n_out_of(w: ki.Workload) -> int:
    return 0 if w.outlier_frac == 0 else max(1, int(math.floor(w.outlier_frac * w.D)))


def make_cache(w: ki.Workload, T_max: int, device="cuda") -> kvq.QuantizedKVCache:
    return kvq.QuantizedKVCache(w.B, w.H_kv, w.D, T_max, w.bits, w.key_block, w.value_group,
                                w.outlier_frac, H_q=w.H_q, rope_theta=w.rope_theta, device=device)


def append_pieces(cache, K, V, pieces):
    """Append K, V [B, H, T, D] (device) in consecutive pieces of the given sizes."""
    t = 0
    for n in pieces:
        cache.append(K[:, :, t:t + n].contiguous(), V[:, :, t:t + n].contiguous())
        t += n
    assert t == K.shape[2]


def host_streams(w: ki.Workload, streams, T: int, layer: int = 0):
    """fp16 K, V [P, T, D] of the given (b, h) streams, regenerated with numpy."""
    return ki.streams_np(w, streams, T, layer)


def compare_streams(cache, streams, enc, T: int):
    """Bit-exact comparison of every buffer of the given streams with the oracle."""
    v = {k: t.cpu().numpy() for k, t in cache.views().items()}
    Bk = cache.cfg.key_block
    nb = T // Bk
    tail = T - nb * Bk
    for p, (b, h) in enumerate(streams):
        def eq(name, gpu, ora):
            g = np.ascontiguousarray(gpu).view(np.uint8)
            o = np.ascontiguousarray(ora).view(np.uint8)
            if not np.array_equal(g, o):
                bad = np.argwhere(np.asarray(gpu).view(np.uint8) != np.asarray(ora).view(np.uint8))
                raise AssertionError(f"{name} differs for stream {(b, h)}: {len(bad)} bytes, first {bad[:5].tolist()}")
        eq("v_codes", v["v_codes"][b, h, :T], enc["v_codes"][p])
        eq("v_meta", v["v_meta"][b, h, :T], enc["v_meta"][p])
        eq("k_codes", v["k_codes"][b, h, :nb * Bk], enc["k_codes"][p, :nb * Bk])
        eq("k_meta", v["k_meta"][b, h, :nb], enc["k_meta"][p])
        eq("k_tail", v["k_tail"][b, h, :tail], enc["k_tail"][p, :tail])
        if cache.n_out:
            eq("v_outl", v["v_outl"][b, h, :T], enc["v_outl"][p])
            eq("k_outl", v["k_outl"][b, h, :nb * Bk], enc["k_outl"][p, :nb * Bk])


def oracle_encode(w, K, V):
    return oc.encode(K, V, w.bits, w.key_block, w.value_group, n_out_of(w))


def oracle_decode(w, enc, T, q_heads, q_pos, sm_scale=None):
    """Float64 attention of q_heads [P, G, D] (fp16) on the oracle's own encoding."""
    Kh, Vh = oc.dequant(enc, T, w.D, w.bits, w.key_block, w.value_group, n_out_of(w))
    scale = 1.0 / math.sqrt(w.D) if sm_scale is None else sm_scale
    return oc.attention(Kh, Vh, q_heads, q_pos, w.rope_theta, scale)


def check_decode(gpu_out: np.ndarray, ref: np.ndarray, what=""):
    g = gpu_out.astype(np.float64)
    err = np.abs(g - ref)
    max_abs = float(err.max())
    rel = float(np.linalg.norm(g - ref) / max(np.linalg.norm(ref), 1e-30))
    assert max_abs <= ATOL, f"{what}: max abs error {max_abs:.3g} > {ATOL}"
    assert rel <= RTOL, f"{what}: relative error {rel:.3g} > {RTOL}"
    return max_abs, rel


def q_of_streams(q: np.ndarray, w: ki.Workload, streams):
    """The G query heads of each (b, h_kv) stream: q[b, h*G:(h+1)*G]."""
    return np.stack([q[b, h * w.G:(h + 1) * w.G] for (b, h) in streams])


def sync():
    torch.cuda.synchronize()

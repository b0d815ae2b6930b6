"""Seeded synthetic inputs for the KV-cache quantizer and decode attention.

This module holds no quantization or attention arithmetic: only the workload
shapes and the random inputs. It is the one piece shared by the CUDA-path tests
and benchmark and by the CPU oracle checks, so both sides see the same fp16
tensors.

Distribution (per layer), following the workloads the KVQuant summary targets
(keys with strong per-channel spread and a few outlier channels; values and
queries near-normal):
  * sigma[h_kv, c] ~ LogNormal(0, 0.5), drawn with numpy PCG64 seeded by
    (seed, layer); per kv head two distinct channels get sigma * 20;
  * K[t, c] = fp16(z * sigma[h_kv, c]); V = fp16(z); q = fp16(z * fp32(1/sqrt(D)));
    z ~ approximately N(0, 1).

z comes from a counter-based generator so any (layer, b, h, t) slice can be
regenerated alone, on the host with numpy or on the device with torch, with the
same bits: u = splitmix64(key + (i + 1) * GAMMA) (Steele, Lea & Flood's
SplitMix, with Vigna's splitmix64 output mix); z = (sum of the four 16-bit
fields of u - 2 * 65535) / sqrt((65536^2 - 1) / 3), an Irwin-Hall(4) sum
scaled to unit variance (range +-3.46). Every step is integer arithmetic
except two binary32 multiplies and one rounding to fp16, which numpy and
torch (CPU or CUDA) perform identically.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

GAMMA = 0x9E3779B97F4A7C15
MIX1 = 0xBF58476D1CE4E5B9
MIX2 = 0x94D049BB133111EB
M64 = (1 << 64) - 1
NORM_C = np.float32(1.0 / math.sqrt((65536.0 ** 2 - 1.0) / 3.0))
TAG_K, TAG_V, TAG_Q = 1, 2, 3


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H_q: int
    H_kv: int
    D: int
    T: int
    bits: int
    key_block: int
    value_group: int
    outlier_frac: float
    rope_theta: float
    seed: int
    layers: int = 1

    @property
    def G(self) -> int:
        return self.H_q // self.H_kv

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


# The five workloads of the decode study (shapes of Llama-7B / Llama-3-8B style
# models); "int3"/"int2" are the aggressive-bits variants of "gqa8b".
WORKLOADS = {
    "tiny_mha": Workload("tiny_mha", 1, 4, 4, 64, 512, 4, 64, 64, 0.0, 0.0, 0),
    "mha7b": Workload("mha7b", 8, 32, 32, 128, 32768, 4, 64, 64, 0.0, 1e4, 2),
    "gqa8b": Workload("gqa8b", 4, 32, 8, 128, 131072, 4, 64, 64, 0.01, 5e5, 3),
    "int3": Workload("int3", 4, 32, 8, 128, 131072, 3, 128, 32, 0.01, 5e5, 4),
    "int2": Workload("int2", 4, 32, 8, 128, 131072, 2, 128, 32, 0.01, 5e5, 4),
    "long1m": Workload("long1m", 1, 32, 8, 128, 1 << 20, 4, 64, 64, 0.01, 5e5, 5, layers=32),
    # 8-bit variant of the "gqa8b" shape (the prefill-append variant at INT8)
    "int8": Workload("int8", 4, 32, 8, 128, 131072, 8, 64, 64, 0.01, 5e5, 6),
}


# ------------------------------------------------------------------ generator
def _mix64_int(z: int) -> int:
    z &= M64
    z = ((z ^ (z >> 30)) * MIX1) & M64
    z = ((z ^ (z >> 27)) * MIX2) & M64
    return z ^ (z >> 31)


def stream_key(seed: int, tag: int, layer: int, b: int, h: int) -> int:
    """64-bit key of one (tensor, layer, batch, head) stream."""
    k = _mix64_int(seed * GAMMA + tag)
    k = _mix64_int(k + ((layer * 4096 + b) * 4096 + h))
    return k


def _normal_np(key: int, start: int, count: int) -> np.ndarray:
    i = np.arange(start + 1, start + 1 + count, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = np.uint64(key) + i * np.uint64(GAMMA)
        z = (z ^ (z >> np.uint64(30))) * np.uint64(MIX1)
        z = (z ^ (z >> np.uint64(27))) * np.uint64(MIX2)
        z = z ^ (z >> np.uint64(31))
    m = np.uint64(0xFFFF)
    s = ((z & m) + ((z >> np.uint64(16)) & m) + ((z >> np.uint64(32)) & m)
         + ((z >> np.uint64(48)) & m)).astype(np.int64) - 131070
    return s.astype(np.float32) * NORM_C


def _s64(x: int) -> int:
    x &= M64
    return x - (1 << 64) if x >> 63 else x


def _normal_torch(key: int, start: int, count: int, device):
    import torch
    i = torch.arange(start + 1, start + 1 + count, dtype=torch.int64, device=device)
    z = i * _s64(GAMMA) + _s64(key)
    z = (z ^ ((z >> 30) & ((1 << 34) - 1))) * _s64(MIX1)
    z = (z ^ ((z >> 27) & ((1 << 37) - 1))) * _s64(MIX2)
    z = z ^ ((z >> 31) & ((1 << 33) - 1))
    s = (z & 0xFFFF) + ((z >> 16) & 0xFFFF) + ((z >> 32) & 0xFFFF) + ((z >> 48) & 0xFFFF)
    s = (s - 131070).to(torch.float32)
    return s * torch.tensor(float(NORM_C), dtype=torch.float32, device=device)


# ------------------------------------------------------------------ tensors
def channel_sigma(w: Workload, layer: int = 0) -> np.ndarray:
    """sigma[h_kv, c] (float32): LogNormal(0, 0.5), two channels per head x20."""
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence([w.seed, layer])))
    sigma = rng.lognormal(0.0, 0.5, size=(w.H_kv, w.D))
    for h in range(w.H_kv):
        ch = rng.choice(w.D, size=2, replace=False)
        sigma[h, ch] *= 20.0
    return sigma.astype(np.float32)


def keys_np(w: Workload, layer: int, b: int, h: int, t0: int, n: int, sigma=None) -> np.ndarray:
    """fp16 keys [n, D] of stream (layer, b, h_kv), positions t0 .. t0+n-1."""
    sigma = channel_sigma(w, layer) if sigma is None else sigma
    z = _normal_np(stream_key(w.seed, TAG_K, layer, b, h), t0 * w.D, n * w.D).reshape(n, w.D)
    return (z * sigma[h][None, :]).astype(np.float16)


def values_np(w: Workload, layer: int, b: int, h: int, t0: int, n: int) -> np.ndarray:
    z = _normal_np(stream_key(w.seed, TAG_V, layer, b, h), t0 * w.D, n * w.D).reshape(n, w.D)
    return z.astype(np.float16)


def queries_np(w: Workload, layer: int, step: int) -> np.ndarray:
    """fp16 queries [B, H_q, D] of one decode step."""
    out = np.empty((w.B, w.H_q, w.D), np.float16)
    c = np.float32(1.0 / math.sqrt(w.D))
    for b in range(w.B):
        z = _normal_np(stream_key(w.seed, TAG_Q, layer, b, step), 0, w.H_q * w.D)
        out[b] = (z * c).astype(np.float16).reshape(w.H_q, w.D)
    return out


def streams_np(w: Workload, streams, T: int, layer: int = 0, chunk: int = 1 << 16):
    """fp16 K, V [P, T, D] of the given (b, h_kv) streams, positions 0 .. T-1."""
    sigma = channel_sigma(w, layer)
    K = np.empty((len(streams), T, w.D), np.float16)
    V = np.empty((len(streams), T, w.D), np.float16)
    for p, (b, h) in enumerate(streams):
        for t0 in range(0, T, chunk):
            n = min(chunk, T - t0)
            K[p, t0:t0 + n] = keys_np(w, layer, b, h, t0, n, sigma)
            V[p, t0:t0 + n] = values_np(w, layer, b, h, t0, n)
    return K, V


def kv_torch(w: Workload, layer: int, t0: int, n: int, device, sigma=None, which="kv"):
    """fp16 K and V [B, H_kv, n, D] for positions t0 .. t0+n-1, built on ``device``."""
    import torch
    sigma = channel_sigma(w, layer) if sigma is None else sigma
    sig = torch.from_numpy(sigma).to(device)
    K = torch.empty((w.B, w.H_kv, n, w.D), dtype=torch.float16, device=device) if "k" in which else None
    V = torch.empty((w.B, w.H_kv, n, w.D), dtype=torch.float16, device=device) if "v" in which else None
    chunk_rows = max(1, (1 << 24) // w.D)
    for b in range(w.B):
        for h in range(w.H_kv):
            for r0 in range(0, n, chunk_rows):
                r = min(chunk_rows, n - r0)
                start = (t0 + r0) * w.D
                if K is not None:
                    z = _normal_torch(stream_key(w.seed, TAG_K, layer, b, h), start, r * w.D, device)
                    K[b, h, r0:r0 + r] = (z.view(r, w.D) * sig[h][None, :]).to(torch.float16)
                if V is not None:
                    z = _normal_torch(stream_key(w.seed, TAG_V, layer, b, h), start, r * w.D, device)
                    V[b, h, r0:r0 + r] = z.view(r, w.D).to(torch.float16)
    return K, V


def queries_torch(w: Workload, layer: int, step: int, device):
    import torch
    out = torch.empty((w.B, w.H_q, w.D), dtype=torch.float16, device=device)
    c = torch.tensor(float(np.float32(1.0 / math.sqrt(w.D))), dtype=torch.float32, device=device)
    for b in range(w.B):
        z = _normal_torch(stream_key(w.seed, TAG_Q, layer, b, step), 0, w.H_q * w.D, device)
        out[b] = (z * c).to(torch.float16).view(w.H_q, w.D)
    return out

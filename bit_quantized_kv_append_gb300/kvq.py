"""Python binding of libkvq (ctypes): argument marshalling only.

Every step of append and decode runs in the library's CUDA kernels; PyTorch
only provides device memory and streams. There is no CPU fallback: if the
library is missing, the calls raise.

Entry points mirror include/kvq.h: ``layout``, ``rope_init``, ``append``,
``decode_attn``, ``decode_step``, ``decode_attn_noalloc``, ``paged_layout``,
``paged_append``, ``paged_decode_attn``, ``fit_levels``, ``append_levels``,
``decode_attn_levels``. ``QuantizedKVCache`` owns one layer's
buffers; ``PagedKVCache`` owns the pools, block table and lengths of a paged,
ragged batch.
"""
from __future__ import annotations

import ctypes
import math
import os
from typing import Optional

import torch


BUFFERS = ("k_codes", "k_meta", "k_tail", "k_outl", "v_codes", "v_meta", "v_outl")
STATUS = {0: "KVQ_OK", 1: "KVQ_ERR_ARG", 2: "KVQ_ERR_UNSUPPORTED", 3: "KVQ_ERR_CAPACITY",
          4: "KVQ_ERR_WORKSPACE", 5: "KVQ_ERR_CUDA", 6: "KVQ_ERR_TIMEOUT"}
STATUS_TIMEOUT = 1          # bit of the device status word (first 4 bytes of a decode workspace)
WS_HEADER_BYTES = 256
EXPORTS = ("kvq_layout", "kvq_rope_init", "kvq_append", "kvq_append_window", "kvq_decode_attn", "kvq_decode_step",
           "kvq_paged_layout", "kvq_paged_append", "kvq_paged_decode_attn",
           "kvq_fit_levels", "kvq_append_levels", "kvq_decode_attn_levels", "kvq_decode_step_levels",
           "kvq_decode_attn_noalloc", "kvq_decode_attn_diag", "kvq_status_string", "kvq_version")


class KvqError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {STATUS.get(status, status)} ({_status_string(status)})")


class Config(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int32), ("H_kv", ctypes.c_int32), ("D", ctypes.c_int32),
                ("T_max", ctypes.c_int32), ("bits", ctypes.c_int32),
                ("key_block", ctypes.c_int32), ("value_group", ctypes.c_int32),
                ("outlier_frac", ctypes.c_float), ("flags", ctypes.c_int32)]


FLAG_PRECISE_SCORES = 1


class Layout(ctypes.Structure):
    _fields_ = [("bytes", ctypes.c_size_t * 7), ("stream_bytes", ctypes.c_size_t * 7),
                ("cache_bytes", ctypes.c_size_t), ("fp16_equiv_bytes", ctypes.c_size_t),
                ("rope_bytes", ctypes.c_size_t), ("workspace_bytes", ctypes.c_size_t),
                ("n_out", ctypes.c_int32), ("code_row_bytes", ctypes.c_int32)]


class CacheRef(ctypes.Structure):
    _fields_ = [(name, ctypes.c_void_p) for name in BUFFERS] + [("T_cur", ctypes.c_int32)]


class PagedCacheRef(ctypes.Structure):
    _fields_ = [(name, ctypes.c_void_p) for name in BUFFERS] + [
        ("block_table", ctypes.c_void_p), ("seq_len", ctypes.c_void_p),
        ("n_blocks", ctypes.c_int32), ("max_len", ctypes.c_int32)]


LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libkvq.so")
_LIB = None


def lib():
    """The loaded libkvq.so (raises if it has not been built)."""
    global _LIB
    if _LIB is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libkvq.so is not built ({LIB_PATH}); run "
                               "`python -m bit_quantized_kv_append_gb300.build`")
        L = ctypes.CDLL(LIB_PATH)
        vp, i32 = ctypes.c_void_p, ctypes.c_int32
        L.kvq_layout.argtypes = [ctypes.POINTER(Config), i32, ctypes.POINTER(Layout)]
        L.kvq_rope_init.argtypes = [ctypes.POINTER(Config), ctypes.c_double, vp, ctypes.c_size_t, vp]
        L.kvq_append.argtypes = [ctypes.POINTER(Config), ctypes.POINTER(CacheRef), vp, vp, i32, vp]
        L.kvq_append_window.argtypes = [ctypes.POINTER(Config), ctypes.POINTER(CacheRef), vp, vp, i32, i32, vp, vp]
        L.kvq_decode_attn.argtypes = [ctypes.POINTER(Config), ctypes.POINTER(CacheRef), vp, i32, i32,
                                      vp, ctypes.c_float, vp, vp, ctypes.c_size_t, vp]
        L.kvq_decode_step.argtypes = [ctypes.POINTER(Config), ctypes.POINTER(CacheRef), vp, vp, vp, i32,
                                      vp, ctypes.c_float, vp, vp, ctypes.c_size_t, vp]
        L.kvq_paged_layout.argtypes = [ctypes.POINTER(Config), i32, i32, ctypes.POINTER(Layout)]
        L.kvq_paged_append.argtypes = [ctypes.POINTER(Config), ctypes.POINTER(PagedCacheRef), vp, vp, i32, vp]
        L.kvq_paged_decode_attn.argtypes = [ctypes.POINTER(Config), ctypes.POINTER(PagedCacheRef), vp, i32, vp,
                                            ctypes.c_float, vp, vp, ctypes.c_size_t, vp]
        L.kvq_fit_levels.argtypes = [vp, ctypes.c_size_t, i32, i32, vp]
        L.kvq_append_levels.argtypes = [ctypes.POINTER(Config), ctypes.POINTER(CacheRef), vp, vp, i32, vp, vp]
        L.kvq_decode_attn_levels.argtypes = [ctypes.POINTER(Config), ctypes.POINTER(CacheRef), vp, i32, i32, vp,
                                             ctypes.c_float, vp, vp, ctypes.c_size_t, vp, vp]
        L.kvq_decode_step_levels.argtypes = [ctypes.POINTER(Config), ctypes.POINTER(CacheRef), vp, vp, vp, i32,
                                             vp, ctypes.c_float, vp, vp, ctypes.c_size_t, vp, vp]
        L.kvq_decode_attn_noalloc.argtypes = [ctypes.POINTER(Config), ctypes.POINTER(CacheRef), vp,
                                              i32, i32, vp, ctypes.c_float, vp, vp]
        L.kvq_decode_attn_diag.argtypes = [ctypes.POINTER(Config), ctypes.POINTER(CacheRef), vp, i32, i32, vp,
                                           ctypes.c_float, vp, vp, ctypes.c_size_t, ctypes.c_uint32, vp]
        L.kvq_status_string.argtypes = [ctypes.c_int]
        L.kvq_status_string.restype = ctypes.c_char_p
        L.kvq_version.restype = ctypes.c_char_p
        for fn in ("kvq_layout", "kvq_rope_init", "kvq_append", "kvq_append_window", "kvq_decode_attn", "kvq_decode_step",
                   "kvq_paged_layout", "kvq_paged_append", "kvq_paged_decode_attn", "kvq_fit_levels",
                   "kvq_append_levels", "kvq_decode_attn_levels", "kvq_decode_step_levels", "kvq_decode_attn_noalloc",
                   "kvq_decode_attn_diag"):
            getattr(L, fn).restype = ctypes.c_int
        _LIB = L
    return _LIB


def _status_string(status: int) -> str:
    try:
        return lib().kvq_status_string(status).decode()
    except Exception:  # noqa: BLE001 - message only
        return "?"


def _check(rc: int, what: str):
    if rc != 0:
        raise KvqError(rc, what)


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None or t.numel() == 0 else ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def make_config(B, H_kv, D, T_max, bits=4, key_block=64, value_group=64, outlier_frac=0.0,
                flags=0) -> Config:
    return Config(B, H_kv, D, T_max, bits, key_block, value_group, float(outlier_frac), int(flags))


def layout(cfg: Config, H_q: int) -> Layout:
    out = Layout()
    _check(lib().kvq_layout(ctypes.byref(cfg), int(H_q), ctypes.byref(out)), "kvq_layout")
    return out


def rope_init(cfg: Config, theta: float, table: torch.Tensor, stream=None):
    _check(lib().kvq_rope_init(ctypes.byref(cfg), float(theta), _ptr(table), table.numel() * table.element_size(),
                               _stream(stream)), "kvq_rope_init")


def append(cfg: Config, ref: CacheRef, k_new: torch.Tensor, v_new: torch.Tensor, n_new: int, stream=None):
    _check(lib().kvq_append(ctypes.byref(cfg), ctypes.byref(ref), _ptr(k_new), _ptr(v_new), int(n_new),
                            _stream(stream)), "kvq_append")


def append_window(cfg: Config, ref: CacheRef, k_new: torch.Tensor, v_new: torch.Tensor, n_new: int,
                  window: int, k_bstat: torch.Tensor, stream=None):
    _check(lib().kvq_append_window(ctypes.byref(cfg), ctypes.byref(ref), _ptr(k_new), _ptr(v_new), int(n_new),
                                   int(window), _ptr(k_bstat), _stream(stream)), "kvq_append_window")


def decode_attn(cfg: Config, ref: CacheRef, q: torch.Tensor, H_q: int, q_pos: int,
                rope: Optional[torch.Tensor], sm_scale: float, out: torch.Tensor,
                workspace: torch.Tensor, stream=None):
    _check(lib().kvq_decode_attn(ctypes.byref(cfg), ctypes.byref(ref), _ptr(q), int(H_q), int(q_pos),
                                 _ptr(rope), float(sm_scale), _ptr(out), _ptr(workspace),
                                 workspace.numel(), _stream(stream)), "kvq_decode_attn")


def decode_attn_diag(cfg: Config, ref: CacheRef, q: torch.Tensor, H_q: int, q_pos: int,
                     rope: Optional[torch.Tensor], sm_scale: float, out: torch.Tensor,
                     workspace: torch.Tensor, tx_pad: int, stream=None):
    _check(lib().kvq_decode_attn_diag(ctypes.byref(cfg), ctypes.byref(ref), _ptr(q), int(H_q), int(q_pos),
                                      _ptr(rope), float(sm_scale), _ptr(out), _ptr(workspace), workspace.numel(),
                                      int(tx_pad), _stream(stream)), "kvq_decode_attn_diag")


def decode_step(cfg: Config, ref: CacheRef, k_new: torch.Tensor, v_new: torch.Tensor, q: torch.Tensor,
                H_q: int, rope: Optional[torch.Tensor], sm_scale: float, out: torch.Tensor,
                workspace: torch.Tensor, stream=None):
    """kvq_decode_step: append one token per sequence, then decode attention
    of q at the new token's position over every cached token (ref.T_cur
    advances by one on success)."""
    _check(lib().kvq_decode_step(ctypes.byref(cfg), ctypes.byref(ref), _ptr(k_new), _ptr(v_new), _ptr(q),
                                 int(H_q), _ptr(rope), float(sm_scale), _ptr(out), _ptr(workspace),
                                 workspace.numel(), _stream(stream)), "kvq_decode_step")


def _host_levels(levels, bits):
    import numpy as np
    lv = np.ascontiguousarray(levels, dtype=np.float32)
    if lv.shape != (1 << bits,):
        raise ValueError(f"expected {1 << bits} levels, got {lv.shape}")
    return lv


def fit_levels(u, bits: int, iters: int = 100):
    """kvq_fit_levels: 2^bits levels (numpy float32) fitted to samples u in [0, 1]."""
    import numpy as np
    x = np.ascontiguousarray(u, dtype=np.float64).ravel()
    lv = np.zeros(1 << bits, np.float32)
    _check(lib().kvq_fit_levels(x.ctypes.data_as(ctypes.c_void_p), x.size, int(bits), int(iters),
                                lv.ctypes.data_as(ctypes.c_void_p)), "kvq_fit_levels")
    return lv


def append_levels(cfg: Config, ref: CacheRef, k_new: torch.Tensor, v_new: torch.Tensor, n_new: int, levels,
                  stream=None):
    lv = _host_levels(levels, cfg.bits)
    _check(lib().kvq_append_levels(ctypes.byref(cfg), ctypes.byref(ref), _ptr(k_new), _ptr(v_new), int(n_new),
                                   lv.ctypes.data_as(ctypes.c_void_p), _stream(stream)), "kvq_append_levels")


def decode_attn_levels(cfg: Config, ref: CacheRef, q: torch.Tensor, H_q: int, q_pos: int,
                       rope: Optional[torch.Tensor], sm_scale: float, out: torch.Tensor,
                       workspace: torch.Tensor, levels, stream=None):
    lv = _host_levels(levels, cfg.bits)
    _check(lib().kvq_decode_attn_levels(ctypes.byref(cfg), ctypes.byref(ref), _ptr(q), int(H_q), int(q_pos),
                                        _ptr(rope), float(sm_scale), _ptr(out), _ptr(workspace),
                                        workspace.numel(), lv.ctypes.data_as(ctypes.c_void_p), _stream(stream)),
           "kvq_decode_attn_levels")


def decode_step_levels(cfg: Config, ref: CacheRef, k_new: torch.Tensor, v_new: torch.Tensor, q: torch.Tensor,
                       H_q: int, rope: Optional[torch.Tensor], sm_scale: float, out: torch.Tensor,
                       workspace: torch.Tensor, levels, stream=None):
    """kvq_decode_step_levels: kvq_decode_step on a level-table cache."""
    lv = _host_levels(levels, cfg.bits)
    _check(lib().kvq_decode_step_levels(ctypes.byref(cfg), ctypes.byref(ref), _ptr(k_new), _ptr(v_new), _ptr(q),
                                        int(H_q), _ptr(rope), float(sm_scale), _ptr(out), _ptr(workspace),
                                        workspace.numel(), lv.ctypes.data_as(ctypes.c_void_p), _stream(stream)),
           "kvq_decode_step_levels")


def decode_attn_noalloc(cfg: Config, ref: CacheRef, q: torch.Tensor, H_q: int, q_pos: int,
                        rope: Optional[torch.Tensor], sm_scale: float, out: torch.Tensor, stream=None):
    """kvq_decode_attn_noalloc: decode attention with the library's own fixed
    8 MiB device scratch instead of a workspace (see include/kvq.h)."""
    _check(lib().kvq_decode_attn_noalloc(ctypes.byref(cfg), ctypes.byref(ref), _ptr(q), int(H_q),
                                         int(q_pos), _ptr(rope), float(sm_scale), _ptr(out),
                                         _stream(stream)), "kvq_decode_attn_noalloc")


class QuantizedKVCache:
    """One layer's low-bit KV cache in device memory (buffers sized by kvq_layout)."""

    def __init__(self, B, H_kv, D, T_max, bits=4, key_block=64, value_group=64, outlier_frac=0.0,
                 H_q=None, rope_theta=0.0, device="cuda", rope_table: Optional[torch.Tensor] = None,
                 precise=False):
        self.cfg = make_config(B, H_kv, D, T_max, bits, key_block, value_group, outlier_frac,
                               FLAG_PRECISE_SCORES if precise else 0)
        self.H_q = H_q or H_kv
        self.layout = layout(self.cfg, self.H_q)
        self.device = torch.device(device)
        if self.device.type == "cuda" and self.device.index is None:
            self.device = torch.device("cuda", torch.cuda.current_device())
        self.buffers = {name: torch.empty(self.layout.bytes[i], dtype=torch.uint8, device=self.device)
                        for i, name in enumerate(BUFFERS)}
        self.workspace = torch.empty(self.layout.workspace_bytes, dtype=torch.uint8, device=self.device)
        self.workspace[:WS_HEADER_BYTES].zero_()      # the device status word starts cleared
        self.rope_theta = float(rope_theta)
        self.rope = rope_table
        if self.rope is None and self.rope_theta > 0:
            self.rope = torch.empty(self.layout.rope_bytes, dtype=torch.uint8, device=self.device)
            rope_init(self.cfg, self.rope_theta, self.rope)
        self.T_cur = 0

    def status(self) -> int:
        """The device status word of this cache's decode workspace (reads it
        back, which waits for the work queued so far)."""
        return int(self.workspace[:4].view(torch.int32).item())

    def clear_status(self):
        self.workspace[:WS_HEADER_BYTES].zero_()

    # -- shape helpers
    @property
    def n_out(self) -> int:
        return self.layout.n_out

    def ref(self) -> CacheRef:
        r = CacheRef()
        for name in BUFFERS:
            t = self.buffers[name]
            setattr(r, name, None if t.numel() == 0 else t.data_ptr())
        r.T_cur = self.T_cur
        return r

    def views(self) -> dict:
        """Typed views of the buffers, shaped as include/kvq.h documents."""
        c = self.cfg
        n_out, cb = self.layout.n_out, self.layout.code_row_bytes
        B, H, T = c.B, c.H_kv, c.T_max
        bf = self.buffers
        return {
            "k_codes": bf["k_codes"].view(B, H, T, cb),
            "k_meta": bf["k_meta"].view(torch.int16).view(B, H, T // c.key_block, c.D, 2),
            "k_tail": bf["k_tail"].view(torch.float16).view(B, H, c.key_block, c.D),
            "k_outl": bf["k_outl"].view(torch.int16).view(B, H, T, n_out, 2),
            "v_codes": bf["v_codes"].view(B, H, T, cb),
            "v_meta": bf["v_meta"].view(torch.int16).view(B, H, T, c.D // c.value_group, 2),
            "v_outl": bf["v_outl"].view(torch.int16).view(B, H, T, n_out, 2),
        }

    def reset(self, T_cur: int = 0):
        self.T_cur = int(T_cur)

    # -- the two paths
    def _check_kv(self, k_new, v_new):
        c = self.cfg
        for t in (k_new, v_new):
            if t.dtype != torch.float16 or not t.is_contiguous() or t.device != self.device:
                raise ValueError("k_new/v_new must be contiguous fp16 tensors on the cache device")
            if t.dim() != 4 or t.shape[0] != c.B or t.shape[1] != c.H_kv or t.shape[3] != c.D:
                raise ValueError(f"expected [B={c.B}, H_kv={c.H_kv}, n, D={c.D}], got {tuple(t.shape)}")
        if k_new.shape != v_new.shape:
            raise ValueError("k_new and v_new shapes differ")

    def append(self, k_new: torch.Tensor, v_new: torch.Tensor, stream=None):
        """k_new, v_new: fp16 [B, H_kv, n, D] on the cache's device (pre-RoPE keys)."""
        self._check_kv(k_new, v_new)
        ref = self.ref()
        append(self.cfg, ref, k_new, v_new, k_new.shape[2], stream)
        self.T_cur = ref.T_cur

    def append_window(self, k_new: torch.Tensor, v_new: torch.Tensor, window: int, stream=None):
        """kvq_append with key statistics over the last `window` tokens; the
        block statistics buffer (the size of K_META) is allocated on first use
        and kept with the cache."""
        self._check_kv(k_new, v_new)
        if getattr(self, "k_bstat", None) is None:
            self.k_bstat = torch.empty(self.layout.bytes[BUFFERS.index("k_meta")], dtype=torch.uint8,
                                       device=self.device)
        ref = self.ref()
        append_window(self.cfg, ref, k_new, v_new, k_new.shape[2], window, self.k_bstat, stream)
        self.T_cur = ref.T_cur

    def decode(self, q: torch.Tensor, q_pos: Optional[int] = None, sm_scale: Optional[float] = None,
               out: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
        """q: fp16 [B, H_q, D] pre-RoPE at position q_pos (default T_cur - 1)."""
        c = self.cfg
        if q.dtype != torch.float16 or not q.is_contiguous() or q.device != self.device:
            raise ValueError("q must be a contiguous fp16 tensor on the cache device")
        if tuple(q.shape) != (c.B, self.H_q, c.D):
            raise ValueError(f"expected q [B={c.B}, H_q={self.H_q}, D={c.D}], got {tuple(q.shape)}")
        if out is None:
            out = torch.empty_like(q)
        q_pos = self.T_cur - 1 if q_pos is None else q_pos
        sm_scale = 1.0 / math.sqrt(c.D) if sm_scale is None else sm_scale
        decode_attn(self.cfg, self.ref(), q, self.H_q, q_pos, self.rope, sm_scale, out,
                    self.workspace, stream)
        return out

    def append_levels(self, k_new: torch.Tensor, v_new: torch.Tensor, levels, stream=None):
        """Non-uniform codes against the level table ``levels`` (2^bits values,
        0 first, 1 last, increasing); any number of tokens (the keys of an
        unfinished key block wait as fp16, as in append)."""
        c = self.cfg
        for t in (k_new, v_new):
            if t.dtype != torch.float16 or not t.is_contiguous() or t.device != self.device:
                raise ValueError("k_new/v_new must be contiguous fp16 tensors on the cache device")
            if t.dim() != 4 or t.shape[0] != c.B or t.shape[1] != c.H_kv or t.shape[3] != c.D:
                raise ValueError(f"expected [B={c.B}, H_kv={c.H_kv}, n, D={c.D}], got {tuple(t.shape)}")
        ref = self.ref()
        append_levels(self.cfg, ref, k_new, v_new, k_new.shape[2], levels, stream)
        self.T_cur = ref.T_cur

    def decode_levels(self, q: torch.Tensor, levels, q_pos: Optional[int] = None,
                      sm_scale: Optional[float] = None, out: Optional[torch.Tensor] = None,
                      stream=None) -> torch.Tensor:
        """Decode attention over a cache filled by append_levels with the same table."""
        c = self.cfg
        if q.dtype != torch.float16 or not q.is_contiguous() or q.device != self.device:
            raise ValueError("q must be a contiguous fp16 tensor on the cache device")
        if tuple(q.shape) != (c.B, self.H_q, c.D):
            raise ValueError(f"expected q [B={c.B}, H_q={self.H_q}, D={c.D}], got {tuple(q.shape)}")
        if out is None:
            out = torch.empty_like(q)
        q_pos = self.T_cur - 1 if q_pos is None else q_pos
        sm_scale = 1.0 / math.sqrt(c.D) if sm_scale is None else sm_scale
        decode_attn_levels(self.cfg, self.ref(), q, self.H_q, q_pos, self.rope, sm_scale, out, self.workspace,
                           levels, stream)
        return out

    def decode_step_levels(self, k_new: torch.Tensor, v_new: torch.Tensor, q: torch.Tensor, levels,
                           sm_scale: Optional[float] = None, out: Optional[torch.Tensor] = None,
                           stream=None) -> torch.Tensor:
        """decode_step on a cache filled by append_levels, with the same table."""
        c = self.cfg
        for t in (k_new, v_new):
            if t.dtype != torch.float16 or not t.is_contiguous() or t.device != self.device:
                raise ValueError("k_new/v_new must be contiguous fp16 tensors on the cache device")
            if tuple(t.shape) != (c.B, c.H_kv, 1, c.D):
                raise ValueError(f"expected [B={c.B}, H_kv={c.H_kv}, 1, D={c.D}], got {tuple(t.shape)}")
        if q.dtype != torch.float16 or not q.is_contiguous() or q.device != self.device:
            raise ValueError("q must be a contiguous fp16 tensor on the cache device")
        if tuple(q.shape) != (c.B, self.H_q, c.D):
            raise ValueError(f"expected q [B={c.B}, H_q={self.H_q}, D={c.D}], got {tuple(q.shape)}")
        if out is None:
            out = torch.empty_like(q)
        sm_scale = 1.0 / math.sqrt(c.D) if sm_scale is None else sm_scale
        ref = self.ref()
        decode_step_levels(self.cfg, ref, k_new, v_new, q, self.H_q, self.rope, sm_scale, out, self.workspace,
                           levels, stream)
        self.T_cur = ref.T_cur
        return out

    def decode_step(self, k_new: torch.Tensor, v_new: torch.Tensor, q: torch.Tensor,
                    sm_scale: Optional[float] = None, out: Optional[torch.Tensor] = None,
                    stream=None) -> torch.Tensor:
        """One decode step: store the new token (k_new, v_new: fp16 [B, H_kv, 1, D],
        pre-RoPE key) at position T_cur and attend q (fp16 [B, H_q, D], pre-RoPE,
        at that position) over all T_cur + 1 tokens."""
        c = self.cfg
        for t in (k_new, v_new):
            if t.dtype != torch.float16 or not t.is_contiguous() or t.device != self.device:
                raise ValueError("k_new/v_new must be contiguous fp16 tensors on the cache device")
            if tuple(t.shape) != (c.B, c.H_kv, 1, c.D):
                raise ValueError(f"expected [B={c.B}, H_kv={c.H_kv}, 1, D={c.D}], got {tuple(t.shape)}")
        if q.dtype != torch.float16 or not q.is_contiguous() or q.device != self.device:
            raise ValueError("q must be a contiguous fp16 tensor on the cache device")
        if tuple(q.shape) != (c.B, self.H_q, c.D):
            raise ValueError(f"expected q [B={c.B}, H_q={self.H_q}, D={c.D}], got {tuple(q.shape)}")
        if out is None:
            out = torch.empty_like(q)
        sm_scale = 1.0 / math.sqrt(c.D) if sm_scale is None else sm_scale
        ref = self.ref()
        decode_step(self.cfg, ref, k_new, v_new, q, self.H_q, self.rope, sm_scale, out, self.workspace, stream)
        self.T_cur = ref.T_cur
        return out


# ----------------------------------------------------------------------------- paged, ragged batches
def paged_layout(cfg: Config, n_blocks: int, H_q: int) -> Layout:
    out = Layout()
    _check(lib().kvq_paged_layout(ctypes.byref(cfg), int(n_blocks), int(H_q), ctypes.byref(out)), "kvq_paged_layout")
    return out


def paged_append(cfg: Config, ref: PagedCacheRef, k_new: torch.Tensor, v_new: torch.Tensor, n_new: int,
                 stream=None):
    _check(lib().kvq_paged_append(ctypes.byref(cfg), ctypes.byref(ref), _ptr(k_new), _ptr(v_new), int(n_new),
                                  _stream(stream)), "kvq_paged_append")


def paged_decode_attn(cfg: Config, ref: PagedCacheRef, q: torch.Tensor, H_q: int, rope: Optional[torch.Tensor],
                      sm_scale: float, out: torch.Tensor, workspace: torch.Tensor, stream=None):
    _check(lib().kvq_paged_decode_attn(ctypes.byref(cfg), ctypes.byref(ref), _ptr(q), int(H_q), _ptr(rope),
                                       float(sm_scale), _ptr(out), _ptr(workspace), workspace.numel(),
                                       _stream(stream)), "kvq_paged_decode_attn")


class PagedKVCache:
    """One layer of a paged, ragged batch: pools of n_blocks physical key
    blocks (Bk tokens x H_kv heads each) shared by B sequences through
    ``block_table`` [B, T_max // Bk] (int32, device; the caller assigns
    blocks), per-sequence lengths ``seq_len`` [B] (int32, device), and each
    sequence's fp16 tail of keys. ``lengths`` mirrors seq_len on the host."""

    def __init__(self, B, H_kv, D, T_max, n_blocks, bits=4, key_block=64, value_group=64, outlier_frac=0.0,
                 H_q=None, rope_theta=0.0, device="cuda", rope_table: Optional[torch.Tensor] = None,
                 precise=False):
        self.cfg = make_config(B, H_kv, D, T_max, bits, key_block, value_group, outlier_frac,
                               FLAG_PRECISE_SCORES if precise else 0)
        self.H_q = H_q or H_kv
        self.n_blocks = int(n_blocks)
        self.layout = paged_layout(self.cfg, self.n_blocks, self.H_q)
        self.device = torch.device(device)
        if self.device.type == "cuda" and self.device.index is None:
            self.device = torch.device("cuda", torch.cuda.current_device())
        self.buffers = {name: torch.empty(self.layout.bytes[i], dtype=torch.uint8, device=self.device)
                        for i, name in enumerate(BUFFERS)}
        self.block_table = torch.zeros((B, T_max // key_block), dtype=torch.int32, device=self.device)
        self.seq_len = torch.zeros(B, dtype=torch.int32, device=self.device)
        self.lengths = [0] * B
        self.workspace = torch.empty(self.layout.workspace_bytes, dtype=torch.uint8, device=self.device)
        self.workspace[:WS_HEADER_BYTES].zero_()      # the device status word starts cleared
        self.rope_theta = float(rope_theta)
        self.rope = rope_table
        if self.rope is None and self.rope_theta > 0:
            self.rope = torch.empty(self.layout.rope_bytes, dtype=torch.uint8, device=self.device)
            rope_init(self.cfg, self.rope_theta, self.rope)

    @property
    def n_out(self) -> int:
        return self.layout.n_out

    def ref(self, seq: Optional[int] = None) -> PagedCacheRef:
        """The whole batch, or (seq = b) a one-sequence view for kvq_config.B = 1."""
        r = PagedCacheRef()
        for name in BUFFERS:
            t = self.buffers[name]
            setattr(r, name, None if t.numel() == 0 else t.data_ptr())
        r.block_table = self.block_table.data_ptr()
        r.seq_len = self.seq_len.data_ptr()
        r.n_blocks = self.n_blocks
        r.max_len = max(self.lengths) if seq is None else self.lengths[seq]
        if seq is not None:
            r.block_table += seq * self.block_table.shape[1] * 4
            r.seq_len += seq * 4
            r.k_tail += seq * self.layout.stream_bytes[BUFFERS.index("k_tail")]
        return r

    def _cfg_one(self) -> Config:
        c = self.cfg
        return make_config(1, c.H_kv, c.D, c.T_max, c.bits, c.key_block, c.value_group, c.outlier_frac, c.flags)

    def _check_kv(self, k_new, v_new, B):
        c = self.cfg
        for t in (k_new, v_new):
            if t.dtype != torch.float16 or not t.is_contiguous() or t.device != self.device:
                raise ValueError("k_new/v_new must be contiguous fp16 tensors on the cache device")
            if t.dim() != 4 or t.shape[0] != B or t.shape[1] != c.H_kv or t.shape[3] != c.D:
                raise ValueError(f"expected [B={B}, H_kv={c.H_kv}, n, D={c.D}], got {tuple(t.shape)}")
        if k_new.shape != v_new.shape:
            raise ValueError("k_new and v_new shapes differ")

    def append(self, k_new: torch.Tensor, v_new: torch.Tensor, stream=None):
        """n new tokens for every sequence (k_new, v_new: fp16 [B, H_kv, n, D]),
        each stored at its own length."""
        self._check_kv(k_new, v_new, self.cfg.B)
        n = k_new.shape[2]
        paged_append(self.cfg, self.ref(), k_new, v_new, n, stream)
        self.lengths = [x + n for x in self.lengths]

    def append_seq(self, b: int, k_new: torch.Tensor, v_new: torch.Tensor, stream=None):
        """n new tokens of sequence b alone (k_new, v_new: fp16 [1, H_kv, n, D])."""
        self._check_kv(k_new, v_new, 1)
        n = k_new.shape[2]
        paged_append(self._cfg_one(), self.ref(b), k_new, v_new, n, stream)
        self.lengths[b] += n

    def decode(self, q: torch.Tensor, sm_scale: Optional[float] = None, out: Optional[torch.Tensor] = None,
               stream=None) -> torch.Tensor:
        """q: fp16 [B, H_q, D], pre-RoPE; sequence b's query sits at its newest token."""
        c = self.cfg
        if q.dtype != torch.float16 or not q.is_contiguous() or q.device != self.device:
            raise ValueError("q must be a contiguous fp16 tensor on the cache device")
        if tuple(q.shape) != (c.B, self.H_q, c.D):
            raise ValueError(f"expected q [B={c.B}, H_q={self.H_q}, D={c.D}], got {tuple(q.shape)}")
        if out is None:
            out = torch.empty_like(q)
        sm_scale = 1.0 / math.sqrt(c.D) if sm_scale is None else sm_scale
        paged_decode_attn(self.cfg, self.ref(), q, self.H_q, self.rope, sm_scale, out, self.workspace, stream)
        return out

    def views(self) -> dict:
        """Typed views of the pools ([n_blocks, H_kv, ...]) and of K_TAIL ([B, H_kv, Bk, D])."""
        c = self.cfg
        n_out, cb, N, H, Bk = self.layout.n_out, self.layout.code_row_bytes, self.n_blocks, c.H_kv, c.key_block
        bf = self.buffers
        return {
            "k_codes": bf["k_codes"].view(N, H, Bk, cb),
            "k_meta": bf["k_meta"].view(torch.int16).view(N, H, c.D, 2),
            "k_tail": bf["k_tail"].view(torch.float16).view(c.B, H, Bk, c.D),
            "k_outl": bf["k_outl"].view(torch.int16).view(N, H, Bk, n_out, 2),
            "v_codes": bf["v_codes"].view(N, H, Bk, cb),
            "v_meta": bf["v_meta"].view(torch.int16).view(N, H, Bk, c.D // c.value_group, 2),
            "v_outl": bf["v_outl"].view(torch.int16).view(N, H, Bk, n_out, 2),
        }

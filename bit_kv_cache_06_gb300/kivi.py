"""ctypes binding of libkivi (include/kivi.h): same names, argument marshalling
only.  Every step of the quantise / append / decode path runs in the CUDA
kernels behind the C ABI; there is no CPU fallback -- if the library is
missing, every call raises.

PyTorch is used for device memory and streams only.
"""
import ctypes
import math
import os
from dataclasses import dataclass

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libkivi.so")

KIVI_OK = 0
KIVI_ERR_INVALID_ARG = -1
KIVI_ERR_UNSUPPORTED = -2
KIVI_ERR_CAPACITY = -3
KIVI_ERR_WORKSPACE = -4
KIVI_ERR_CUDA = -5
KIVI_ERR_EMPTY = -6

KIVI_LAYOUT_BHTD = 0
KIVI_LAYOUT_BTHD = 1

KIVI_META_FP32 = 0
KIVI_META_FP16 = 1
KIVI_FLUSH_WINDOW = 0
KIVI_FLUSH_GROUP = 1
KIVI_FP8_NONE = 0
KIVI_FP8_E4M3 = 1
KIVI_FP8_E5M2 = 2
KIVI_STATUS_WAIT_TIMEOUT = 1

BUFFER_NAMES = ("history", "k_fp16", "v_fp16")
BUFFER_DTYPES = (torch.uint8, torch.float16, torch.float16)

EXPORTED = (
    "kivi_params_validate", "kivi_cache_buffer_bytes", "kivi_history_record_bytes",
    "kivi_cache_init", "kivi_cache_reset",
    "kivi_quantize_prefill", "kivi_append_token", "kivi_decode_max_splits",
    "kivi_decode_workspace_bytes", "kivi_decode_num_splits", "kivi_decode_attention",
    "kivi_decode_partial", "kivi_decode_combine", "kivi_kv_bytes", "kivi_status_string",
    "kivi_abi_version", "kivi_sizeof_params", "kivi_sizeof_cache",
    "kivi_decode_attention_static", "kivi_decode_static_scratch_bytes",
    "kivi_decode_static_status", "kivi_test_decode_wait_timeout",
)


class KiviError(RuntimeError):
    def __init__(self, status, what=""):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} ({status})")


class kivi_params(ctypes.Structure):
    _fields_ = [("bits", ctypes.c_int32), ("group", ctypes.c_int32),
                ("residual", ctypes.c_int32), ("batch", ctypes.c_int32),
                ("num_q_heads", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("sink_tokens", ctypes.c_int32),
                ("capacity_tokens", ctypes.c_int64), ("meta", ctypes.c_int32),
                ("flush", ctypes.c_int32), ("fp8_format", ctypes.c_int32),
                ("fp8_k_scale", ctypes.c_float), ("fp8_v_scale", ctypes.c_float),
                ("reserved", ctypes.c_int32)]


class kivi_cache(ctypes.Structure):
    _fields_ = [("p", kivi_params),
                ("history", ctypes.c_void_p), ("k_fp16", ctypes.c_void_p),
                ("v_fp16", ctypes.c_void_p),
                ("n_quant", ctypes.c_int64), ("n_resid", ctypes.c_int32),
                ("n_sink", ctypes.c_int32), ("resid_head", ctypes.c_int32),
                ("reserved", ctypes.c_int32), ("kernel_launches", ctypes.c_uint64)]


_lib = None


def load(path: str = LIB_PATH):
    """Load libkivi.so; raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"libkivi.so not found at {path}; build it with "
                           "bit_kv_cache_06_gb300.build.build() (needs nvcc)")
    L = ctypes.CDLL(path)
    P, C = ctypes.POINTER(kivi_params), ctypes.POINTER(kivi_cache)
    vp, i32, i64, sz, f32 = (ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64,
                             ctypes.c_size_t, ctypes.c_float)
    sigs = {
        "kivi_params_validate": (ctypes.c_int, [P]),
        "kivi_cache_buffer_bytes": (sz, [P, ctypes.c_int]),
        "kivi_history_record_bytes": (sz, [P]),
        "kivi_cache_init": (ctypes.c_int, [C, P] + [vp] * 3),
        "kivi_cache_reset": (ctypes.c_int, [C]),
        "kivi_quantize_prefill": (ctypes.c_int, [C, vp, vp, i64, ctypes.c_int, vp]),
        "kivi_append_token": (ctypes.c_int, [C, vp, vp, vp]),
        "kivi_decode_max_splits": (i32, [P]),
        "kivi_decode_workspace_bytes": (sz, [P]),
        "kivi_decode_num_splits": (i32, [C, i32]),
        "kivi_decode_attention": (ctypes.c_int, [C, vp, vp, f32, i32, vp, sz, vp]),
        "kivi_decode_partial": (ctypes.c_int, [C, vp, f32, i32, vp, sz, vp]),
        "kivi_decode_combine": (ctypes.c_int, [C, vp, i32, vp, sz, vp]),
        "kivi_kv_bytes": (ctypes.c_double, [i64, i64, i64, i64, i64, ctypes.c_double]),
        "kivi_status_string": (ctypes.c_char_p, [ctypes.c_int]),
        "kivi_abi_version": (ctypes.c_int, []),
        "kivi_sizeof_params": (sz, []),
        "kivi_sizeof_cache": (sz, []),
        "kivi_decode_attention_static": (ctypes.c_int, [C, vp, vp, f32, i32, vp]),
        "kivi_decode_static_scratch_bytes": (sz, []),
        "kivi_decode_static_status": (ctypes.c_int, [vp, vp]),
        "kivi_test_decode_wait_timeout": (ctypes.c_int, [C, vp, vp, vp, sz, vp]),
    }
    for name, (res, args) in sigs.items():
        fn = getattr(L, name)
        fn.restype = res
        fn.argtypes = args
    if L.kivi_sizeof_params() != ctypes.sizeof(kivi_params) or \
            L.kivi_sizeof_cache() != ctypes.sizeof(kivi_cache):
        raise RuntimeError("libkivi struct layout does not match the Python mirror")
    _lib = L
    return L


def status_string(status: int) -> str:
    return load().kivi_status_string(status).decode()


def _check(status, what):
    if status != KIVI_OK:
        raise KiviError(status, what)
    return status


def _stream_ptr(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def make_params(bits, group, residual, batch, num_q_heads, num_kv_heads, head_dim,
                capacity_tokens, sink_tokens=0, meta=KIVI_META_FP32,
                flush=KIVI_FLUSH_WINDOW, fp8_format=KIVI_FP8_NONE, fp8_k_scale=1.0,
                fp8_v_scale=1.0) -> kivi_params:
    return kivi_params(bits, group, residual, batch, num_q_heads, num_kv_heads, head_dim,
                       sink_tokens, capacity_tokens, meta, flush, fp8_format, fp8_k_scale,
                       fp8_v_scale, 0)


def params_validate(p: kivi_params) -> int:
    return load().kivi_params_validate(ctypes.byref(p))


def cache_buffer_bytes(p: kivi_params, which: int) -> int:
    return load().kivi_cache_buffer_bytes(ctypes.byref(p), which)


def history_record_bytes(p: kivi_params) -> int:
    return load().kivi_history_record_bytes(ctypes.byref(p))


def decode_workspace_bytes(p: kivi_params) -> int:
    return load().kivi_decode_workspace_bytes(ctypes.byref(p))


def decode_max_splits(p: kivi_params) -> int:
    return load().kivi_decode_max_splits(ctypes.byref(p))


def kv_bytes(L, B, T, H_kv, d, bytes_per_elem) -> float:
    return load().kivi_kv_bytes(L, B, T, H_kv, d, float(bytes_per_elem))


@dataclass
class CacheShape:
    bits: int
    group: int
    residual: int
    batch: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    capacity_tokens: int
    sink_tokens: int = 0
    meta: int = KIVI_META_FP32
    flush: int = KIVI_FLUSH_WINDOW
    fp8_format: int = KIVI_FP8_NONE
    fp8_k_scale: float = 1.0
    fp8_v_scale: float = 1.0

    def params(self) -> kivi_params:
        return make_params(self.bits, self.group, self.residual, self.batch, self.num_q_heads,
                           self.num_kv_heads, self.head_dim, self.capacity_tokens,
                           self.sink_tokens, self.meta, self.flush, self.fp8_format,
                           self.fp8_k_scale, self.fp8_v_scale)


class KiviCache:
    """One layer's KIVI cache: the three device buffers (allocated with torch)
    bound to a kivi_cache struct, plus the decode workspace."""

    def __init__(self, shape: CacheShape, device="cuda", buffers=None):
        L = load()
        self.shape = shape
        self.params = shape.params()
        st = L.kivi_params_validate(ctypes.byref(self.params))
        _check(st, "kivi_params_validate")
        self.device = torch.device(device)
        if buffers is None:
            buffers = []
            for w in range(len(BUFFER_NAMES)):
                nbytes = L.kivi_cache_buffer_bytes(ctypes.byref(self.params), w)
                elem = torch.empty((), dtype=BUFFER_DTYPES[w]).element_size()
                buffers.append(torch.empty(max(nbytes // elem, 1), dtype=BUFFER_DTYPES[w],
                                           device=self.device))
        self.buffers = buffers
        self.c = kivi_cache()
        _check(L.kivi_cache_init(ctypes.byref(self.c), ctypes.byref(self.params),
                                 *[_ptr(b) for b in buffers]), "kivi_cache_init")
        ws_bytes = L.kivi_decode_workspace_bytes(ctypes.byref(self.params))
        self.workspace = torch.zeros(ws_bytes, dtype=torch.uint8, device=self.device)

    # ---- state ------------------------------------------------------------
    @property
    def n_quant(self) -> int:
        return self.c.n_quant

    @property
    def n_resid(self) -> int:
        return self.c.n_resid

    @property
    def n_sink(self) -> int:
        return self.c.n_sink

    @property
    def resid_head(self) -> int:
        return self.c.resid_head

    @property
    def kernel_launches(self) -> int:
        return self.c.kernel_launches

    def reset(self):
        _check(load().kivi_cache_reset(ctypes.byref(self.c)), "kivi_cache_reset")

    def view(self, name: str) -> torch.Tensor:
        """Typed, shaped view of a cache buffer (see include/kivi.h): history
        as uint8 [P][cap / G][record bytes], k_fp16 / v_fp16 as fp16
        [P][N_s + R][d] (sink rows first, then the residual slots)."""
        s = self.shape
        P, cap, d, G, R = s.batch * s.num_kv_heads, s.capacity_tokens, s.head_dim, s.group, \
            s.residual
        w = BUFFER_NAMES.index(name)
        rec = history_record_bytes(self.params)
        rows = s.sink_tokens + R
        shapes = [(P, cap // G, rec), (P, rows, d), (P, rows, d)]
        n = 1
        for x in shapes[w]:
            n *= x
        return self.buffers[w][:n].view(shapes[w])

    # ---- the hot path -----------------------------------------------------
    def quantize_prefill(self, k: torch.Tensor, v: torch.Tensor, layout=KIVI_LAYOUT_BHTD,
                         stream=None):
        """k, v fp16 [B, Hkv, T, d] (BHTD) or [B, T, Hkv, d] (BTHD), contiguous."""
        assert k.dtype == torch.float16 and v.dtype == torch.float16
        assert k.is_contiguous() and v.is_contiguous() and k.shape == v.shape
        T = k.shape[2] if layout == KIVI_LAYOUT_BHTD else k.shape[1]
        st = load().kivi_quantize_prefill(ctypes.byref(self.c), _ptr(k), _ptr(v), T, layout,
                                          _stream_ptr(stream))
        return _check(st, "kivi_quantize_prefill")

    def append_token(self, k_new: torch.Tensor, v_new: torch.Tensor, stream=None):
        """k_new, v_new fp16 [B, Hkv, d], contiguous."""
        assert k_new.is_contiguous() and v_new.is_contiguous()
        st = load().kivi_append_token(ctypes.byref(self.c), _ptr(k_new), _ptr(v_new),
                                      _stream_ptr(stream))
        return _check(st, "kivi_append_token")

    def num_splits(self, requested: int = 0) -> int:
        s = load().kivi_decode_num_splits(ctypes.byref(self.c), requested)
        if s < 0:
            raise KiviError(s, "kivi_decode_num_splits")
        return s

    def decode_attention(self, q: torch.Tensor, out: torch.Tensor = None, softmax_scale=0.0,
                         num_splits: int = 0, stream=None) -> torch.Tensor:
        """q fp16 [B, Hq, d] -> out fp16 [B, Hq, d]."""
        assert q.dtype == torch.float16 and q.is_contiguous()
        if out is None:
            out = torch.empty_like(q)
        st = load().kivi_decode_attention(
            ctypes.byref(self.c), _ptr(q), _ptr(out), float(softmax_scale), int(num_splits),
            _ptr(self.workspace), self.workspace.numel(), _stream_ptr(stream))
        _check(st, "kivi_decode_attention")
        return out

    def decode_partial(self, q, softmax_scale=0.0, num_splits=0, stream=None):
        st = load().kivi_decode_partial(ctypes.byref(self.c), _ptr(q), float(softmax_scale),
                                        int(num_splits), _ptr(self.workspace),
                                        self.workspace.numel(), _stream_ptr(stream))
        return _check(st, "kivi_decode_partial")

    def decode_combine(self, out, num_splits, stream=None):
        st = load().kivi_decode_combine(ctypes.byref(self.c), _ptr(out), int(num_splits),
                                        _ptr(self.workspace), self.workspace.numel(),
                                        _stream_ptr(stream))
        return _check(st, "kivi_decode_combine")

    def workspace_status(self) -> int:
        """Error bits the kernels set in the workspace header (0 = none)."""
        return int(self.workspace[:4].view(torch.int32).item())


def default_softmax_scale(d: int) -> float:
    return 1.0 / math.sqrt(d)

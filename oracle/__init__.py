"""CPU oracle for KIVI-style asymmetric low-bit KV-cache quantisation.

TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the benchmark's
CPU-baseline leg may import this package; the product path
(``bit_kv_cache_06_gb300``) never does, and the two share no code.

Thin numpy/ctypes wrapper over ``kivi_oracle.c`` (plain fp32 quantiser, fp64
attention).  Sources, by page title and section:

* "KV Cache INT4 Quantization for 1M+ Token Context Windows", section 2 --
  the quantiser q = clamp(round(x/S) + Z, 0, 2^b - 1), the 1e-8 scale floor,
  zero = round(-min/scale).
* "4.4 KV Cache quantization", section 1 (byte formula), section 2 (softmax
  attention), sections 3.1-3.2 (grouping directions, residual cache).
* "KIVI: A Tuning-Free Asymmetric 2bit Quantization for KV Cache",
  "The streaming complication" (residual window, groups frozen once full).
"""
import ctypes
import math

import numpy as np

from . import build as _build

_lib = None

_u16p = ctypes.POINTER(ctypes.c_uint16)
_u8p = ctypes.POINTER(ctypes.c_uint8)
_f32p = ctypes.POINTER(ctypes.c_float)
_f64p = ctypes.POINTER(ctypes.c_double)
_i64p = ctypes.POINTER(ctypes.c_int64)


class _Cache(ctypes.Structure):
    _fields_ = [
        ("bits", ctypes.c_int32), ("G", ctypes.c_int32), ("R", ctypes.c_int32),
        ("d", ctypes.c_int32), ("P", ctypes.c_int64), ("cap", ctypes.c_int64),
        ("n_quant", ctypes.c_int64), ("n_resid", ctypes.c_int64),
        ("kc", _u8p), ("vc", _u8p),
        ("ks", _f32p), ("kz", _f32p), ("vs", _f32p), ("vz", _f32p),
        ("kr", _u16p), ("vr", _u16p),
        ("Ns", ctypes.c_int64), ("n_sink", ctypes.c_int64), ("meta", ctypes.c_int64),
        ("flush", ctypes.c_int64), ("fp8", ctypes.c_int64),
        ("fp8_k_scale", ctypes.c_float), ("fp8_v_scale", ctypes.c_float),
    ]


def lib():
    """Load (building first if needed) the oracle shared library."""
    global _lib
    if _lib is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        L.orc_kv_bytes.restype = ctypes.c_double
        L.orc_kv_bytes.argtypes = [ctypes.c_int64] * 5 + [ctypes.c_double]
        L.orc_half_to_double.restype = ctypes.c_double
        L.orc_half_to_double.argtypes = [ctypes.c_uint16]
        L.orc_quant_params.restype = None
        L.orc_quant_params.argtypes = [ctypes.c_float, ctypes.c_float, ctypes.c_int,
                                       _f32p, _f32p]
        L.orc_encode.restype = ctypes.c_int
        L.orc_encode.argtypes = [ctypes.c_float, ctypes.c_float, ctypes.c_float, ctypes.c_int]
        L.orc_quantize_k_group.restype = None
        L.orc_quantize_k_group.argtypes = [_f32p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                           _f32p, _f32p, _u8p]
        L.orc_quantize_v_token.restype = None
        L.orc_quantize_v_token.argtypes = [_f32p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                           _f32p, _f32p, _u8p]
        L.orc_pack_row.restype = None
        L.orc_pack_row.argtypes = [_u8p, ctypes.c_int, ctypes.c_int, _u8p]
        L.orc_unpack_row.restype = None
        L.orc_unpack_row.argtypes = [_u8p, ctypes.c_int, ctypes.c_int, _u8p]
        L.orc_prefill.restype = ctypes.c_int
        L.orc_prefill.argtypes = [ctypes.POINTER(_Cache), _u16p, _u16p, ctypes.c_int64,
                                  ctypes.c_int]
        L.orc_append.restype = ctypes.c_int
        L.orc_append.argtypes = [ctypes.POINTER(_Cache), _u16p, _u16p]
        L.orc_dequant_k.restype = None
        L.orc_dequant_k.argtypes = [ctypes.POINTER(_Cache), ctypes.c_int64, _f64p]
        L.orc_dequant_v.restype = None
        L.orc_dequant_v.argtypes = [ctypes.POINTER(_Cache), ctypes.c_int64, _f64p]
        L.orc_attention.restype = ctypes.c_int
        L.orc_attention.argtypes = [ctypes.POINTER(_Cache), ctypes.c_int, _u16p,
                                    ctypes.c_double, _i64p, ctypes.c_int64, _f64p,
                                    ctypes.c_int]
        L.orc_attention_partial.restype = None
        L.orc_attention_partial.argtypes = [ctypes.POINTER(_Cache), ctypes.c_int, _u16p,
                                            ctypes.c_double, ctypes.c_int64, ctypes.c_int64,
                                            ctypes.c_int64, _f64p, _f64p, _f64p]
        L.orc_value_position.restype = ctypes.c_int
        L.orc_value_position.argtypes = [ctypes.c_int] * 4
        L.orc_record_bytes.restype = ctypes.c_int64
        L.orc_record_bytes.argtypes = [ctypes.c_int] * 4
        L.orc_fp8_round.restype = ctypes.c_double
        L.orc_fp8_round.argtypes = [ctypes.c_double, ctypes.c_int]
        L.orc_fp8_bits.restype = ctypes.c_uint8
        L.orc_fp8_bits.argtypes = [ctypes.c_double, ctypes.c_int]
        L.orc_fp8_value.restype = ctypes.c_double
        L.orc_fp8_value.argtypes = [ctypes.c_uint8, ctypes.c_int]
        L.orc_quant_params_f16.restype = None
        L.orc_quant_params_f16.argtypes = [ctypes.c_float, ctypes.c_float, ctypes.c_int,
                                           _f32p, _f32p]
        L.orc_export_history.restype = None
        L.orc_export_history.argtypes = [ctypes.POINTER(_Cache), ctypes.c_int64, _u8p]
        _lib = L
    return _lib


def value_position(c, d, G, bits) -> int:
    """Stored position of value channel c (see kivi_oracle.h)."""
    return lib().orc_value_position(c, d, G, bits)


META_FP32, META_FP16 = 0, 1
FLUSH_WINDOW, FLUSH_GROUP = 0, 1
FP8_E4M3, FP8_E5M2 = 1, 2


def record_bytes(d, G, bits, meta=META_FP32) -> int:
    return lib().orc_record_bytes(d, G, bits, meta)


def fp8_round(x, fmt) -> float:
    return lib().orc_fp8_round(float(x), fmt)


def fp8_bits(v, fmt) -> int:
    return lib().orc_fp8_bits(float(v), fmt)


def fp8_value(b, fmt) -> float:
    return lib().orc_fp8_value(int(b), fmt)


def quant_params_f16(mn, mx, bits):
    """(scale, zero) of one group with fp16 storage (range-guarded form)."""
    s, z = ctypes.c_float(), ctypes.c_float()
    lib().orc_quant_params_f16(float(np.float32(mn)), float(np.float32(mx)), bits,
                               ctypes.byref(s), ctypes.byref(z))
    return np.float32(s.value), np.float32(z.value)


def _ptr(a, t):
    return a.ctypes.data_as(t)


def _as_u16(x):
    """fp16 array (numpy float16 or uint16 bit patterns) -> contiguous uint16."""
    x = np.ascontiguousarray(x)
    if x.dtype == np.float16:
        return x.view(np.uint16)
    if x.dtype != np.uint16:
        raise TypeError(f"expected float16 data, got {x.dtype}")
    return x


# ---------------------------------------------------------------- scalars ---

def kv_bytes(L, B, T, H_kv, d, bytes_per_elem):
    """M_KV = 2 L B T H_kv d b ("4.4 KV Cache quantization", section 1)."""
    return lib().orc_kv_bytes(L, B, T, H_kv, d, float(bytes_per_elem))


def half_to_double(bits: int) -> float:
    return lib().orc_half_to_double(int(bits) & 0xFFFF)


def quant_params(mn, mx, bits):
    """(scale, zero) of one group in fp32 (returned as numpy float32)."""
    s, z = ctypes.c_float(), ctypes.c_float()
    lib().orc_quant_params(float(np.float32(mn)), float(np.float32(mx)), bits,
                           ctypes.byref(s), ctypes.byref(z))
    return np.float32(s.value), np.float32(z.value)


def encode(x, s, z, bits) -> int:
    return lib().orc_encode(float(np.float32(x)), float(np.float32(s)),
                            float(np.float32(z)), bits)


# ----------------------------------------------------------------- blocks ---

def quantize_k_group(x, bits):
    """Per-channel key quantisation of one [G][d] token block (fp32 input)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    G, d = x.shape
    s = np.empty(d, np.float32)
    z = np.empty(d, np.float32)
    codes = np.empty((G, d), np.uint8)
    lib().orc_quantize_k_group(_ptr(x, _f32p), G, d, bits, _ptr(s, _f32p),
                               _ptr(z, _f32p), _ptr(codes, _u8p))
    return s, z, codes


def quantize_v_token(x, G, bits):
    """Per-token value quantisation of one token row [d] in groups of G channels."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    d = x.shape[0]
    s = np.empty(d // G, np.float32)
    z = np.empty(d // G, np.float32)
    codes = np.empty(d, np.uint8)
    lib().orc_quantize_v_token(_ptr(x, _f32p), G, d, bits, _ptr(s, _f32p),
                               _ptr(z, _f32p), _ptr(codes, _u8p))
    return s, z, codes


def pack_row(codes, bits):
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    d = codes.shape[0]
    out = np.empty(d * bits // 8, np.uint8)
    lib().orc_pack_row(_ptr(codes, _u8p), d, bits, _ptr(out, _u8p))
    return out


def unpack_row(packed, d, bits):
    packed = np.ascontiguousarray(packed, dtype=np.uint8)
    out = np.empty(d, np.uint8)
    lib().orc_unpack_row(_ptr(packed, _u8p), d, bits, _ptr(out, _u8p))
    return out


def unpack_codes(packed, d, bits):
    """Unpack a [..., d*bits/8] packed array into [..., d] codes."""
    packed = np.asarray(packed, dtype=np.uint8)
    flat = packed.reshape(-1, packed.shape[-1])
    out = np.empty((flat.shape[0], d), np.uint8)
    for i in range(flat.shape[0]):
        out[i] = unpack_row(flat[i], d, bits)
    return out.reshape(*packed.shape[:-1], d)


# ------------------------------------------------------------------ cache ---

class OracleCache:
    """P = batch * kv_heads independent (batch, kv-head) pairs; same buffer
    layout as the CUDA library (see kivi_oracle.h)."""

    def __init__(self, P, d, bits, G, R, cap, Ns=0, meta=META_FP32, flush=FLUSH_WINDOW,
                 fp8=0, fp8_k_scale=1.0, fp8_v_scale=1.0):
        if bits not in (2, 4, 8) or (bits == 8) != (fp8 != 0) or d % G or R % G or cap % G \
                or Ns < 0 or (flush == FLUSH_WINDOW and cap % R):
            raise ValueError("need bits in {2,4} (or 8 with an fp8 format), G | d, G | R, "
                             "G | cap (R | cap for the window flush), Ns >= 0")
        self.P, self.d, self.bits, self.G, self.R, self.cap = P, d, bits, G, R, cap
        self.Ns = Ns
        self.meta = meta
        self.flush = flush
        self.fp8 = fp8
        rb = d * bits // 8
        self.kc = np.zeros((P, cap, rb), np.uint8)
        self.vc = np.zeros((P, cap, rb), np.uint8)
        self.ks = np.zeros((P, cap // G, d), np.float32)
        self.kz = np.zeros((P, cap // G, d), np.float32)
        self.vs = np.zeros((P, cap, d // G), np.float32)
        self.vz = np.zeros((P, cap, d // G), np.float32)
        # fp16 rows: Ns sink rows, then the R residual slots
        self.kr = np.zeros((P, Ns + R, d), np.uint16)
        self.vr = np.zeros((P, Ns + R, d), np.uint16)
        self._c = _Cache(bits, G, R, d, P, cap, 0, 0,
                         _ptr(self.kc, _u8p), _ptr(self.vc, _u8p),
                         _ptr(self.ks, _f32p), _ptr(self.kz, _f32p),
                         _ptr(self.vs, _f32p), _ptr(self.vz, _f32p),
                         _ptr(self.kr, _u16p), _ptr(self.vr, _u16p), Ns, 0, meta, flush,
                         fp8, fp8_k_scale, fp8_v_scale)

    @property
    def n_quant(self):
        return self._c.n_quant

    @property
    def n_resid(self):
        return self._c.n_resid

    @property
    def n_sink(self):
        return self._c.n_sink

    @property
    def n_tokens(self):
        return self.n_sink + self.n_quant + self.n_resid

    @property
    def kres(self):
        """Residual slots only: [P][R][d] (the sink rows come first in kr)."""
        return self.kr[:, self.Ns:]

    @property
    def vres(self):
        return self.vr[:, self.Ns:]

    def prefill(self, k, v, nthreads=1):
        """Append T tokens: k, v fp16 [P][T][d].  Returns the status code."""
        k = _as_u16(k)
        v = _as_u16(v)
        assert k.shape == v.shape and k.shape[0] == self.P and k.shape[2] == self.d
        return lib().orc_prefill(ctypes.byref(self._c), _ptr(k, _u16p), _ptr(v, _u16p),
                                 k.shape[1], nthreads)

    def append(self, k, v):
        """One decode-step token: k, v fp16 [P][d]."""
        k = _as_u16(k)
        v = _as_u16(v)
        assert k.shape == (self.P, self.d) and v.shape == (self.P, self.d)
        return lib().orc_append(ctypes.byref(self._c), _ptr(k, _u16p), _ptr(v, _u16p))

    def export_history(self, p):
        """The filled key-group records of pair p in the CUDA library's packed
        history layout: uint8 [n_quant / G][record_bytes]."""
        rec = record_bytes(self.d, self.G, self.bits, self.meta)
        out = np.zeros((self.n_quant // self.G, rec), np.uint8)
        lib().orc_export_history(ctypes.byref(self._c), p, _ptr(out, _u8p))
        return out

    def dequant_k(self, p):
        out = np.empty((self.n_tokens, self.d), np.float64)
        lib().orc_dequant_k(ctypes.byref(self._c), p, _ptr(out, _f64p))
        return out

    def dequant_v(self, p):
        out = np.empty((self.n_tokens, self.d), np.float64)
        lib().orc_dequant_v(ctypes.byref(self._c), p, _ptr(out, _f64p))
        return out

    def attention(self, q, g, tau=None, rows=None, nthreads=1):
        """fp64 attention; q fp16 [P*g][d] (any shape with that many rows)."""
        q = _as_u16(q).reshape(-1, self.d)
        assert q.shape[0] == self.P * g
        if tau is None:
            tau = 1.0 / math.sqrt(self.d)
        if rows is None:
            out = np.empty((self.P * g, self.d), np.float64)
            rp, nr = None, 0
        else:
            rows = np.ascontiguousarray(rows, dtype=np.int64)
            out = np.empty((rows.shape[0], self.d), np.float64)
            rp, nr = _ptr(rows, _i64p), rows.shape[0]
        st = lib().orc_attention(ctypes.byref(self._c), g, _ptr(q, _u16p), float(tau),
                                 rp, nr, _ptr(out, _f64p), nthreads)
        if st != 0:
            raise RuntimeError(f"oracle attention status {st}")
        return out

    def attention_partial(self, q, g, row, t0, t1, tau=None):
        q = _as_u16(q).reshape(-1, self.d)
        if tau is None:
            tau = 1.0 / math.sqrt(self.d)
        m, l = ctypes.c_double(), ctypes.c_double()
        o = np.empty(self.d, np.float64)
        lib().orc_attention_partial(ctypes.byref(self._c), g, _ptr(q, _u16p), float(tau),
                                    row, t0, t1, ctypes.byref(m), ctypes.byref(l),
                                    _ptr(o, _f64p))
        return m.value, l.value, o

"""Host-side checks of the C ABI (no GPU, no CUDA compute call).

The library must load, export every function include/kivi.h declares, agree
with the Python struct mirrors, and reject bad arguments before it launches
anything.  Only calls that return before any CUDA call are made here.
"""
import ctypes
import os
import re
import subprocess

import pytest

from bit_kv_cache_06_gb300 import build as kbuild
from bit_kv_cache_06_gb300 import kivi

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "kivi.h")


@pytest.fixture(scope="module")
def L():
    kbuild.build()
    return kivi.load()


def _declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"\b(kivi_[a-z_0-9]+)\s*\(", src)
    return sorted(set(names))


def test_every_declared_function_is_exported(L):
    names = _declared_functions()
    assert len(names) >= 15
    out = subprocess.run(["nm", "-D", "--defined-only", kivi.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\bT (kivi_\w+)", out))
    missing = [n for n in names if n not in exported]
    assert not missing, missing
    for n in names:
        assert hasattr(L, n)
    assert set(kivi.EXPORTED) == set(names)


def test_struct_layout_matches_mirror(L):
    assert L.kivi_abi_version() == 2
    assert L.kivi_sizeof_params() == ctypes.sizeof(kivi.kivi_params) == 64
    assert L.kivi_sizeof_cache() == ctypes.sizeof(kivi.kivi_cache) == 120


def test_status_strings(L):
    for st in range(-6, 1):
        assert kivi.status_string(st) not in ("", "unknown status")
    assert kivi.status_string(-99) == "unknown status"


def _p(**kw):
    base = dict(bits=2, group=32, residual=128, batch=8, num_q_heads=32, num_kv_heads=8,
                head_dim=128, capacity_tokens=32768)
    base.update(kw)
    return kivi.make_params(**base)


@pytest.mark.parametrize("kw,status", [
    ({}, 0),
    ({"bits": 4, "group": 64}, 0),
    ({"bits": 3}, -2), ({"bits": 16}, -2),
    ({"head_dim": 64}, -2), ({"group": 48}, -2), ({"group": 8}, -2),
    ({"residual": 48, "capacity_tokens": 4800}, -2),  # R not a multiple of G
    ({"num_q_heads": 33}, -1),                   # Hq % Hkv
    ({"num_q_heads": 128, "num_kv_heads": 8}, -2),  # query group 16 > 8
    ({"capacity_tokens": 1000}, -1),             # not a multiple of R
    ({"batch": 0}, -1), ({"residual": 0}, -1), ({"capacity_tokens": -128}, -1),
    ({"batch": 10000}, -2),                      # > 65535 pairs
    ({"sink_tokens": 4}, 0), ({"sink_tokens": 256}, 0),
    ({"sink_tokens": 257}, -2), ({"sink_tokens": -1}, -1),
    ({"meta": 7}, -2), ({"meta": 1}, 0),
    ({"flush": 1}, 0), ({"flush": 2}, -2),
    ({"bits": 8, "fp8_format": 1}, 0), ({"bits": 8, "fp8_format": 2, "fp8_v_scale": 0.5}, 0),
    ({"bits": 8}, -1),                           # FP8 needs a format
    ({"bits": 8, "fp8_format": 1, "fp8_k_scale": 0.0}, -1),
    ({"bits": 8, "fp8_format": 1, "group": 64}, -2),
    ({"bits": 2, "fp8_format": 1}, -1),
])
def test_params_validate(L, kw, status):
    assert kivi.params_validate(_p(**kw)) == status


def test_cache_state_fields_are_checked(L):
    """The reserved word must stay 0; the ring head must be a slot, and 0
    with the whole-window flush."""
    k = ctypes.c_void_p(0x900000)
    s = ctypes.c_void_p(0)
    _, c = _fake_cache(L, _p())
    c.reserved = 1
    assert L.kivi_quantize_prefill(ctypes.byref(c), k, k, 1, 0, s) == -1
    _, c = _fake_cache(L, _p(), n_quant=128, n_resid=5)
    c.resid_head = 3                                    # whole-window flush: head is 0
    assert L.kivi_quantize_prefill(ctypes.byref(c), k, k, 1, 0, s) == -1
    _, c = _fake_cache(L, _p(flush=1), n_quant=96, n_resid=100)
    c.resid_head = 128                                  # not a slot of R = 128
    assert L.kivi_quantize_prefill(ctypes.byref(c), k, k, 1, 0, s) == -1
    c.resid_head = 96
    c.n_quant = 100                                     # not a multiple of G
    assert L.kivi_quantize_prefill(ctypes.byref(c), k, k, 1, 0, s) == -1
    assert c.kernel_launches == 0


def test_buffer_and_workspace_sizes(L):
    p = _p()
    P, cap = 64, 32768
    # one 4 KiB record per 32 tokens (128 B per token: codes 2 x 32 B, key
    # scale/zero 2 x 128 x 4 B per 32 tokens, value scale/zero 2 x 4 x 4 B)
    assert kivi.history_record_bytes(p) == 4096
    assert kivi.history_record_bytes(_p(bits=4, group=64)) == 64 * 160
    assert [kivi.cache_buffer_bytes(p, w) for w in range(3)] == [
        P * (cap // 32) * 4096, P * 128 * 128 * 2, P * 128 * 128 * 2]
    # FP8: 32-token records of key then value bytes (256 B per token)
    assert kivi.history_record_bytes(_p(bits=8, fp8_format=1)) == 32 * 256
    # sink rows come in front of the residual slots
    ps = _p(sink_tokens=16)
    assert kivi.cache_buffer_bytes(ps, 1) == P * (16 + 128) * 128 * 2
    assert kivi.cache_buffer_bytes(p, 3) == 0 and kivi.cache_buffer_bytes(p, -1) == 0
    assert kivi.cache_buffer_bytes(_p(bits=3), 0) == 0
    # 4096 (pair, split) blocks at most: 64 pairs -> 64 splits
    assert kivi.decode_max_splits(p) == 64
    # header + 64 pair counters (rounded to 256 B) + 65 partials per query row
    assert kivi.decode_workspace_bytes(p) == 256 + 256 + 8 * 32 * (64 + 1) * 130 * 4
    # never more splits than 128-token chunks of capacity
    assert kivi.decode_max_splits(_p(batch=1, num_kv_heads=1, num_q_heads=4,
                                     residual=32, capacity_tokens=256)) == 2


def test_kv_bytes_formula_in_library(L):
    assert kivi.kv_bytes(32, 1, 32768, 8, 128, 2) == 4 * 2 ** 30
    assert kivi.kv_bytes(80, 1, 1048576, 8, 128, 2) == 343597383680


def _fake_cache(L, p, n_quant=0, n_resid=0, align=0):
    c = kivi.kivi_cache()
    ptrs = [ctypes.c_void_p(0x100000 * (i + 1) + align) for i in range(3)]
    st = L.kivi_cache_init(ctypes.byref(c), ctypes.byref(p), *ptrs)
    if st == 0:
        c.n_quant, c.n_resid = n_quant, n_resid
    return st, c


def test_cache_init_validation(L):
    p = _p()
    st, c = _fake_cache(L, p)
    assert st == 0 and c.n_quant == 0 and c.n_resid == 0
    assert _fake_cache(L, p, align=8)[0] == -1           # misaligned buffer
    c2 = kivi.kivi_cache()
    assert L.kivi_cache_init(ctypes.byref(c2), ctypes.byref(p), *([None] * 3)) == -1
    assert L.kivi_cache_init(None, ctypes.byref(p), *([ctypes.c_void_p(16)] * 3)) == -1
    assert _fake_cache(L, _p(bits=3))[0] == -2


def test_prefill_rejects_before_launch(L):
    p = _p(capacity_tokens=256)
    _, c = _fake_cache(L, p)
    k = ctypes.c_void_p(0x900000)
    s = ctypes.c_void_p(0)
    assert L.kivi_quantize_prefill(ctypes.byref(c), k, k, 0, 0, s) == 0      # no-op
    assert L.kivi_quantize_prefill(ctypes.byref(c), k, k, -1, 0, s) == -1
    assert L.kivi_quantize_prefill(ctypes.byref(c), k, k, 10, 2, s) == -1    # bad layout
    assert L.kivi_quantize_prefill(ctypes.byref(c), None, k, 10, 0, s) == -1
    assert L.kivi_quantize_prefill(ctypes.byref(c), ctypes.c_void_p(0x900008), k, 10, 0, s) == -1
    # 385 tokens: 384 would be quantised (> capacity 256) -> capacity, state unchanged
    assert L.kivi_quantize_prefill(ctypes.byref(c), k, k, 385, 0, s) == -3
    assert (c.n_quant, c.n_resid, c.kernel_launches) == (0, 0, 0)
    # inconsistent bookkeeping is rejected
    c.n_quant, c.n_resid = 128, 0
    assert L.kivi_quantize_prefill(ctypes.byref(c), k, k, 1, 0, s) == -1
    c.n_quant, c.n_resid = 100, 5
    assert L.kivi_quantize_prefill(ctypes.byref(c), k, k, 1, 0, s) == -1
    # full cache: appending one token would flush past capacity
    c.n_quant, c.n_resid = 256, 128
    assert L.kivi_append_token(ctypes.byref(c), k, k, s) == -3
    assert (c.n_quant, c.n_resid) == (256, 128)


def test_sink_bookkeeping_rejects_before_launch(L):
    """With N_s sink tokens: tokens after the sink only once it is full; the
    capacity check counts only the tokens after the sink."""
    p = _p(capacity_tokens=256, sink_tokens=8)
    _, c = _fake_cache(L, p)
    k = ctypes.c_void_p(0x900000)
    s = ctypes.c_void_p(0)
    # 8 sink + 385 more: 384 would be quantised (> 256) -> capacity, unchanged
    assert L.kivi_quantize_prefill(ctypes.byref(c), k, k, 8 + 385, 0, s) == -3
    assert (c.n_sink, c.n_quant, c.n_resid, c.kernel_launches) == (0, 0, 0, 0)
    # a partial sink with tokens after it is an inconsistent state
    c.n_sink, c.n_quant, c.n_resid = 3, 0, 1
    assert L.kivi_quantize_prefill(ctypes.byref(c), k, k, 1, 0, s) == -1
    c.n_sink, c.n_quant, c.n_resid = 9, 0, 0                # more than N_s
    assert L.kivi_quantize_prefill(ctypes.byref(c), k, k, 1, 0, s) == -1
    # a sink-only cache is not empty
    c.n_sink, c.n_quant, c.n_resid = 5, 0, 0
    q = ctypes.c_void_p(0x900000)
    assert L.kivi_decode_attention(ctypes.byref(c), q, q, 0.0, 0, ctypes.c_void_p(0xA00000),
                                   0, s) == -4          # not -6: it holds tokens


def test_decode_rejects_before_launch(L):
    p = _p(capacity_tokens=1024)
    ws_need = kivi.decode_workspace_bytes(p)
    _, c = _fake_cache(L, p)
    q = ctypes.c_void_p(0x900000)
    ws = ctypes.c_void_p(0xA00000)
    s = ctypes.c_void_p(0)
    # empty cache
    assert L.kivi_decode_attention(ctypes.byref(c), q, q, 0.0, 0, ws, ws_need, s) == -6
    c.n_quant, c.n_resid = 512, 7
    # workspace too small / misaligned / null
    assert L.kivi_decode_attention(ctypes.byref(c), q, q, 0.0, 1, ws, ws_need - 1, s) == -4
    assert L.kivi_decode_attention(ctypes.byref(c), q, q, 0.0, 1, ctypes.c_void_p(0xA00004),
                                   ws_need, s) == -1
    assert L.kivi_decode_attention(ctypes.byref(c), q, q, 0.0, 1, None, ws_need, s) == -1
    # misaligned q / out
    assert L.kivi_decode_attention(ctypes.byref(c), ctypes.c_void_p(0x900002), q, 0.0, 1, ws,
                                   ws_need, s) == -1
    assert L.kivi_decode_attention(ctypes.byref(c), q, None, 0.0, 1, ws, ws_need, s) == -1
    assert L.kivi_decode_num_splits(ctypes.byref(c), -1) == -1
    # explicit split counts are clamped to one per 128 quantised tokens (512 -> 4)
    assert L.kivi_decode_num_splits(ctypes.byref(c), 3) == 3
    assert L.kivi_decode_num_splits(ctypes.byref(c), 8) == 4
    assert L.kivi_decode_num_splits(ctypes.byref(c), 1000) == 4
    # more splits than the workspace was sized for: 64 pairs -> at most 64
    p2 = _p()
    _, c2 = _fake_cache(L, p2, n_quant=32640, n_resid=128)
    ws2 = kivi.decode_workspace_bytes(p2)
    assert kivi.decode_max_splits(p2) == 64
    assert L.kivi_decode_num_splits(ctypes.byref(c2), 64) == 64
    assert L.kivi_decode_num_splits(ctypes.byref(c2), 65) == -4
    assert L.kivi_decode_attention(ctypes.byref(c2), q, q, 0.0, 65, ws, ws2, s) == -4
    assert c.kernel_launches == 0 and c2.kernel_launches == 0


def test_product_package_does_not_import_oracle():
    pkg = os.path.join(ROOT, "bit_kv_cache_06_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                src = open(os.path.join(dirpath, f)).read()
                assert "oracle" not in src.lower() or f == "synth.py" and \
                    "import oracle" not in src, f


def test_missing_library_fails_loudly(tmp_path, monkeypatch):
    """No silent fallback: without libkivi.so the binding raises."""
    monkeypatch.setattr(kivi, "_lib", None)
    with pytest.raises(RuntimeError, match="libkivi.so not found"):
        kivi.load(str(tmp_path / "libkivi.so"))

"""The allocation-free decode entry point (kivi_decode_attention_static).

It exists for callers that cannot allocate device memory where they decode;
its split-K scratch is a fixed array inside the library.  These tests call it
through the C ABI and compare it with kivi_decode_attention (caller-provided
workspace) on the same cache.  The file is named so that pytest collects it
last; it must also pass alone in a fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

from _helpers import ATTN_TOL, check_pairs_in_chunks, row_rel_err
from bit_kv_cache_06_gb300 import build as kbuild
from bit_kv_cache_06_gb300 import kivi, synth

pytestmark = pytest.mark.gpu


def _call_static(L, cache, q, out, num_splits=0):
    return L.kivi_decode_attention_static(
        ctypes.byref(cache.c), ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(out.data_ptr()),
        0.0, num_splits, ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def test_static_scratch_decode_matches_workspace_decode_twice():
    assert torch.cuda.is_available()
    kbuild.build()
    L = kivi.load()
    assert L.kivi_decode_static_scratch_bytes() == 8 << 20
    w = synth.C2.with_(name="noalloc", B=2, T=4096 + 77)
    K, V = synth.make_kv(w)
    cache = kivi.KiviCache(kivi.CacheShape(w.bits, w.G, w.R, w.B, w.Hq, w.Hkv, w.d,
                                           w.capacity()))
    cache.quantize_prefill(K.cuda(), V.cuda())
    for call in range(2):                       # two calls in a row, different queries
        q = synth.make_q(w, step=call).cuda()
        ref = cache.decode_attention(q)
        out = torch.full_like(q, float("nan"))
        assert _call_static(L, cache, q, out) == kivi.KIVI_OK
        torch.cuda.synchronize()
        got = out.float().cpu().numpy().reshape(-1, w.d)
        exp = ref.float().cpu().numpy().reshape(-1, w.d)
        assert np.all(np.isfinite(got))
        assert row_rel_err(got, exp).max() <= ATTN_TOL
    # an explicit split count runs the same kernel with the same splits as
    # the workspace path: the outputs agree bit for bit
    S = cache.num_splits(3)
    out = torch.empty_like(q)
    assert _call_static(L, cache, q, out, num_splits=S) == kivi.KIVI_OK
    ref = cache.decode_attention(q, num_splits=S)
    torch.cuda.synchronize()
    assert torch.equal(out, ref)
    # no bounded wait gave up: the status word of the fixed scratch is 0
    status = ctypes.c_uint32(0xFFFFFFFF)
    assert L.kivi_decode_static_status(ctypes.byref(status), ctypes.c_void_p(
        torch.cuda.current_stream().cuda_stream)) == kivi.KIVI_OK
    torch.cuda.synchronize()
    assert status.value == 0


def test_static_scratch_rejects_explicit_splits_that_do_not_fit():
    """700 pairs with query group 8: one split per pair fits the 8 MiB array
    (5600 rows x 2 partials x 520 B), two do not (x 3 = 8.7 MB), although the
    workspace path would allow 6.  The explicit request is refused before
    anything is launched; the automatic count is clamped to what fits."""
    kbuild.build()
    L = kivi.load()
    p = kivi.make_params(2, 32, 32, 700, 8, 1, 128, 4096)
    assert L.kivi_decode_max_splits(ctypes.byref(p)) == 6
    c = kivi.kivi_cache()
    ptrs = [ctypes.c_void_p(0x100000 * (i + 1)) for i in range(3)]
    assert L.kivi_cache_init(ctypes.byref(c), ctypes.byref(p), *ptrs) == 0
    c.n_quant, c.n_resid = 4096, 1
    q = ctypes.c_void_p(0x900000)
    assert L.kivi_decode_attention_static(ctypes.byref(c), q, q, 0.0, 2, None) == \
        kivi.KIVI_ERR_WORKSPACE
    assert c.kernel_launches == 0


def test_static_scratch_rejects_oversized_problems_before_launch():
    kbuild.build()
    L = kivi.load()
    # 16384 pairs x 4 query heads: one split per pair needs 65536 * 130 * 4 B > 8 MiB
    p = kivi.make_params(2, 32, 32, 2048, 32, 8, 128, 0)
    c = kivi.kivi_cache()
    ptrs = [ctypes.c_void_p(0x100000 * (i + 1)) for i in range(3)]
    assert L.kivi_cache_init(ctypes.byref(c), ctypes.byref(p), *ptrs) == 0
    c.n_resid = 1
    q = ctypes.c_void_p(0x900000)
    assert L.kivi_decode_attention_static(ctypes.byref(c), q, q, 0.0, 1, None) == \
        kivi.KIVI_ERR_WORKSPACE
    assert c.kernel_launches == 0


def _static_fit(p):
    """Splits the fixed array holds for these parameters (0: not even one)."""
    rows = p.batch * p.num_q_heads
    fixed = 256 + ((p.batch * p.num_kv_heads * 4 + 255) // 256) * 256
    per_split = rows * (p.head_dim + 2) * 4
    return max(0, ((8 << 20) - fixed) // per_split - 1)


def test_static_scratch_lowers_the_automatic_split_count_to_what_fits():
    """512 pairs with query group 8, just above the 456 resident blocks: the
    cost model prefers several splits to a nearly empty second wave, more
    than the 8 MiB array holds.  The allocation-free entry point lowers the
    automatic count to one that fits: KIVI_OK, an output equal bit for bit to
    the workspace path's at that count, and sampled pairs within 2e-3 of the
    oracle."""
    kbuild.build()
    L = kivi.load()
    w = synth.C2.with_(name="noalloc-lower", B=64, Hq=64, Hkv=8, T=32768 + 1, bits=4, G=32)
    cache = kivi.KiviCache(kivi.CacheShape(w.bits, w.G, w.R, w.B, w.Hq, w.Hkv, w.d,
                                           w.capacity()))
    fit = _static_fit(cache.params)
    K, V = synth.make_kv(w, device="cuda")
    cache.quantize_prefill(K, V)
    auto = cache.num_splits(0)
    assert 1 <= fit < auto, (fit, auto)            # the lowering rule is exercised
    q = synth.make_q(w).cuda()
    out = torch.empty_like(q)
    assert _call_static(L, cache, q, out) == kivi.KIVI_OK
    torch.cuda.synchronize()
    assert any(torch.equal(out, cache.decode_attention(q, num_splits=S))
               for S in range(1, fit + 1))
    check_pairs_in_chunks(cache, w, K, V, q, out, [0, 255, 511])


def test_static_automatic_decode_equals_workspace_automatic_decode():
    """Same automatic split count on both paths: bit-identical outputs."""
    kbuild.build()
    L = kivi.load()
    w = synth.C2.with_(name="noalloc-auto", B=4, T=8192 + 5)
    K, V = synth.make_kv(w)
    cache = kivi.KiviCache(kivi.CacheShape(w.bits, w.G, w.R, w.B, w.Hq, w.Hkv, w.d,
                                           w.capacity()))
    cache.quantize_prefill(K.cuda(), V.cuda())
    q = synth.make_q(w).cuda()
    ref = cache.decode_attention(q)
    out = torch.empty_like(q)
    assert _call_static(L, cache, q, out) == kivi.KIVI_OK
    torch.cuda.synchronize()
    assert torch.equal(out, ref)

"""GPU parity: the CUDA path through the C ABI against the CPU oracle.

Codes, scales, zero points, residual bytes and the bookkeeping must match bit
for bit; attention rows within 2e-3 max relative error (fp32 accumulation
against the fp64 oracle).  Sizes span several 128-token tiles and a ragged
tail; the named workloads run at full size with sampled attention rows.
"""
import numpy as np
import pytest
import torch

from _helpers import (ORACLE_THREADS, check_attention, check_pairs_in_chunks, compare_buffers,
                      new_pair,
                      to_oracle_kv)
from bit_kv_cache_06_gb300 import build as kbuild
from bit_kv_cache_06_gb300 import kivi, synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available(), "GPU tests need CUDA"
    kbuild.build()
    kivi.load()


def _prefill_both(w, gc, oc, K, V, layout=kivi.KIVI_LAYOUT_BHTD):
    if layout == kivi.KIVI_LAYOUT_BTHD:
        gc.quantize_prefill(synth.to_bthd(K).cuda(), synth.to_bthd(V).cuda(), layout=layout)
    else:
        gc.quantize_prefill(K.cuda(), V.cuda())
    assert oc.prefill(to_oracle_kv(K), to_oracle_kv(V), nthreads=ORACLE_THREADS) == 0
    torch.cuda.synchronize()


# --------------------------------------------------------------- tiny C1 ---

@pytest.mark.parametrize("layout", [kivi.KIVI_LAYOUT_BHTD, kivi.KIVI_LAYOUT_BTHD])
def test_tiny_2bit_prefill_and_decode(layout):
    w = synth.C1
    K, V = synth.make_kv(w)
    gc, oc = new_pair(w)
    _prefill_both(w, gc, oc, K, V, layout)
    assert (gc.n_quant, gc.n_resid) == (256, 32)
    compare_buffers(gc, oc)
    q = synth.make_q(w).cuda()
    for S in range(1, gc.num_splits(kivi.decode_max_splits(gc.params)) + 1):
        out = gc.decode_attention(q, num_splits=S)
        torch.cuda.synchronize()
        check_attention(gc, oc, q, w.g, out)
    assert gc.workspace_status() == 0


def _offset16(x):
    """A contiguous copy of x whose data starts 16 bytes past a 32-byte boundary."""
    buf = torch.empty(x.numel() + 16, dtype=x.dtype, device="cuda")
    base = (-(buf.data_ptr() // 2)) % 16 + 8             # elements to the first 16 (mod 32) byte
    y = buf[base:base + x.numel()].view(x.shape)
    y.copy_(x.cuda())
    assert y.data_ptr() % 32 == 16
    return y


@pytest.mark.parametrize("bits,G,R", [(2, 32, 128), (4, 64, 128), (4, 16, 32)])
def test_inputs_16_byte_aligned_only(bits, G, R):
    """Inputs aligned to 16 bytes but not 32 (the quantiser's two-load path):
    same records as the oracle, for a prefill and for appends that flush."""
    w = synth.C2.with_(name="align16", B=2, Hq=8, Hkv=2, T=3 * R + 50, bits=bits, G=G, R=R)
    K, V = synth.make_kv(w)
    gc, oc = new_pair(w, cap=8 * R)
    gc.quantize_prefill(_offset16(K), _offset16(V))
    assert oc.prefill(to_oracle_kv(K), to_oracle_kv(V), nthreads=ORACLE_THREADS) == 0
    torch.cuda.synchronize()
    compare_buffers(gc, oc)
    g = torch.Generator().manual_seed(7)
    for _ in range(R):
        k1 = torch.randn(w.B, w.Hkv, w.d, generator=g).half()
        v1 = torch.randn(w.B, w.Hkv, w.d, generator=g).half()
        gc.append_token(_offset16(k1), _offset16(v1))
        assert oc.append(k1.reshape(w.pairs, w.d).numpy(), v1.reshape(w.pairs, w.d).numpy()) == 0
    torch.cuda.synchronize()
    compare_buffers(gc, oc)


# ------------------------------------------------------ shape/param sweep ---

SWEEP = [
    # bits, G, R, Hq, Hkv, B, T
    (2, 32, 32, 4, 1, 1, 288),
    (2, 32, 128, 32, 8, 2, 3 * 128 + 77),
    (4, 64, 128, 32, 8, 2, 5 * 128 + 1),
    (4, 32, 64, 8, 8, 3, 700),
    (2, 16, 32, 6, 2, 2, 555),
    (4, 16, 16, 3, 1, 2, 400),
    (2, 64, 64, 16, 2, 1, 1000),
    (2, 128, 128, 8, 1, 2, 1100),
    (4, 128, 256, 2, 2, 1, 1500),
    (2, 32, 128, 1, 1, 4, 129),
    (4, 32, 32, 7, 1, 1, 97),
]


@pytest.mark.parametrize("bits,G,R,Hq,Hkv,B,T", SWEEP)
def test_sweep_prefill_decode(bits, G, R, Hq, Hkv, B, T):
    w = synth.C2.with_(name="sweep", B=B, Hq=Hq, Hkv=Hkv, T=T, bits=bits, G=G, R=R,
                       index=100 + bits * 10 + G)
    K, V = synth.make_kv(w)
    gc, oc = new_pair(w)
    _prefill_both(w, gc, oc, K, V)
    compare_buffers(gc, oc)
    q = synth.make_q(w).cuda()
    Smax = gc.num_splits(kivi.decode_max_splits(gc.params))
    for S in sorted({1, 2, Smax, 0}):
        out = gc.decode_attention(q, num_splits=S)
        torch.cuda.synchronize()
        check_attention(gc, oc, q, w.g, out)


def test_chunked_prefill_and_appends_match_oracle():
    w = synth.C2.with_(name="chunks", B=2, Hq=8, Hkv=2, T=300, bits=2, G=32, R=64, steps=150)
    K, V = synth.make_kv(w, T=w.T)
    gc, oc = new_pair(w)
    for a, b in ((0, 1), (1, 65), (65, 200), (200, 300)):
        gc.quantize_prefill(K[:, :, a:b].contiguous().cuda(), V[:, :, a:b].contiguous().cuda())
        oc.prefill(to_oracle_kv(K[:, :, a:b]), to_oracle_kv(V[:, :, a:b]))
        torch.cuda.synchronize()
        compare_buffers(gc, oc)
    for step in range(w.steps):
        k, v = synth.make_token(w, step)
        gc.append_token(k.cuda(), v.cuda())
        oc.append(k.reshape(w.pairs, w.d).numpy(), v.reshape(w.pairs, w.d).numpy())
        if step % 37 == 0 or gc.n_resid == 1:
            torch.cuda.synchronize()
            compare_buffers(gc, oc)
            q = synth.make_q(w, step).cuda()
            out = gc.decode_attention(q)
            torch.cuda.synchronize()
            check_attention(gc, oc, q, w.g, out)
    torch.cuda.synchronize()
    compare_buffers(gc, oc)


# ----------------------------------------------------------- sink tokens ---
# "09 -- KV Cache Quantization", "Anti-patterns": keep the first N_s tokens of
# the sequence unquantised (preserve-first-N).

SINK_CFGS = [
    # bits, G, R, Hq, Hkv, B, N_s, T
    (2, 32, 128, 8, 2, 2, 4, 3),         # sink not yet full
    (2, 32, 128, 8, 2, 2, 4, 4),         # exactly full, nothing after it
    (2, 32, 128, 8, 2, 2, 4, 700),
    (4, 64, 128, 16, 2, 1, 37, 1000),    # query group 8, odd sink length
    (2, 16, 32, 6, 2, 2, 16, 555),       # CUDA-core kernel (G = 16)
    (4, 32, 64, 4, 4, 1, 128, 900),
    (2, 128, 128, 8, 1, 2, 256, 1500),   # the largest sink
]


@pytest.mark.parametrize("bits,G,R,Hq,Hkv,B,Ns,T", SINK_CFGS)
def test_sink_tokens_prefill_appends_decode(bits, G, R, Hq, Hkv, B, Ns, T):
    w = synth.C2.with_(name="sink", B=B, Hq=Hq, Hkv=Hkv, T=T, bits=bits, G=G, R=R,
                       index=600 + Ns + bits, steps=40)
    K, V = synth.make_kv(w)
    gc, oc = new_pair(w, sink=Ns)
    _prefill_both(w, gc, oc, K, V)
    assert gc.n_sink == min(Ns, T)
    compare_buffers(gc, oc)
    q = synth.make_q(w).cuda()
    for S in (1, 0):
        out = gc.decode_attention(q, num_splits=S)
        torch.cuda.synchronize()
        check_attention(gc, oc, q, w.g, out)
    for step in range(w.steps):
        k, v = synth.make_token(w, step)
        gc.append_token(k.cuda(), v.cuda())
        oc.append(k.reshape(w.pairs, w.d).numpy(), v.reshape(w.pairs, w.d).numpy())
        if step % 13 == 0 or gc.n_resid == 1:
            torch.cuda.synchronize()
            compare_buffers(gc, oc)
            q = synth.make_q(w, step).cuda()
            out = gc.decode_attention(q)
            torch.cuda.synchronize()
            check_attention(gc, oc, q, w.g, out)


def test_sink_chunked_prefill_equals_appends():
    w = synth.C2.with_(name="sinkchunks", B=1, Hq=8, Hkv=2, T=260, bits=2, G=32, R=64)
    K, V = synth.make_kv(w)
    gc, oc = new_pair(w, sink=10)
    for a, b in ((0, 3), (3, 11), (11, 12), (12, 200), (200, 260)):
        gc.quantize_prefill(K[:, :, a:b].contiguous().cuda(), V[:, :, a:b].contiguous().cuda())
        oc.prefill(to_oracle_kv(K[:, :, a:b]), to_oracle_kv(V[:, :, a:b]))
        torch.cuda.synchronize()
        compare_buffers(gc, oc)
    q = synth.make_q(w).cuda()
    out = gc.decode_attention(q)
    torch.cuda.synchronize()
    check_attention(gc, oc, q, w.g, out)


# ------------------------------------------------- fp16 scale / zero point ---
# "09 -- KV Cache Quantization", "KIVI -- the reference paper": scale and zero
# in fp16 (range-guarded: s rounded up to binary16, at least 2^-24 and
# |min| / 2048).

F16_CFGS = [
    # bits, G, R, Hq, Hkv, B, T
    (2, 32, 128, 32, 8, 2, 3 * 128 + 77),
    (4, 64, 128, 32, 8, 2, 5 * 128 + 1),
    (4, 32, 64, 8, 8, 3, 700),
    (2, 16, 32, 6, 2, 2, 555),
    (2, 64, 64, 16, 2, 1, 1000),
    (2, 128, 128, 8, 1, 2, 1100),
    (4, 128, 256, 2, 2, 1, 1500),
]


@pytest.mark.parametrize("bits,G,R,Hq,Hkv,B,T", F16_CFGS)
def test_fp16_metadata_prefill_decode(bits, G, R, Hq, Hkv, B, T):
    w = synth.C2.with_(name="f16", B=B, Hq=Hq, Hkv=Hkv, T=T, bits=bits, G=G, R=R,
                       index=700 + bits * 10 + G)
    K, V = synth.make_kv(w)
    K[0, 0, 0:G] = 100.0 + K[0, 0, 0:G] * 0.001        # narrow groups far from zero: the guard
    gc, oc = new_pair(w, meta=1)
    _prefill_both(w, gc, oc, K, V)
    compare_buffers(gc, oc)
    q = synth.make_q(w).cuda()
    for S in sorted({1, 0, gc.num_splits(kivi.decode_max_splits(gc.params))}):
        out = gc.decode_attention(q, num_splits=S)
        torch.cuda.synchronize()
        check_attention(gc, oc, q, w.g, out)


def test_fp16_metadata_llama3_8b_layer_full_size():
    """The 8B layer at 32K context with fp16 metadata (96 B per token-pair):
    every buffer and every query row, after the flushing append."""
    w = synth.C2
    K, V = synth.make_kv(w)
    gc, oc = new_pair(w, meta=1)
    _prefill_both(w, gc, oc, K, V)
    k, v = synth.make_token(w, 0)
    gc.append_token(k.cuda(), v.cuda())
    oc.append(k.reshape(w.pairs, w.d).numpy(), v.reshape(w.pairs, w.d).numpy())
    torch.cuda.synchronize()
    compare_buffers(gc, oc)
    q = synth.make_q(w).cuda()
    out = gc.decode_attention(q)
    torch.cuda.synchronize()
    check_attention(gc, oc, q, w.g, out)


# ------------------------------------------------ residual flush by group ---
# "KIVI: ...", "The streaming complication": a completed key group leaves the
# window as it slides (KIVI_FLUSH_GROUP); the residual slots form a ring.

FLUSH_CFGS = [
    # bits, G, R, Hq, Hkv, B, Ns, T
    (2, 32, 128, 8, 2, 2, 0, 700),
    (4, 64, 128, 16, 2, 1, 0, 1000),     # query group 8
    (2, 16, 32, 6, 2, 2, 0, 555),        # CUDA-core kernel
    (2, 32, 64, 8, 2, 1, 5, 300),        # with sink tokens
    (4, 32, 128, 4, 4, 1, 0, 130),       # still below the first flush
]


@pytest.mark.parametrize("bits,G,R,Hq,Hkv,B,Ns,T", FLUSH_CFGS)
def test_group_flush_prefill_appends_decode(bits, G, R, Hq, Hkv, B, Ns, T):
    w = synth.C2.with_(name="flushg", B=B, Hq=Hq, Hkv=Hkv, T=T, bits=bits, G=G, R=R,
                       index=800 + G + bits + Ns, steps=3 * R // 2)
    K, V = synth.make_kv(w)
    gc, oc = new_pair(w, sink=Ns, flush=1)
    _prefill_both(w, gc, oc, K, V)
    compare_buffers(gc, oc)
    heads = set()
    for step in range(w.steps):
        k, v = synth.make_token(w, step)
        gc.append_token(k.cuda(), v.cuda())
        oc.append(k.reshape(w.pairs, w.d).numpy(), v.reshape(w.pairs, w.d).numpy())
        heads.add(gc.resid_head)
        if step % 11 == 0 or gc.n_resid == R - G + 1:
            torch.cuda.synchronize()
            compare_buffers(gc, oc)
            q = synth.make_q(w, step).cuda()
            for S in (1, 0):
                out = gc.decode_attention(q, num_splits=S)
                torch.cuda.synchronize()
                check_attention(gc, oc, q, w.g, out)
    assert len(heads) == R // G or T + w.steps - Ns <= R   # the ring wrapped


# ------------------------------------------------------------------ FP8 KV ---
# "09 -- KV Cache Quantization", "The lazy default: FP8 KV"; "4.4 KV Cache
# quantization", section 4.2 (per-tensor scale, 1.0 uncalibrated).

FP8_CFGS = [
    # fmt, k_scale, v_scale, R, Hq, Hkv, B, T
    (1, 1.0, 1.0, 128, 32, 8, 2, 3 * 128 + 77),
    (2, 1.0, 1.0, 128, 32, 8, 2, 3 * 128 + 77),
    (1, 0.25, 2.0, 64, 16, 2, 1, 1000),      # query group 8, calibrated-style scales
    (2, 4.0, 0.5, 32, 6, 2, 2, 555),
]


@pytest.mark.parametrize("fmt,ks,vs,R,Hq,Hkv,B,T", FP8_CFGS)
def test_fp8_kv_prefill_appends_decode(fmt, ks, vs, R, Hq, Hkv, B, T):
    """Bytes of the FP8 history equal the oracle's (x / scale rounded to the
    format, saturated -- value outliers x200 exceed E4M3's 448); attention
    within 2e-3 of the fp64 oracle over the dequantised FP8 cache."""
    w = synth.C2.with_(name="fp8", B=B, Hq=Hq, Hkv=Hkv, T=T, bits=8, G=32, R=R,
                       index=900 + fmt, steps=40)
    K, V = synth.make_kv(w)
    gc, oc = new_pair(w, fp8=(fmt, ks, vs))
    _prefill_both(w, gc, oc, K, V)
    compare_buffers(gc, oc)
    q = synth.make_q(w).cuda()
    for S in (1, 0):
        out = gc.decode_attention(q, num_splits=S)
        torch.cuda.synchronize()
        check_attention(gc, oc, q, w.g, out)
    for step in range(w.steps):
        k, v = synth.make_token(w, step)
        gc.append_token(k.cuda(), v.cuda())
        oc.append(k.reshape(w.pairs, w.d).numpy(), v.reshape(w.pairs, w.d).numpy())
    torch.cuda.synchronize()
    compare_buffers(gc, oc)
    out = gc.decode_attention(q)
    torch.cuda.synchronize()
    check_attention(gc, oc, q, w.g, out)


# ------------------------------------------------------------ edge cases ---

def test_residual_only_cache_and_single_token():
    w = synth.C1.with_(T=1)
    K, V = synth.make_kv(w)
    gc, oc = new_pair(w)
    _prefill_both(w, gc, oc, K, V)
    assert (gc.n_quant, gc.n_resid) == (0, 1)
    compare_buffers(gc, oc)
    q = synth.make_q(w).cuda()
    out = gc.decode_attention(q)
    torch.cuda.synchronize()
    # one token: every head returns that token's value (fp16-rounded)
    ref = V[0, 0, 0].float()
    assert torch.equal(out.cpu().float()[0], ref.expand(w.Hq, -1))


RESID_CFGS = [
    # bits, G, R, Hq, Hkv: query groups 4 and 8, one head per kv head, a
    # 256-token window (several 16-token residual tiles per warp)
    (2, 32, 128, 8, 2),
    (2, 32, 128, 16, 2),
    (2, 64, 128, 2, 2),
    (4, 64, 256, 12, 3),
]


@pytest.mark.parametrize("bits,G,R,Hq,Hkv", RESID_CFGS)
def test_residual_window_fill_levels(bits, G, R, Hq, Hkv):
    """Decode after prefills that leave 1..R tokens in the fp16 window: the
    residual runs in 16-token tiles dealt to the last split's warps, with
    ragged last tiles."""
    for n_resid in sorted({1, 2, 15, 16, 17, 31, 33, 64, R - 1, R}):
        T = 2 * R + n_resid
        w = synth.C2.with_(name="resid", B=1, Hq=Hq, Hkv=Hkv, T=T, bits=bits, G=G, R=R,
                           index=300 + n_resid)
        K, V = synth.make_kv(w)
        gc, oc = new_pair(w)
        _prefill_both(w, gc, oc, K, V)
        assert (gc.n_quant, gc.n_resid) == (2 * R, n_resid)
        q = synth.make_q(w).cuda()
        for S in (1, 0):
            out = gc.decode_attention(q, num_splits=S)
            torch.cuda.synchronize()
            check_attention(gc, oc, q, w.g, out)


TWO_LAUNCH_CFGS = [
    # bits, G, R, Hq, Hkv, B, T
    (2, 16, 32, 8, 2, 1, 300),      # G = 16: CUDA-core kernel, residual as partial S
    (2, 32, 128, 8, 2, 2, 700),     # tensor cores, query group 4
    (2, 32, 128, 16, 2, 1, 650),    # tensor cores, query group 8
    (4, 64, 128, 4, 4, 1, 900),     # tensor cores, one query head per kv head
]


@pytest.mark.parametrize("bits,G,R,Hq,Hkv,B,T", TWO_LAUNCH_CFGS)
def test_two_launch_decode_equals_one_launch(bits, G, R, Hq, Hkv, B, T):
    """kivi_decode_partial + kivi_decode_combine give the one-launch output
    bit for bit (both merges run the same per-channel arithmetic)."""
    w = synth.C2.with_(name="two", B=B, Hq=Hq, Hkv=Hkv, T=T, bits=bits, G=G, R=R,
                       index=400 + G + bits)
    K, V = synth.make_kv(w)
    gc, oc = new_pair(w)
    _prefill_both(w, gc, oc, K, V)
    q = synth.make_q(w).cuda()
    for req in (0, 1, 3):
        S = gc.num_splits(req)
        one = gc.decode_attention(q, num_splits=S).clone()
        gc.decode_partial(q, num_splits=S)
        two = torch.empty_like(one)
        gc.decode_combine(two, S)
        torch.cuda.synchronize()
        assert torch.equal(one, two), f"S={S}"
        assert gc.workspace_status() == 0
    check_attention(gc, oc, q, w.g, two)


def test_cache_filled_to_capacity_then_capacity_error():
    w = synth.C1.with_(T=256 + 32)
    K, V = synth.make_kv(w)
    gc, oc = new_pair(w, cap=256)
    _prefill_both(w, gc, oc, K, V)
    assert gc.n_quant == 256 and gc.n_resid == 32
    k, v = synth.make_token(w, 0)
    with pytest.raises(kivi.KiviError) as e:
        gc.append_token(k.cuda(), v.cuda())
    assert e.value.status == kivi.KIVI_ERR_CAPACITY
    assert (gc.n_quant, gc.n_resid) == (256, 32)
    compare_buffers(gc, oc)
    q = synth.make_q(w).cuda()
    out = gc.decode_attention(q)
    torch.cuda.synchronize()
    check_attention(gc, oc, q, w.g, out)


def _edge_kv(w, key_const):
    K, V = synth.make_kv(w)
    K[0, 0, 0:64] = 1.5                     # constant key groups (scale floor)
    V[0, 0, 0:10] = 0.0                     # zero value tokens
    V[0, 1, 10:20] = -0.0
    K[0, 1, 64:96, 5] = key_const           # one constant, large key channel
    V[0, 1, 100] = -60000.0                 # near fp16 max value token
    K[0, 0, 128:160] = torch.round(K[0, 0, 128:160] * 2) / 2   # many exact ties
    V[0, 0, 200:260] = 7.0                  # constant value tokens
    return K, V


@pytest.mark.parametrize("meta", [0, 1])
@pytest.mark.parametrize("bits", [2, 4])
def test_quantizer_fp16_extremes_bit_exact(bits, meta):
    """Constant groups, zeros and -0, ties and fp16-range values (60000): codes,
    scales, zero points and residual still match the oracle bit for bit."""
    w = synth.C2.with_(name="edge", B=1, Hq=8, Hkv=2, T=600, bits=bits, G=32, R=64)
    K, V = _edge_kv(w, 60000.0)
    K[0, 1, 300:340, 77] = -65504.0
    gc, oc = new_pair(w, meta=meta)
    _prefill_both(w, gc, oc, K, V)
    compare_buffers(gc, oc)


@pytest.mark.parametrize("bits", [2, 4])
@pytest.mark.parametrize("key_const", [1000.0, 60000.0])
def test_attention_on_edge_groups(bits, key_const):
    """The same edge cases, attention within 2e-3: constant key groups (the
    1e-8 scale floor of the INT4 page's listing), zero and -0 value tokens, a
    near-fp16-max value token, and one constant key channel at the pages'
    largest stated outlier scale (1000) or near the fp16 maximum (60000).  At
    60000 the channel's zero point is about -6e12 and a query head that sees
    it scores its 32 tokens near |tau q.k| = 7.6e3 (log2 units), so a plain
    fp32 rounding of each score is already 2.4e-4."""
    w = synth.C2.with_(name="edge", B=1, Hq=8, Hkv=2, T=600, bits=bits, G=32, R=64)
    K, V = _edge_kv(w, key_const)
    gc, oc = new_pair(w)
    _prefill_both(w, gc, oc, K, V)
    compare_buffers(gc, oc)
    q = synth.make_q(w).cuda()
    out = gc.decode_attention(q)
    torch.cuda.synchronize()
    check_attention(gc, oc, q, w.g, out)


def test_split_count_invariance():
    w = synth.C2.with_(name="splits", B=1, Hq=8, Hkv=2, T=4096 + 100, bits=2, G=32, R=128)
    K, V = synth.make_kv(w)
    gc, oc = new_pair(w)
    _prefill_both(w, gc, oc, K, V)
    q = synth.make_q(w).cuda()
    outs = []
    for S in (1, 2, 3, 7, 16, 31):
        outs.append(gc.decode_attention(q, num_splits=S).float().cpu())
    base = outs[0]
    for o in outs[1:]:
        assert (o - base).abs().max().item() <= 2e-3 * base.abs().max().item()
    check_attention(gc, oc, q, w.g, gc.decode_attention(q, num_splits=5))


def test_explicit_softmax_scale():
    w = synth.C1
    K, V = synth.make_kv(w)
    gc, oc = new_pair(w)
    _prefill_both(w, gc, oc, K, V)
    q = synth.make_q(w).cuda()
    for tau in (0.02, 0.3):
        out = gc.decode_attention(q, softmax_scale=tau)
        torch.cuda.synchronize()
        check_attention(gc, oc, q, w.g, out, tau=tau)


# ------------------------------------------------------ named workloads ---

def test_c2_llama3_8b_layer_full_size():
    """Llama-3-8B layer, 32K context, 2-bit: every buffer and every one of the
    256 query rows, after the prefill (full 128-token residual) and after the
    flushing append (one residual token) -- the bench's decode state."""
    w = synth.C2
    K, V = synth.make_kv(w)
    gc, oc = new_pair(w)
    _prefill_both(w, gc, oc, K, V)
    assert (gc.n_quant, gc.n_resid) == (32640, 128)
    compare_buffers(gc, oc)
    q = synth.make_q(w).cuda()
    out = gc.decode_attention(q)          # the bench's launch configuration
    torch.cuda.synchronize()
    check_attention(gc, oc, q, w.g, out)
    # the next token flushes the full residual: 32768 quantised + 1 residual
    k, v = synth.make_token(w, 0)
    gc.append_token(k.cuda(), v.cuda())
    oc.append(k.reshape(w.pairs, w.d).numpy(), v.reshape(w.pairs, w.d).numpy())
    torch.cuda.synchronize()
    assert (gc.n_quant, gc.n_resid) == (32768, 1)
    compare_buffers(gc, oc)
    out = gc.decode_attention(q)
    torch.cuda.synchronize()
    check_attention(gc, oc, q, w.g, out)


def test_c3_streaming_4bit_every_step():
    """Streaming 4-bit, batch 32: 256 steps of append + decode; every buffer
    after every flush and every one of the 1024 query rows at every step."""
    w = synth.C3
    K, V = synth.make_kv(w)
    gc, oc = new_pair(w)
    _prefill_both(w, gc, oc, K, V)
    compare_buffers(gc, oc)
    for step in range(w.steps):
        k, v = synth.make_token(w, step)
        gc.append_token(k.cuda(), v.cuda())
        oc.append(k.reshape(w.pairs, w.d).numpy(), v.reshape(w.pairs, w.d).numpy())
        q = synth.make_q(w, step).cuda()
        out = gc.decode_attention(q)
        torch.cuda.synchronize()
        if gc.n_resid == 1:
            compare_buffers(gc, oc)
        check_attention(gc, oc, q, w.g, out)
    assert gc.n_quant == 8064 + 256 and gc.n_resid == 128
    compare_buffers(gc, oc)


@pytest.mark.slow
@pytest.mark.parametrize("sink", [0, 4])
def test_c4_llama3_70b_layer_1m_context(sink):
    """Llama-3-70B layer, 1M context, 2-bit, x1000 sink value token: every
    buffer and all 64 query rows; quantised as plain KIVI and with the first
    4 tokens kept fp16 ("09 -- KV Cache Quantization", Anti-patterns)."""
    w = synth.C4
    K, V = synth.make_kv(w)
    gc, oc = new_pair(w, sink=sink)
    _prefill_both(w, gc, oc, K, V)
    tq = w.T - sink                        # tokens after the sink
    r = (tq - 1) % w.R + 1
    assert (gc.n_sink, gc.n_quant, gc.n_resid) == (sink, tq - r, r)
    compare_buffers(gc, oc)
    del K, V
    q = synth.make_q(w).cuda()
    out = gc.decode_attention(q)
    torch.cuda.synchronize()
    check_attention(gc, oc, q, w.g, out)


C5_CELLS = [(bits, B, T) for bits in synth.C5_BITS for B in synth.C5_BATCHES
            for T in synth.C5_CONTEXTS]


@pytest.mark.slow
@pytest.mark.parametrize("bits,B,T", C5_CELLS, ids=lambda x: str(x))
def test_c5_32_layer_sweep_cell(bits, B, T):
    """One (batch, context, bits) cell of the 32-layer Llama-3-8B sweep, as the
    sweep runs it: a prefill of the whole context (one chunk of at most
    131072 tokens), one appended token and one decode per layer.  Layer 0:
    every pair's buffers and every query row (oracle built 64 pairs at a
    time); layers 1..31: a strided pair sample (buffers and those pairs'
    rows) -- every layer on cells up to 512K tokens, layers 7, 15 and 31 on
    the larger ones."""
    base = synth.C5.with_(bits=bits, B=B, T=T)
    big = B * T > (1 << 19)
    layers = [0] + ([7, 15, 31] if big else list(range(1, base.layers)))
    for layer in layers:
        w = base
        K, V = synth.make_kv(w, layer=layer, device="cuda")
        gc = kivi.KiviCache(kivi.CacheShape(w.bits, w.G, w.R, w.B, w.Hq, w.Hkv, w.d,
                                            w.capacity()))
        gc.quantize_prefill(K, V)
        k, v = synth.make_token(w, 0, layer=layer, device="cuda")
        gc.append_token(k, v)
        K = torch.cat([K, k[:, :, None]], dim=2)
        V = torch.cat([V, v[:, :, None]], dim=2)
        q = synth.make_q(w, layer=layer, device="cuda")
        out = gc.decode_attention(q)
        torch.cuda.synchronize()
        if layer == 0:
            pairs = range(w.pairs)
        else:
            pairs = range(layer % 3, w.pairs, max(1, w.pairs // 2))
        check_pairs_in_chunks(gc, w, K, V, q, out, pairs)
        del K, V, gc
        torch.cuda.empty_cache()

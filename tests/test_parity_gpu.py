"""GPU parity: the CUDA path through the C ABI against the CPU oracle.

Codes, scales, zero points, residual bytes and the bookkeeping must match bit
for bit; attention rows within 2e-3 max relative error (fp32 accumulation
against the fp64 oracle).  Sizes span several 128-token tiles and a ragged
tail; the named workloads run at full size with sampled attention rows.
"""
import numpy as np
import pytest
import torch

from _helpers import (ORACLE_THREADS, check_attention, compare_buffers, new_pair,
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


@pytest.mark.parametrize("bits", [2, 4])
def test_quantizer_fp16_extremes_bit_exact(bits):
    """Constant groups, zeros and -0, ties and fp16-range values (60000): codes,
    scales, zero points and residual still match the oracle bit for bit."""
    w = synth.C2.with_(name="edge", B=1, Hq=8, Hkv=2, T=600, bits=bits, G=32, R=64)
    K, V = _edge_kv(w, 60000.0)
    K[0, 1, 300:340, 77] = -65504.0
    gc, oc = new_pair(w)
    _prefill_both(w, gc, oc, K, V)
    compare_buffers(gc, oc)


@pytest.mark.parametrize("bits", [2, 4])
def test_attention_on_edge_groups(bits):
    """The same edge cases with the key outlier at the pages' largest stated
    scale (1000x): attention within 2e-3.  (A constant key channel near the
    fp16 maximum puts |tau q.k| in the thousands, where fp32 accumulation of
    a score alone exceeds the tolerance.)"""
    w = synth.C2.with_(name="edge", B=1, Hq=8, Hkv=2, T=600, bits=bits, G=32, R=64)
    K, V = _edge_kv(w, 1000.0)
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
    w = synth.C2
    K, V = synth.make_kv(w)
    gc, oc = new_pair(w)
    _prefill_both(w, gc, oc, K, V)
    assert (gc.n_quant, gc.n_resid) == (32640, 128)
    compare_buffers(gc, oc)
    q = synth.make_q(w).cuda()
    out = gc.decode_attention(q)          # the bench's launch configuration
    torch.cuda.synchronize()
    rows = np.random.default_rng(2).choice(w.B * w.Hq, 24, replace=False)
    check_attention(gc, oc, q, w.g, out, rows=rows)
    # the next token flushes the full residual: 32768 quantised + 1 residual
    k, v = synth.make_token(w, 0)
    gc.append_token(k.cuda(), v.cuda())
    oc.append(k.reshape(w.pairs, w.d).numpy(), v.reshape(w.pairs, w.d).numpy())
    torch.cuda.synchronize()
    assert (gc.n_quant, gc.n_resid) == (32768, 1)
    compare_buffers(gc, oc)
    out = gc.decode_attention(q)
    torch.cuda.synchronize()
    check_attention(gc, oc, q, w.g, out, rows=rows)


def test_c3_streaming_4bit_every_step():
    w = synth.C3
    K, V = synth.make_kv(w)
    gc, oc = new_pair(w)
    _prefill_both(w, gc, oc, K, V)
    compare_buffers(gc, oc)
    rng = np.random.default_rng(3)
    for step in range(w.steps):
        k, v = synth.make_token(w, step)
        gc.append_token(k.cuda(), v.cuda())
        oc.append(k.reshape(w.pairs, w.d).numpy(), v.reshape(w.pairs, w.d).numpy())
        q = synth.make_q(w, step).cuda()
        out = gc.decode_attention(q)
        torch.cuda.synchronize()
        flush = gc.n_resid == 1
        if flush:
            compare_buffers(gc, oc)
        rows = None if flush else rng.choice(w.B * w.Hq, 16, replace=False)
        check_attention(gc, oc, q, w.g, out, rows=rows)
    assert gc.n_quant == 8064 + 256 and gc.n_resid == 128
    compare_buffers(gc, oc)


@pytest.mark.slow
def test_c4_llama3_70b_layer_1m_context():
    w = synth.C4
    K, V = synth.make_kv(w)
    gc, oc = new_pair(w)
    _prefill_both(w, gc, oc, K, V)
    assert (gc.n_quant, gc.n_resid) == (1048448, 128)
    compare_buffers(gc, oc)
    del K, V
    q = synth.make_q(w).cuda()
    out = gc.decode_attention(q)
    torch.cuda.synchronize()
    rows = np.array([0, 9, 18, 27, 36, 45, 54, 63])   # one query head per kv head
    check_attention(gc, oc, q, w.g, out, rows=rows)


@pytest.mark.parametrize("bits", [2, 4])
def test_c5_32_layer_sweep_cells(bits):
    """Two cells of the 32-layer sweep: (B=1, T=4096) every layer, layer 0
    fully compared and the others on sampled heads; (B=16, T=32768) layer 0
    with a strided pair sample."""
    base = synth.C5.with_(bits=bits)
    rng = np.random.default_rng(50 + bits)
    w = base.with_(B=1, T=4096)
    for layer in range(w.layers):
        K, V = synth.make_kv(w, layer=layer)
        gc, oc = new_pair(w)
        _prefill_both(w, gc, oc, K, V)
        compare_buffers(gc, oc) if layer == 0 else compare_buffers(gc, oc, pairs=[layer % 8])
        q = synth.make_q(w, layer=layer).cuda()
        out = gc.decode_attention(q)
        torch.cuda.synchronize()
        rows = None if layer == 0 else rng.choice(w.B * w.Hq, 4, replace=False)
        check_attention(gc, oc, q, w.g, out, rows=rows)
    w = base.with_(B=16, T=32768)
    K, V = synth.make_kv(w)
    gc, oc = new_pair(w)
    _prefill_both(w, gc, oc, K, V)
    compare_buffers(gc, oc, pairs=list(range(0, w.pairs, 9)))
    q = synth.make_q(w).cuda()
    out = gc.decode_attention(q)
    torch.cuda.synchronize()
    check_attention(gc, oc, q, w.g, out, rows=rng.choice(w.B * w.Hq, 16, replace=False))

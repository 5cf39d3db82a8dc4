"""Guard bytes around every caller-owned buffer: the history, the fp16 rows,
the decode workspace, the query and the output each sit in the middle of a
larger allocation whose 4 KB margins hold a fixed pattern.  After prefills,
appends that flush, decodes with automatic and explicit split counts and the
two-launch decode, every margin must still hold its pattern (no kernel
writes or clobbers memory outside the buffers it was given), and the cache
must still match the oracle."""
import ctypes

import pytest
import torch

from _helpers import check_attention, compare_buffers, shape_of, to_oracle_kv, ORACLE_THREADS
from bit_kv_cache_06_gb300 import kivi, synth
import oracle

pytestmark = pytest.mark.gpu

GUARD = 4096
PATTERN = 0xA5


def _guarded(nbytes, dtype):
    """(view of nbytes as dtype, the whole uint8 allocation)."""
    raw = torch.full((nbytes + 2 * GUARD,), PATTERN, dtype=torch.uint8, device="cuda")
    inner = raw[GUARD:GUARD + nbytes]
    return inner.view(dtype), raw


def _intact(raw, nbytes):
    head = raw[:GUARD]
    tail = raw[GUARD + nbytes:]
    return bool((head == PATTERN).all()) and bool((tail == PATTERN).all())


CFGS = [
    # bits, G, R, Hq, Hkv, B, T, sink, meta, flush, fp8
    (2, 32, 128, 8, 2, 2, 700, 0, 0, 0, (0, 1.0, 1.0)),
    (4, 64, 128, 16, 2, 1, 1000, 5, 1, 1, (0, 1.0, 1.0)),
    (2, 16, 32, 6, 2, 2, 555, 0, 0, 0, (0, 1.0, 1.0)),
    (8, 32, 64, 8, 2, 2, 600, 0, 0, 0, (1, 0.5, 2.0)),
]


@pytest.mark.parametrize("bits,G,R,Hq,Hkv,B,T,sink,meta,flush,fp8", CFGS)
def test_no_kernel_writes_outside_its_buffers(bits, G, R, Hq, Hkv, B, T, sink, meta, flush, fp8):
    w = synth.C2.with_(name="guard", B=B, Hq=Hq, Hkv=Hkv, T=T, bits=bits, G=G, R=R)
    cap = w.capacity() + 4 * R
    shape = shape_of(w, cap, sink, meta, flush, fp8)
    L = kivi.load()
    params = shape.params()
    guarded = []
    bufs = []
    for i, dt in enumerate(kivi.BUFFER_DTYPES):
        nbytes = L.kivi_cache_buffer_bytes(ctypes.byref(params), i)
        inner, raw = _guarded(nbytes, dt)
        bufs.append(inner)
        guarded.append((raw, nbytes))
    gc = kivi.KiviCache(shape, buffers=bufs)
    ws_bytes = gc.workspace.numel()
    ws, ws_raw = _guarded(ws_bytes, torch.uint8)
    ws.zero_()
    gc.workspace = ws
    guarded.append((ws_raw, ws_bytes))
    oc = oracle.OracleCache(w.pairs, w.d, w.bits, w.G, w.R, cap, Ns=sink, meta=meta,
                            flush=flush, fp8=fp8[0], fp8_k_scale=fp8[1], fp8_v_scale=fp8[2])

    K, V = synth.make_kv(w)
    gc.quantize_prefill(K.cuda(), V.cuda())
    assert oc.prefill(to_oracle_kv(K), to_oracle_kv(V), nthreads=ORACLE_THREADS) == 0
    for step in range(R + 3):                      # crosses at least one flush
        k, v = synth.make_token(w, step)
        gc.append_token(k.cuda(), v.cuda())
        assert oc.append(k.reshape(w.pairs, w.d).numpy(), v.reshape(w.pairs, w.d).numpy()) == 0
    torch.cuda.synchronize()
    compare_buffers(gc, oc)

    qn = B * Hq * w.d * 2
    q_in, q_raw = _guarded(qn, torch.float16)
    q_in.copy_(synth.make_q(w).reshape(-1).cuda())
    q = q_in.view(B, Hq, w.d)
    o_flat, o_raw = _guarded(qn, torch.float16)
    out = o_flat.view(B, Hq, w.d)
    guarded += [(q_raw, qn), (o_raw, qn)]
    smax = gc.num_splits(kivi.decode_max_splits(gc.params))
    for S in sorted({0, 1, smax}):
        gc.decode_attention(q, out, num_splits=S)
        torch.cuda.synchronize()
        check_attention(gc, oc, q, w.g, out)
    gc.decode_partial(q, num_splits=smax)
    gc.decode_combine(out, num_splits=smax)
    torch.cuda.synchronize()
    check_attention(gc, oc, q, w.g, out)
    assert gc.workspace_status() == 0
    for raw, nbytes in guarded:
        assert _intact(raw, nbytes)

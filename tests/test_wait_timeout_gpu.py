"""The failure path of the decode's bounded waits, exercised on the GPU
without a fault: kivi_test_decode_wait_timeout arms one warp's first bulk
copy for 16 bytes more than it brings, so that warp's wait on it runs out
after its bound (about 2 s).  The call must return, set the status bit,
leave every other row exactly as a normal decode computes it, and leave the
context usable for the next decode."""
import ctypes
import time

import pytest
import torch

from _helpers import check_attention, new_pair, to_oracle_kv, ORACLE_THREADS
from bit_kv_cache_06_gb300 import kivi, synth

pytestmark = pytest.mark.gpu


def test_decode_bounded_wait_gives_up_cleanly():
    w = synth.C2.with_(name="timeout", B=2, Hq=8, Hkv=2, T=4096 + 1, bits=2, G=32, R=128)
    K, V = synth.make_kv(w)
    gc, oc = new_pair(w)
    gc.quantize_prefill(K.cuda(), V.cuda())
    assert oc.prefill(to_oracle_kv(K), to_oracle_kv(V), nthreads=ORACLE_THREADS) == 0
    q = synth.make_q(w).cuda()
    ref = gc.decode_attention(q)
    torch.cuda.synchronize()
    assert gc.workspace_status() == 0

    L = kivi.load()
    out = torch.full_like(q, float("nan"))
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    t0 = time.time()
    st = L.kivi_test_decode_wait_timeout(
        ctypes.byref(gc.c), ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(out.data_ptr()),
        ctypes.c_void_p(gc.workspace.data_ptr()), gc.workspace.numel(), stream)
    torch.cuda.synchronize()
    elapsed = time.time() - t0
    assert st == kivi.KIVI_OK
    assert gc.workspace_status() & kivi.KIVI_STATUS_WAIT_TIMEOUT
    assert 0.5 < elapsed < 60.0                   # the bounded wait ran out, then returned
    # pair 0 is batch 0, kv head 0: query heads 0 .. g-1 of batch 0
    g = w.Hq // w.Hkv
    assert torch.isfinite(out[0, :g].float()).all()
    assert torch.equal(out[0, g:], ref[0, g:])
    assert torch.equal(out[1:], ref[1:])

    # the context stays usable: clear the sticky status word, decode again
    gc.workspace.zero_()
    again = gc.decode_attention(q)
    torch.cuda.synchronize()
    assert gc.workspace_status() == 0
    assert torch.equal(again, ref)
    check_attention(gc, oc, q, w.g, again)


def test_test_hook_refuses_caches_without_the_tensor_core_decode():
    for bits, G, nq in ((2, 16, 4096), (2, 32, 0)):
        w = synth.C2.with_(name="hook", B=1, Hq=4, Hkv=1, T=64, bits=bits, G=G, R=32)
        gc, _ = new_pair(w, cap=4096)
        gc.c.n_quant, gc.c.n_resid = nq, 1
        q = torch.zeros(1, 4, 128, dtype=torch.float16, device="cuda")
        out = torch.empty_like(q)
        st = kivi.load().kivi_test_decode_wait_timeout(
            ctypes.byref(gc.c), ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(out.data_ptr()),
            ctypes.c_void_p(gc.workspace.data_ptr()), gc.workspace.numel(), None)
        assert st == kivi.KIVI_ERR_UNSUPPORTED

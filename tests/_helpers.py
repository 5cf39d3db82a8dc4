"""Shared helpers for the parity tests: build matching GPU and oracle caches
from the same seeded inputs and compare them."""
import os

import numpy as np
import torch

import oracle
from bit_kv_cache_06_gb300 import kivi
from bit_kv_cache_06_gb300.synth import Workload

ORACLE_THREADS = max(1, min(16, os.cpu_count() or 1))
ATTN_TOL = 2e-3      # max relative error per output row (spec tolerance)


def shape_of(w: Workload, cap: int, sink: int = 0, meta: int = 0, flush: int = 0,
             fp8=(0, 1.0, 1.0)) -> kivi.CacheShape:
    return kivi.CacheShape(bits=w.bits, group=w.G, residual=w.R, batch=w.B, num_q_heads=w.Hq,
                           num_kv_heads=w.Hkv, head_dim=w.d, capacity_tokens=cap,
                           sink_tokens=sink, meta=meta, flush=flush, fp8_format=fp8[0],
                           fp8_k_scale=fp8[1], fp8_v_scale=fp8[2])


def new_pair(w: Workload, cap: int = None, sink: int = 0, meta: int = 0, flush: int = 0,
             fp8=(0, 1.0, 1.0)):
    """A GPU cache and an oracle cache of the same shape (meta: 0 = fp32
    scales and zero points, 1 = fp16; flush: 0 = whole window, 1 = one key
    group at a time; fp8: (format, k scale, v scale) with bits 8)."""
    cap = w.capacity() if cap is None else cap
    gc = kivi.KiviCache(shape_of(w, cap, sink, meta, flush, fp8))
    oc = oracle.OracleCache(w.pairs, w.d, w.bits, w.G, w.R, cap, Ns=sink, meta=meta,
                            flush=flush, fp8=fp8[0], fp8_k_scale=fp8[1], fp8_v_scale=fp8[2])
    return gc, oc


def to_oracle_kv(x: torch.Tensor) -> np.ndarray:
    """fp16 [B, Hkv, T, d] (any device) -> numpy fp16 [P, T, d]."""
    B, H, T, d = x.shape
    return x.detach().cpu().reshape(B * H, T, d).numpy()


def _record_part(oc, off):
    """Name of the record field at byte offset `off` (for failure messages)."""
    d, G, rb = oc.d, oc.G, oc.d * oc.bits // 8
    if oc.fp8:
        return "K8" if off < 32 * d else "V8"
    mw = 2 if oc.meta else 4
    if off < mw * d:
        return "Ks"
    if off < 2 * mw * d:
        return "Kz"
    sl = min(G, 32)
    o = (off - 2 * mw * d) % (sl * (2 * rb + 2 * mw * (d // G)))
    for name, size in (("Kc", sl * rb), ("Vc", sl * rb), ("Vs", mw * sl * (d // G)),
                       ("Vz", mw * sl * (d // G))):
        if o < size:
            return name
        o -= size
    return "?"


def compare_buffers(gc: kivi.KiviCache, oc: oracle.OracleCache, pairs=None):
    """Bit-exact comparison of every filled cache region -- the history
    records (codes, scales, zero points) against the oracle's own export of
    the same layout, the sink rows and the residual slots -- and of the
    bookkeeping."""
    assert (gc.n_quant, gc.n_resid, gc.n_sink) == (oc.n_quant, oc.n_resid, oc.n_sink)
    nq, nr, ns, G, Ns = oc.n_quant, oc.n_resid, oc.n_sink, oc.G, oc.Ns
    gpairs = list(range(oc.P)) if pairs is None else list(pairs)
    # with an explicit pair list the oracle may hold exactly those pairs
    opairs = list(range(len(gpairs))) if oc.P == len(gpairs) else gpairs
    idx = torch.as_tensor(gpairs, device=gc.device)
    hist = gc.view("history")[idx, :nq // G].cpu().numpy()
    for i, (gp, op) in enumerate(zip(gpairs, opairs)):
        ref = oc.export_history(op)
        if not np.array_equal(hist[i], ref):
            bad = np.argwhere(hist[i] != ref)
            j, off = bad[0]
            raise AssertionError(f"history pair {gp}: {len(bad)} bytes differ, first in record "
                                 f"{j} at byte {off} ({_record_part(oc, off)})")
    kf = gc.view("k_fp16")[idx].cpu().numpy().view(np.uint16)
    vf = gc.view("v_fp16")[idx].cpu().numpy().view(np.uint16)
    # the residual slots are a ring: oldest token in slot resid_head (the
    # oracle keeps its residual oldest first)
    ring = [Ns + (gc.resid_head + i) % oc.R for i in range(nr)]
    checks = [
        ("k_sink", kf[:, :ns], oc.kr[opairs, :ns]),
        ("v_sink", vf[:, :ns], oc.vr[opairs, :ns]),
        ("k_resid", kf[:, ring], oc.kres[opairs, :nr]),
        ("v_resid", vf[:, ring], oc.vres[opairs, :nr]),
    ]
    for name, got, ref in checks:
        if not np.array_equal(got, ref):
            bad = np.argwhere(got != ref)
            raise AssertionError(f"{name}: {len(bad)} mismatches, first at {bad[:5].tolist()}")


def row_rel_err(out: np.ndarray, ref: np.ndarray) -> np.ndarray:
    """Per-row max |o - o_ref| / max |o_ref| (rows = query heads)."""
    out = out.reshape(-1, out.shape[-1]).astype(np.float64)
    ref = ref.reshape(-1, ref.shape[-1])
    num = np.abs(out - ref).max(axis=1)
    den = np.abs(ref).max(axis=1)
    return num / np.maximum(den, 1e-300)


def check_attention(gc, oc, q: torch.Tensor, g: int, out: torch.Tensor, rows=None,
                    tau=None, tol=ATTN_TOL):
    """Compare GPU decode output (all or sampled rows) with the fp64 oracle."""
    qn = q.detach().cpu().numpy().reshape(-1, q.shape[-1])
    ref = oc.attention(qn, g, tau=tau, rows=rows, nthreads=ORACLE_THREADS)
    got = out.detach().cpu().float().numpy().reshape(-1, q.shape[-1])
    if rows is not None:
        got = got[np.asarray(rows)]
    err = row_rel_err(got, ref)
    assert np.all(np.isfinite(got)), "non-finite attention output"
    assert err.max() <= tol, f"max row rel err {err.max():.3e} > {tol} (row {err.argmax()})"
    return float(err.max())


def check_pairs_in_chunks(gc, w, K, V, q, out, pairs, chunk=64, tau=None, tol=ATTN_TOL):
    """Bit-exact buffers and attention rows of the listed (batch, kv-head)
    pairs, with the oracle built for `chunk` pairs at a time so that host
    memory stays bounded on full-size layers.  K, V: fp16 [B, Hkv, T, d]
    (any device) as handed to the GPU prefill; q, out: [B, Hq, d]."""
    import oracle as _oracle
    P, T, d = w.pairs, K.shape[2], w.d
    Kp, Vp = K.reshape(P, T, d), V.reshape(P, T, d)
    qn = q.detach().cpu().numpy().reshape(P, w.g, d)
    got_all = out.detach().cpu().float().numpy().reshape(P, w.g, d)
    worst = 0.0
    pairs = list(pairs)
    for c0 in range(0, len(pairs), chunk):
        sel = pairs[c0:c0 + chunk]
        idx = torch.as_tensor(sel, device=Kp.device)
        sh = gc.shape
        oc = _oracle.OracleCache(len(sel), d, w.bits, w.G, w.R, sh.capacity_tokens,
                                 Ns=sh.sink_tokens, meta=sh.meta, flush=sh.flush,
                                 fp8=sh.fp8_format, fp8_k_scale=sh.fp8_k_scale,
                                 fp8_v_scale=sh.fp8_v_scale)
        assert oc.prefill(Kp[idx].cpu().numpy(), Vp[idx].cpu().numpy(),
                          nthreads=ORACLE_THREADS) == 0
        compare_buffers(gc, oc, pairs=sel)
        ref = oc.attention(qn[sel].reshape(-1, d), w.g, tau=tau, nthreads=ORACLE_THREADS)
        got = got_all[sel].reshape(-1, d)
        err = row_rel_err(got, ref)
        assert np.all(np.isfinite(got)), "non-finite attention output"
        assert err.max() <= tol, f"pairs {sel[:4]}...: max row rel err {err.max():.3e} > {tol}"
        worst = max(worst, float(err.max()))
        del oc
    return worst

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


def shape_of(w: Workload, cap: int) -> kivi.CacheShape:
    return kivi.CacheShape(bits=w.bits, group=w.G, residual=w.R, batch=w.B, num_q_heads=w.Hq,
                           num_kv_heads=w.Hkv, head_dim=w.d, capacity_tokens=cap)


def new_pair(w: Workload, cap: int = None):
    cap = w.capacity() if cap is None else cap
    gc = kivi.KiviCache(shape_of(w, cap))
    oc = oracle.OracleCache(w.pairs, w.d, w.bits, w.G, w.R, cap)
    return gc, oc


def to_oracle_kv(x: torch.Tensor) -> np.ndarray:
    """fp16 [B, Hkv, T, d] (any device) -> numpy fp16 [P, T, d]."""
    B, H, T, d = x.shape
    return x.detach().cpu().reshape(B * H, T, d).numpy()


def compare_buffers(gc: kivi.KiviCache, oc: oracle.OracleCache, pairs=None):
    """Bit-exact comparison of every filled cache region (codes, scales, zero
    points, residual) and of the bookkeeping."""
    assert (gc.n_quant, gc.n_resid) == (oc.n_quant, oc.n_resid)
    nq, nr, G = oc.n_quant, oc.n_resid, oc.G
    sel = slice(None) if pairs is None else pairs

    def g(name, rows):
        t = gc.view(name)
        if pairs is None:
            return t[:, :rows].cpu().numpy()
        return t[torch.as_tensor(pairs, device=t.device), :rows].cpu().numpy()

    # with an explicit pair list the oracle may hold exactly those pairs
    if pairs is not None and oc.P == len(pairs):
        sel = slice(None)
    checks = [
        ("k_codes", g("k_codes", nq), oc.kc[sel, :nq]),
        ("v_codes", g("v_codes", nq), oc.vc[sel, :nq]),
        ("k_scale", g("k_scale", nq // G).view(np.uint32), oc.ks[sel, :nq // G].view(np.uint32)),
        ("k_zero", g("k_zero", nq // G).view(np.uint32), oc.kz[sel, :nq // G].view(np.uint32)),
        ("v_scale", g("v_scale", nq).view(np.uint32), oc.vs[sel, :nq].view(np.uint32)),
        ("v_zero", g("v_zero", nq).view(np.uint32), oc.vz[sel, :nq].view(np.uint32)),
        ("k_resid", g("k_resid", nr).view(np.uint16), oc.kres[sel, :nr]),
        ("v_resid", g("v_resid", nr).view(np.uint16), oc.vres[sel, :nr]),
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
        oc = _oracle.OracleCache(len(sel), d, w.bits, w.G, w.R, gc.shape.capacity_tokens)
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

"""Pins of the CPU oracle to facts outside itself (no GPU needed).

Each test checks the oracle against something the pages print, a closed form,
a brute-force search, or a library routine -- chosen so that a dropped term,
a wrong sign or index, or a transposed operand in the oracle fails one.
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ------------------------------------------------------------ byte formula ---

def _golden_rows(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            nums, src = line.split("|", 1)
            L, B, T, H, d, b, exp, tol = nums.split()
            rows.append((int(L), int(B), int(T), int(H), int(d), float(b),
                         float(exp), float(tol), src.strip()))
    return rows


@pytest.mark.parametrize("row", _golden_rows("kv_bytes_pages.txt"), ids=lambda r: r[-1][:48])
def test_kv_bytes_matches_page_values(row):
    L, B, T, H, d, b, exp, tol, src = row
    got = oracle.kv_bytes(L, B, T, H, d, b)
    assert abs(got - exp) <= tol, (got, exp, src)


def test_kv_bytes_is_linear_in_each_factor():
    base = oracle.kv_bytes(3, 5, 7, 11, 13, 2)
    assert base == 2 * 3 * 5 * 7 * 11 * 13 * 2
    for i in range(5):
        args = [3, 5, 7, 11, 13]
        args[i] *= 2
        assert oracle.kv_bytes(*args, 2) == 2 * base


# -------------------------------------------------------- fp16 conversion ---

def test_half_to_double_matches_numpy_for_every_pattern():
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([oracle.half_to_double(int(b)) for b in bits])
    finite = np.isfinite(ref)
    assert np.array_equal(got[finite], ref[finite])
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    assert np.array_equal(np.isinf(got), np.isinf(ref))


# ---------------------------------------------------------- the quantiser ---

def test_hand_worked_2bit_group():
    # x = [-1, 0, 0.5, 1.5, 2]: min -1, max 2 -> s = 3/3 = 1, z = round(1) = 1.
    # codes = round(x/s) + z, round half to even: round(0.5) = 0, round(1.5) = 2
    s, z = oracle.quant_params(-1.0, 2.0, 2)
    assert (s, z) == (1.0, 1.0)
    assert [oracle.encode(x, s, z, 2) for x in (-1, 0, 0.5, 1.5, 2)] == [0, 1, 1, 3, 3]
    # half-to-even at code level: round(2.5) = 2 (not 3) with s = 1, z = 0
    assert oracle.encode(2.5, 1.0, 0.0, 4) == 2
    assert oracle.encode(3.5, 1.0, 0.0, 4) == 4


def test_hand_worked_4bit_group():
    # min 0, max 15 -> s = 1, z = 0, codes = values; 7.5 rounds to 8 (even)
    s, z = oracle.quant_params(0.0, 15.0, 4)
    assert (s, z) == (1.0, 0.0)
    assert [oracle.encode(x, s, z, 4) for x in (0, 7.5, 8.5, 15, 16, -3)] == [0, 8, 8, 15, 15, 0]
    # min -3, max 27 -> s = 30/15 = 2, z = round(1.5) = 2 (half to even)
    s, z = oracle.quant_params(-3.0, 27.0, 4)
    assert (s, z) == (2.0, 2.0)


def test_zero_point_is_not_clamped_to_code_range():
    # all-positive group: z = round(-min/s) is negative and kept as such
    s, z = oracle.quant_params(10.0, 13.0, 2)
    assert s == 1.0 and z == -10.0
    assert [oracle.encode(x, s, z, 2) for x in (10, 11, 12, 13)] == [0, 1, 2, 3]


def test_zero_zero_point_is_positive_zero():
    for mn, mx in ((0.0, 3.0), (-0.0, 3.0), (-0.0, -0.0), (0.0, 0.0), (-0.4, 2.6)):
        s, z = oracle.quant_params(mn, mx, 2)
        assert z == 0 and not np.signbit(z), (mn, mx, z)


def test_scale_floor_and_constant_group():
    for c in (0.0, 1.0, -3.25, 1000.0, 6.1e-5):
        s, z = oracle.quant_params(c, c, 2)
        assert s == np.float32(1e-8)
        assert oracle.encode(c, s, z, 2) == 0
        G, d = 4, 8
        s_, z_, codes = oracle.quantize_k_group(np.full((G, d), c, np.float32), 4)
        assert np.all(codes == 0)
        xhat = (codes.astype(np.float64) - z_.astype(np.float64)) * s_.astype(np.float64)
        # -z*s recovers c to within half a step plus fp32 rounding of z and s
        assert np.all(np.abs(xhat - c) <= 0.5e-8 + 2.0 ** -22 * abs(c))


@pytest.mark.parametrize("bits", [2, 4])
def test_grid_exact_inputs_reconstruct_exactly(bits):
    """Closed form: x = (code - z) * 2^-k with codes spanning 0..2^b-1 must give
    back exactly that s, z, those codes and x_hat == x."""
    rng = np.random.default_rng(bits)
    qmax = (1 << bits) - 1
    for trial in range(50):
        G, d = 32, 128
        k = int(rng.integers(-6, 12))
        s_true = np.float32(2.0 ** -k)
        z_true = rng.integers(0, qmax + 1, size=d)
        codes = rng.integers(0, qmax + 1, size=(G, d))
        codes[0] = 0
        codes[1] = qmax
        x = ((codes - z_true) * float(s_true)).astype(np.float32)
        s, z, got = oracle.quantize_k_group(x, bits)
        assert np.all(s == s_true) and np.all(z == z_true)
        assert np.array_equal(got, codes)
        # values per token: groups of G channels along the row
        xv = x.T.copy()  # [d][G] -> rows of G, each row one "token"
        for t in range(4):
            sv, zv, cv = oracle.quantize_v_token(xv[t], 32, bits)
            assert sv[0] == s_true and zv[0] == z_true[t]
            assert np.array_equal(cv, codes[:, t])


def _xhat(codes, s, z):
    return (codes.astype(np.float64) - z.astype(np.float64)) * s.astype(np.float64)


@pytest.mark.parametrize("bits", [2, 4])
def test_reconstruction_error_at_most_half_a_step(bits):
    rng = np.random.default_rng(10 + bits)
    cases = [
        rng.standard_normal((32, 128)),
        rng.standard_normal((32, 128)) * np.where(rng.random(128) < 0.05, 100.0, 1.0),
        np.round(rng.standard_normal((32, 128)) * 4) / 2,       # many exact ties
        rng.standard_normal((32, 128)) * 1e-3 + 100.0,          # narrow, far from 0
        rng.uniform(-60000, 60000, (32, 128)),                  # fp16 range
    ]
    for x in cases:
        x = x.astype(np.float16).astype(np.float32)
        s, z, codes = oracle.quantize_k_group(x, bits)
        err = np.abs(x - _xhat(codes, s[None, :], z[None, :]))
        slop = 2.0 ** -22 * np.maximum(np.abs(x), np.max(np.abs(x), axis=0)[None, :])
        assert np.all(err <= s[None, :] / 2 + slop)


@pytest.mark.parametrize("bits", [2, 4])
def test_codes_are_nearest_grid_point_brute_force(bits):
    """q must minimise |x - (k - z) s| over all 2^b codes k (fp64 search);
    exact ties and fp32 rounding of x/s allow only a 2^-22 |x| slack."""
    rng = np.random.default_rng(20 + bits)
    for trial in range(300):
        G = 4
        x = (rng.standard_normal((G, 8)) * rng.choice([0.01, 1, 30])).astype(np.float16)
        x = x.astype(np.float32)
        s, z, codes = oracle.quantize_k_group(x, bits)
        cand = np.arange(1 << bits, dtype=np.float64)
        for t in range(G):
            for c in range(8):
                errs = np.abs(x[t, c] - (cand - float(z[c])) * float(s[c]))
                mine = errs[codes[t, c]]
                assert mine <= errs.min() + 2.0 ** -22 * abs(float(x[t, c])) + 1e-30


def test_outlier_channel_does_not_inflate_other_channels():
    """Per-channel keys: one x100 channel changes only its own scale
    ("Quantize along the axis that hides the outliers")."""
    rng = np.random.default_rng(3)
    x = rng.standard_normal((32, 128)).astype(np.float16).astype(np.float32)
    s0, z0, c0 = oracle.quantize_k_group(x, 2)
    y = x.copy()
    y[:, 17] *= 100
    s1, z1, c1 = oracle.quantize_k_group(y, 2)
    other = np.arange(128) != 17
    assert np.array_equal(s0[other], s1[other]) and np.array_equal(c0[:, other], c1[:, other])
    assert s1[17] > 50 * s0[17]


def test_page_int4_pseudocode_per_token_special_case():
    """b = 4 with G = d per token is the page's int4 routine ("KV Cache INT4
    Quantization ...", section 2) evaluated in fp32; it rounds x/scale + zero
    instead of round(x/scale) + zero, which may differ only where x/scale is
    within float rounding of a half-integer."""
    rng = np.random.default_rng(4)
    x = (rng.standard_normal((64, 128)) * 3).astype(np.float16).astype(np.float32)
    mn = x.min(axis=-1, keepdims=True)
    mx = x.max(axis=-1, keepdims=True)
    scale = np.maximum((mx - mn) / np.float32(15.0), np.float32(1e-8)).astype(np.float32)
    zero = np.round(-mn / scale).astype(np.float32)
    ratio = (x / scale).astype(np.float32)
    page_q = np.clip(np.round(ratio + zero), 0, 15).astype(np.uint8)
    ours = np.stack([oracle.quantize_v_token(x[t], 128, 4)[2] for t in range(64)])
    s_ours = np.stack([oracle.quantize_v_token(x[t], 128, 4)[0] for t in range(64)])
    assert np.array_equal(s_ours, scale)
    diff = ours != page_q
    frac = np.abs(ratio - np.floor(ratio) - 0.5)
    assert np.all(frac[diff] < 1e-5)
    assert diff.mean() < 1e-3


def test_packing_is_lsb_first_along_channels():
    assert oracle.pack_row(np.array([1, 2, 3, 0, 3, 3, 3, 3], np.uint8), 2).tolist() == [57, 255]
    assert oracle.pack_row(np.array([5, 10, 15, 0], np.uint8), 4).tolist() == [165, 15]
    rng = np.random.default_rng(5)
    for bits in (2, 4):
        codes = rng.integers(0, 1 << bits, 128).astype(np.uint8)
        assert np.array_equal(oracle.unpack_row(oracle.pack_row(codes, bits), 128, bits), codes)


# ------------------------------------------------------ cache bookkeeping ---

def _rand_kv(rng, P, T, d, scale=1.0):
    k = (rng.standard_normal((P, T, d)) * scale).astype(np.float16)
    v = (rng.standard_normal((P, T, d)) * scale).astype(np.float16)
    return k, v


@pytest.mark.parametrize("T,R,exp_nq,exp_r", [
    (288, 32, 256, 32),        # tiny workload: 256 quantised + full 32-token residual
    (32768, 128, 32640, 128),
    (1048576, 128, 1048448, 128),
    (1, 32, 0, 1), (32, 32, 0, 32), (33, 32, 32, 1), (65, 32, 64, 1), (64, 32, 32, 32),
])
def test_prefill_split_closed_form(T, R, exp_nq, exp_r):
    # r' = ((T - 1) mod R) + 1 residual tokens, the rest quantised
    assert (T - (((T - 1) % R) + 1), ((T - 1) % R) + 1) == (exp_nq, exp_r)
    if T <= 4096:
        c = oracle.OracleCache(1, 16, 2, 16 if R % 16 == 0 else R, R, 4096)
        rng = np.random.default_rng(T)
        k, v = _rand_kv(rng, 1, T, 16)
        assert c.prefill(k, v) == 0
        assert (c.n_quant, c.n_resid) == (exp_nq, exp_r)


def _state(c):
    return [a.copy() for a in (c.kc, c.vc, c.ks, c.kz, c.vs, c.vz)] + \
           [c.kr[:, :c.n_sink].copy(), c.vr[:, :c.n_sink].copy(),
            c.kres[:, :c.n_resid].copy(), c.vres[:, :c.n_resid].copy()]


@pytest.mark.parametrize("bits,G,R", [(2, 32, 32), (4, 16, 64), (2, 16, 16)])
def test_prefill_equals_prefill_then_appends(bits, G, R):
    rng = np.random.default_rng(bits * 100 + G)
    P, d, T, T0 = 3, 64, 200, 37
    k, v = _rand_kv(rng, P, T, d, 3.0)
    a = oracle.OracleCache(P, d, bits, G, R, 256)
    b = oracle.OracleCache(P, d, bits, G, R, 256)
    assert a.prefill(k, v) == 0
    assert b.prefill(k[:, :T0], v[:, :T0]) == 0
    for t in range(T0, T):
        assert b.append(k[:, t], v[:, t]) == 0
    assert (a.n_quant, a.n_resid) == (b.n_quant, b.n_resid)
    for x, y in zip(_state(a), _state(b)):
        assert np.array_equal(x, y)
    # chunked prefill (two chunks) too
    c = oracle.OracleCache(P, d, bits, G, R, 256)
    assert c.prefill(k[:, :T0], v[:, :T0]) == 0 and c.prefill(k[:, T0:], v[:, T0:]) == 0
    for x, y in zip(_state(a), _state(c)):
        assert np.array_equal(x, y)


def test_state_after_appends_follows_lazy_flush():
    R, G = 32, 16
    c = oracle.OracleCache(1, 16, 2, G, R, 1024)
    rng = np.random.default_rng(9)
    for t in range(1, 200):
        k, v = _rand_kv(rng, 1, 1, 16)
        assert c.append(k[:, 0], v[:, 0]) == 0
        # closed form: after t tokens, r = ((t-1) mod R) + 1
        assert c.n_resid == ((t - 1) % R) + 1
        assert c.n_quant == t - c.n_resid


def test_groups_depend_only_on_their_own_tokens():
    rng = np.random.default_rng(11)
    P, d, G, R, T = 1, 32, 16, 32, 161
    k, v = _rand_kv(rng, P, T, d)
    a = oracle.OracleCache(P, d, 2, G, R, 256)
    a.prefill(k, v)
    k2, v2 = k.copy(), v.copy()
    k2[0, 40] *= 7       # token 40 lies in key group 2 (tokens 32..47)
    v2[0, 40] *= 7
    b = oracle.OracleCache(P, d, 2, G, R, 256)
    b.prefill(k2, v2)
    rb = d * 2 // 8
    for grp in range(a.n_quant // G):
        same = np.array_equal(a.ks[0, grp], b.ks[0, grp]) and \
            np.array_equal(a.kc[0, grp * G:(grp + 1) * G], b.kc[0, grp * G:(grp + 1) * G])
        assert same == (grp != 2)
    for t in range(a.n_quant):
        same = np.array_equal(a.vc[0, t], b.vc[0, t]) and np.array_equal(a.vs[0, t], b.vs[0, t])
        assert same == (t != 40)
    assert rb == 8


def test_value_codes_do_not_depend_on_flush_timing():
    """Values are per token: a token's codes are the same whether it was
    quantised by a prefill or by a later residual flush."""
    rng = np.random.default_rng(12)
    P, d, G, R = 2, 64, 32, 64
    k, v = _rand_kv(rng, P, 300, d)
    a = oracle.OracleCache(P, d, 2, G, R, 512)
    a.prefill(k, v)
    for t in range(a.n_quant):
        s, z, codes = oracle.quantize_v_token(v[1, t].astype(np.float32), G, 2)
        assert np.array_equal(a.vs[1, t], s) and np.array_equal(a.vz[1, t], z)
        assert np.array_equal(a.vc[1, t], oracle.pack_row(codes, 2))


def test_capacity_and_empty():
    c = oracle.OracleCache(1, 16, 2, 16, 32, 64)
    rng = np.random.default_rng(13)
    k, v = _rand_kv(rng, 1, 97, 16)
    assert c.prefill(k, v) == -3                        # would need 96 > 64
    assert (c.n_quant, c.n_resid) == (0, 0)
    with pytest.raises(RuntimeError):
        c.attention(np.zeros((1, 16), np.float16), 1)
    assert c.prefill(k[:, :96], v[:, :96]) == 0         # 64 quantised + 32 residual
    assert (c.n_quant, c.n_resid) == (64, 32)
    assert c.append(k[:, 96], v[:, 96]) == -3           # flush would overflow
    assert (c.n_quant, c.n_resid) == (64, 32)
    assert c.prefill(k[:, :0], v[:, :0]) == 0           # empty input is a no-op


# -------------------------------------------------------------- attention ---

@pytest.mark.parametrize("bits,G,R,T,g", [(2, 32, 32, 288, 4), (4, 64, 128, 300, 2),
                                          (2, 16, 32, 70, 8)])
def test_attention_matches_torch_sdpa_fp64(bits, G, R, T, g):
    rng = np.random.default_rng(T + g)
    B, Hkv, d = 2, 2, 64 if G <= 64 else 128
    P = B * Hkv
    k, v = _rand_kv(rng, P, T, d, 2.0)
    c = oracle.OracleCache(P, d, bits, G, R, 512)
    c.prefill(k, v)
    q = rng.standard_normal((P * g, d)).astype(np.float16)
    tau = 1.0 / math.sqrt(d)
    out = c.attention(q, g, tau)
    for p in range(P):
        K, V = c.dequant_k(p), c.dequant_v(p)
        qs = q[p * g:(p + 1) * g].astype(np.float64)
        ref = torch.nn.functional.scaled_dot_product_attention(
            torch.from_numpy(qs)[:, None, :], torch.from_numpy(K)[None].expand(g, -1, -1),
            torch.from_numpy(V)[None].expand(g, -1, -1), scale=tau)[:, 0].numpy()
        np.testing.assert_allclose(out[p * g:(p + 1) * g], ref, rtol=1e-12, atol=1e-12)


def test_attention_uses_kv_head_hq_div_g():
    """Query head h_q reads kv head h_q // g: identical queries in one group
    give identical rows; the same query in another group sees other keys."""
    rng = np.random.default_rng(21)
    P, d, g = 3, 32, 4
    k, v = _rand_kv(rng, P, 64, d)
    c = oracle.OracleCache(P, d, 2, 16, 32, 64)
    c.prefill(k, v)
    q1 = rng.standard_normal(d).astype(np.float16)
    q = np.tile(q1, (P * g, 1))
    out = c.attention(q, g)
    for p in range(P):
        K, V = c.dequant_k(p), c.dequant_v(p)
        s = K @ q1.astype(np.float64) / math.sqrt(d)
        w = np.exp(s - s.max())
        ref = w @ V / w.sum()
        for i in range(g):
            np.testing.assert_allclose(out[p * g + i], ref, rtol=1e-12, atol=1e-13)


def test_dequant_reads_residual_exactly():
    rng = np.random.default_rng(22)
    k, v = _rand_kv(rng, 1, 50, 32)
    c = oracle.OracleCache(1, 32, 2, 16, 32, 64)
    c.prefill(k, v)          # 32 quantised + 18 residual
    assert np.array_equal(c.dequant_k(0)[32:], k[0, 32:].astype(np.float64))
    assert np.array_equal(c.dequant_v(0)[32:], v[0, 32:].astype(np.float64))


def _grid_exact_cache_inputs(rng, P, T, d, bits, G):
    """fp16 K, V [P][T][d] that lie on a quantisation grid by construction.

    Keys: every (G-token group, channel) is (code - z) * 2^-e with its own e
    and integer z in [0, 2^b - 1] and codes that include 0 and 2^b - 1 ("4.4
    KV Cache quantization", section 3.1: keys per channel over G tokens).
    Values: every (token, run of G channels) likewise ("Value per-token").
    For such a group min = -z s and max = (2^b - 1 - z) s, so the quantiser
    of "KV Cache INT4 Quantization ...", section 2 recovers s, z and the codes
    exactly, and (code - z) s gives back the input bit for bit."""
    qmax = (1 << bits) - 1

    def grid(n_groups, n_members):
        e = rng.integers(-5, 5, size=(n_groups, 1))
        z = rng.integers(0, qmax + 1, size=(n_groups, 1))
        codes = rng.integers(0, qmax + 1, size=(n_groups, n_members))
        lo, hi = rng.choice(n_members, 2, replace=False, shuffle=False) if n_members > 1 else (0, 0)
        codes[:, lo] = 0
        codes[:, hi] = qmax
        return ((codes - z) * np.exp2(-e.astype(np.float64))).astype(np.float16)

    K = np.empty((P, T, d), np.float16)
    V = np.empty((P, T, d), np.float16)
    ng = T // G
    for p in range(P):
        # keys: [groups][channel] each spanning G tokens
        kg = grid(ng * d, G).reshape(ng, d, G).transpose(0, 2, 1).reshape(ng * G, d)
        K[p, :ng * G] = kg
        K[p, ng * G:] = rng.standard_normal((T - ng * G, d))
        V[p] = grid(T * (d // G), G).reshape(T, d)
    assert np.all(np.isfinite(K)) and np.all(np.isfinite(V))
    return K, V


@pytest.mark.parametrize("bits,G,R", [(2, 32, 64), (4, 64, 128), (2, 16, 32), (4, 128, 128)])
def test_dequant_of_quantised_tokens_returns_grid_exact_inputs(bits, G, R):
    """Cache-level closed form: after a prefill of grid-exact tokens the
    oracle's dequantised history equals the input tokens exactly, for keys
    (per-channel groups of G tokens) and values (per-token groups of G
    channels).  A wrong group index (z[c % G] for z[c / G], a key group of
    u % G, a transposed scale table) breaks the equality."""
    rng = np.random.default_rng(1000 + bits * 10 + G)
    P, d = 3, 128
    T = 3 * R + 17                       # several flushes of R tokens + residual
    K, V = _grid_exact_cache_inputs(rng, P, T, d, bits, G)
    c = oracle.OracleCache(P, d, bits, G, R, 8 * R)
    assert c.prefill(K, V) == 0
    nq = c.n_quant
    assert nq == 3 * R and c.n_resid == 17
    for p in range(P):
        assert np.array_equal(c.dequant_k(p), K[p].astype(np.float64))
        assert np.array_equal(c.dequant_v(p), V[p].astype(np.float64))


@pytest.mark.parametrize("bits,G", [(2, 32), (4, 64), (2, 16), (4, 32)])
def test_dequant_error_at_most_half_step_of_each_group(bits, G):
    """On random, outlier-laden fp16 tokens, every dequantised history element
    lies within half a quantisation step of the ORIGINAL token, where the step
    (max - min) / (2^b - 1) of its group is computed here from the original
    tokens (keys: the channel over its G-token group; values: the token over
    its G-channel run).  The 1e-8 floor and fp32 rounding of s and z add at
    most 2^-21 relative slack."""
    rng = np.random.default_rng(2000 + bits * 10 + G)
    P, d, R = 2, 128, 2 * G
    T = 5 * R + 3
    K = rng.standard_normal((P, T, d)) * np.where(rng.random(d) < 0.03, 60.0, 1.0)
    V = rng.standard_normal((P, T, d)) * np.where(rng.random((P, T, 1)) < 0.02, 300.0, 1.0)
    K[0, :G] = 2.5                                   # a constant key group
    V[1, 7] = -1.0                                   # a constant value token
    K, V = K.astype(np.float16), V.astype(np.float16)
    c = oracle.OracleCache(P, d, bits, G, R, 8 * R)
    assert c.prefill(K, V) == 0
    nq = c.n_quant
    qmax = (1 << bits) - 1
    for p in range(P):
        k = K[p, :nq].astype(np.float64).reshape(nq // G, G, d)
        step_k = (k.max(axis=1) - k.min(axis=1)) / qmax                  # [groups][d]
        step_k = np.repeat(np.maximum(step_k, 1e-8), G, axis=0)          # [nq][d]
        v = V[p, :nq].astype(np.float64).reshape(nq, d // G, G)
        step_v = np.maximum((v.max(axis=2) - v.min(axis=2)) / qmax, 1e-8)
        step_v = np.repeat(step_v, G, axis=1)                            # [nq][d]
        for x, xhat, step in ((K[p, :nq], c.dequant_k(p)[:nq], step_k),
                              (V[p, :nq], c.dequant_v(p)[:nq], step_v)):
            x = x.astype(np.float64)
            slack = 2.0 ** -21 * (np.abs(x) + step * qmax)
            assert np.all(np.abs(xhat - x) <= step / 2 + slack)


def test_single_token_returns_its_value():
    rng = np.random.default_rng(23)
    k, v = _rand_kv(rng, 1, 1, 64)
    c = oracle.OracleCache(1, 64, 2, 32, 32, 32)
    c.prefill(k, v)
    q = rng.standard_normal((4, 64)).astype(np.float16)
    out = c.attention(q, 4)
    for i in range(4):
        assert np.array_equal(out[i], v[0, 0].astype(np.float64))


def test_equal_scores_give_mean_of_values():
    rng = np.random.default_rng(24)
    k, v = _rand_kv(rng, 2, 200, 64)
    c = oracle.OracleCache(2, 64, 4, 32, 64, 256)
    c.prefill(k, v)
    out = c.attention(np.zeros((2, 64), np.float16), 1)
    for p in range(2):
        np.testing.assert_allclose(out[p], c.dequant_v(p).mean(axis=0), rtol=1e-12, atol=1e-13)


def test_split_and_combine_equals_one_pass():
    """Flash-decoding merge: o = sum_i e^(m_i-M) o_i / sum_i e^(m_i-M) l_i."""
    rng = np.random.default_rng(25)
    k, v = _rand_kv(rng, 1, 500, 64, 3.0)
    c = oracle.OracleCache(1, 64, 2, 32, 64, 512)
    c.prefill(k, v)
    q = rng.standard_normal((4, 64)).astype(np.float16)
    full = c.attention(q, 4)
    n = c.n_quant + c.n_resid
    for row in range(4):
        cuts = [0, 17, 130, 131, 400, n]
        parts = [c.attention_partial(q, 4, row, a, b) for a, b in zip(cuts[:-1], cuts[1:])]
        parts.append(c.attention_partial(q, 4, row, n, n))      # an empty split
        M = max(p[0] for p in parts)
        L = sum(p[1] * math.exp(p[0] - M) for p in parts if p[1] > 0)
        o = sum(p[2] * math.exp(p[0] - M) for p in parts if p[1] > 0) / L
        np.testing.assert_allclose(o, full[row], rtol=1e-12, atol=1e-12)


# ------------------------------------------------------------ sink tokens ---
# "09 -- KV Cache Quantization", "Anti-patterns": the first tokens of a
# sequence absorb large attention scores and are kept unquantised
# (preserve-first-N).

@pytest.mark.parametrize("Ns", [1, 4, 37, 64])
def test_sink_prefill_equals_appends_and_chunks(Ns):
    rng = np.random.default_rng(3000 + Ns)
    P, d, G, R, T = 2, 64, 16, 32, 230
    k, v = _rand_kv(rng, P, T, d, 3.0)
    a = oracle.OracleCache(P, d, 2, G, R, 256, Ns=Ns)
    b = oracle.OracleCache(P, d, 2, G, R, 256, Ns=Ns)
    c = oracle.OracleCache(P, d, 2, G, R, 256, Ns=Ns)
    assert a.prefill(k, v) == 0
    assert b.prefill(k[:, :3], v[:, :3]) == 0
    for t in range(3, T):
        assert b.append(k[:, t], v[:, t]) == 0
    cut = Ns // 2 + 1
    assert c.prefill(k[:, :cut], v[:, :cut]) == 0 and c.prefill(k[:, cut:], v[:, cut:]) == 0
    for other in (b, c):
        assert (a.n_sink, a.n_quant, a.n_resid) == (other.n_sink, other.n_quant, other.n_resid)
        for x, y in zip(_state(a), _state(other)):
            assert np.array_equal(x, y)


@pytest.mark.parametrize("Ns", [3, 32, 100])
def test_sink_keeps_first_tokens_exact_and_the_rest_is_plain_kivi(Ns):
    """The first Ns tokens are stored and dequantised exactly; everything
    after them is bit for bit what a cache without sinks makes of the
    remaining tokens (key groups count from the first token after the sink)."""
    rng = np.random.default_rng(4000 + Ns)
    P, d, G, R, T = 3, 64, 32, 64, 300
    k, v = _rand_kv(rng, P, T, d, 2.0)
    s = oracle.OracleCache(P, d, 4, G, R, 512, Ns=Ns)
    plain = oracle.OracleCache(P, d, 4, G, R, 512)
    assert s.prefill(k, v) == 0 and plain.prefill(k[:, Ns:], v[:, Ns:]) == 0
    assert s.n_sink == Ns and (s.n_quant, s.n_resid) == (plain.n_quant, plain.n_resid)
    for x, y in zip(_state(s)[:6] + _state(s)[8:], _state(plain)[:6] + _state(plain)[8:]):
        assert np.array_equal(x, y)
    for p in range(P):
        K, V = s.dequant_k(p), s.dequant_v(p)
        assert np.array_equal(K[:Ns], k[p, :Ns].astype(np.float64))
        assert np.array_equal(V[:Ns], v[p, :Ns].astype(np.float64))
        assert np.array_equal(K[Ns:], plain.dequant_k(p))
        assert np.array_equal(V[Ns:], plain.dequant_v(p))


def test_sink_covering_everything_is_exact_attention():
    """Ns >= T: nothing is quantised, so the oracle's attention is plain fp64
    softmax attention over the input tokens (torch SDPA in float64)."""
    rng = np.random.default_rng(5000)
    P, d, g, T = 2, 64, 4, 50
    k, v = _rand_kv(rng, P, T, d, 3.0)
    c = oracle.OracleCache(P, d, 2, 16, 32, 64, Ns=64)
    assert c.prefill(k, v) == 0
    assert (c.n_sink, c.n_quant, c.n_resid) == (T, 0, 0)
    q = rng.standard_normal((P * g, d)).astype(np.float16)
    tau = 1.0 / math.sqrt(d)
    out = c.attention(q, g, tau)
    for p in range(P):
        K = torch.from_numpy(k[p].astype(np.float64))
        V = torch.from_numpy(v[p].astype(np.float64))
        qs = torch.from_numpy(q[p * g:(p + 1) * g].astype(np.float64))
        ref = torch.nn.functional.scaled_dot_product_attention(
            qs[:, None, :], K[None].expand(g, -1, -1), V[None].expand(g, -1, -1),
            scale=tau)[:, 0].numpy()
        np.testing.assert_allclose(out[p * g:(p + 1) * g], ref, rtol=1e-12, atol=1e-12)


def test_sink_capacity_error_leaves_state_unchanged():
    rng = np.random.default_rng(6000)
    k, v = _rand_kv(rng, 1, 200, 16)
    c = oracle.OracleCache(1, 16, 2, 16, 32, 64, Ns=8)
    assert c.prefill(k[:, :5], v[:, :5]) == 0
    before = _state(c)
    assert c.prefill(k[:, 5:200], v[:, 5:200]) == -3     # 3 sink + 192 -> 160 quantised
    assert (c.n_sink, c.n_quant, c.n_resid) == (5, 0, 0)
    for x, y in zip(before, _state(c)):
        assert np.array_equal(x, y)
    assert c.prefill(k[:, 5:104], v[:, 5:104]) == 0     # 3 sink + 96 -> 64 + 32
    assert (c.n_sink, c.n_quant, c.n_resid) == (8, 64, 32)


# ----------------------------------------------- packed history layout ---
# The storage format of the CUDA library (the pages fix only the grouping
# axes and the codes per byte); pinned here by hand-worked bytes.

@pytest.mark.parametrize("G,bits", [(16, 2), (16, 4), (32, 2), (32, 4), (64, 2), (64, 4),
                                    (128, 2), (128, 4)])
def test_value_position_is_a_permutation(G, bits):
    pos = [oracle.value_position(c, 128, G, bits) for c in range(128)]
    assert sorted(pos) == list(range(128))
    if G == 128 or (G == 16 and bits == 2):
        assert pos == list(range(128))          # natural order


def test_value_position_hand_worked():
    # d = 128, G = 32: runs of G/8 = 4 channels; channel c of group j at
    # u = c mod 32 sits at 16 (u / 4) + 4 j + (u mod 4)
    assert [oracle.value_position(c, 128, 32, 2) for c in (0, 3, 4, 31, 32, 37, 127)] == \
        [0, 3, 16, 115, 4, 21, 127]
    # d = 32, G = 16, 4-bit: runs of 2 channels, 4 (d/8) positions per run index
    assert [oracle.value_position(c, 32, 16, 4) for c in (0, 1, 2, 16, 17, 18, 31)] == \
        [0, 1, 4, 2, 3, 6, 31]


def test_record_bytes_per_token_match_the_byte_budget():
    # algorithmic bytes per quantised token of one pair (codes + fp32 metadata):
    # 128 B (2-bit, G 32), 160 B (4-bit, G 64), 192 B (4-bit, G 32)
    assert oracle.record_bytes(128, 32, 2) == 32 * 128
    assert oracle.record_bytes(128, 64, 4) == 64 * 160
    assert oracle.record_bytes(128, 32, 4) == 32 * 192


def test_export_history_hand_worked_record():
    """d = 32, G = 16, 4-bit, one key group: every value token holds v[c] =
    c mod 16 (each 16-channel group spans 0..15, so s = 1, z = 0 and the codes
    are the values); keys hold k[t][c] = t (per-channel group over tokens
    0..15: s = 1, z = 0, codes = t)."""
    d, G, bits, T = 32, 16, 4, 16 + 3
    k = np.zeros((1, T, d), np.float16)
    v = np.zeros((1, T, d), np.float16)
    for t in range(T):
        k[0, t, :] = t % 16
        v[0, t, :] = np.arange(d) % 16
    c = oracle.OracleCache(1, d, bits, G, 16, 64)
    assert c.prefill(k, v) == 0 and c.n_quant == 16
    rec = c.export_history(0)
    assert rec.shape == (1, 8 * d + G * (2 * 16 + 8 * 2))
    r = rec[0]
    f = r.view(np.float32)
    assert np.all(f[:d] == 1.0) and np.all(f[d:2 * d] == 0.0)          # Ks, Kz
    base = 8 * d                                                        # the sub-slice
    # key row t: 32 codes = t, two per byte, low nibble first
    for t in range(16):
        assert np.all(r[base + 16 * t: base + 16 * t + 16] == t * 0x11)
    # value row: stored order puts channel pairs (0,1), (16,17), (2,3), (18,19), ...
    vrow = bytes([0x10, 0x10, 0x32, 0x32, 0x54, 0x54, 0x76, 0x76,
                  0x98, 0x98, 0xBA, 0xBA, 0xDC, 0xDC, 0xFE, 0xFE])
    for t in range(16):
        assert bytes(r[base + 256 + 16 * t: base + 256 + 16 * t + 16]) == vrow
    vs = r[base + 512: base + 512 + 16 * 2 * 4].view(np.float32)
    vz = r[base + 640: base + 640 + 16 * 2 * 4].view(np.float32)
    assert np.all(vs == 1.0) and np.all(vz == 0.0)


# ------------------------------------------------- fp16 scale / zero point ---
# "09 -- KV Cache Quantization", "KIVI -- the reference paper": per-channel
# scale and zero in fp16.  Range-guarded form: s rounded UP to binary16, at
# least 2^-24 and |min| / 2048, so that z is an exact binary16 integer.

def _f16_floor_bounds(mn, mx, bits):
    qmax = (1 << bits) - 1
    return max(float(np.float32(np.float32(mx) - np.float32(mn)) / np.float32(qmax)),
               float(np.float32(abs(np.float32(mn)) / np.float32(2048.0))), 2.0 ** -24)


@pytest.mark.parametrize("bits", [2, 4])
def test_f16_scale_is_smallest_binary16_above_the_bounds(bits):
    rng = np.random.default_rng(7000 + bits)
    cases = [(-1.0, 2.0), (0.0, 0.0), (100.0, 100.01), (-60000.0, 60000.0), (1e-6, 2e-6),
             (-3.0, -2.9), (5e-5, 7e-5)]
    cases += [tuple(sorted(rng.standard_normal(2) * rng.choice([1e-4, 1, 300])))
              for _ in range(300)]
    for mn, mx in cases:
        mn, mx = float(np.float16(mn)), float(np.float16(mx))
        s, z = oracle.quant_params_f16(mn, mx, bits)
        bound = _f16_floor_bounds(mn, mx, bits)
        assert float(np.float16(s)) == float(s)                   # a binary16 value
        assert float(s) >= bound
        below = np.nextafter(np.float16(s), np.float16(0))        # the next smaller one
        assert float(below) < bound
        assert abs(float(z)) <= 2048 and float(z) == round(float(z))
        assert float(z) == float(np.rint(np.float32(-np.float32(mn) / np.float32(s)))) + 0.0


def test_f16_scale_hand_worked():
    assert oracle.quant_params_f16(-1.0, 2.0, 2) == (1.0, 1.0)             # as fp32
    # narrow group far from zero: the guard |min| / 2048 = 100 / 2048 sets s
    s, z = oracle.quant_params_f16(100.0, 100.0078125, 2)
    assert s == np.float32(100.0 / 2048) and z == -2048.0
    s, z = oracle.quant_params_f16(0.0, 0.0, 4)                              # floor 2^-24
    assert s == np.float32(2.0 ** -24) and z == 0.0 and not np.signbit(z)


@pytest.mark.parametrize("bits,G", [(2, 32), (4, 64), (4, 32)])
def test_f16_meta_cache_dequant_bounds_and_grid(bits, G):
    rng = np.random.default_rng(8000 + bits + G)
    P, d, R = 2, 128, 2 * G
    # grid-exact tokens reproduce exactly (no guard binds: |z| <= 15)
    K, V = _grid_exact_cache_inputs(rng, P, 3 * R + 5, d, bits, G)
    c = oracle.OracleCache(P, d, bits, G, R, 8 * R, meta=oracle.META_FP16)
    assert c.prefill(K, V) == 0
    for p in range(P):
        assert np.array_equal(c.dequant_k(p), K[p].astype(np.float64))
        assert np.array_equal(c.dequant_v(p), V[p].astype(np.float64))
    # random outlier-laden tokens: within half of the fp16 step of the original
    T = 5 * R + 3
    K = (rng.standard_normal((P, T, d)) * np.where(rng.random(d) < 0.03, 60.0, 1.0) + 3.0)
    V = rng.standard_normal((P, T, d)) * np.where(rng.random((P, T, 1)) < 0.02, 300.0, 1.0)
    K, V = K.astype(np.float16), V.astype(np.float16)
    c = oracle.OracleCache(P, d, bits, G, R, 8 * R, meta=oracle.META_FP16)
    assert c.prefill(K, V) == 0
    nq = c.n_quant
    for p in range(P):
        k = K[p, :nq].astype(np.float64).reshape(nq // G, G, d)
        v = V[p, :nq].astype(np.float64).reshape(nq, d // G, G)
        for x, xhat, lo, hi, rep in ((K[p, :nq], c.dequant_k(p)[:nq], k.min(axis=1),
                                      k.max(axis=1), lambda a: np.repeat(a, G, axis=0)),
                                     (V[p, :nq], c.dequant_v(p)[:nq], v.min(axis=2),
                                      v.max(axis=2), lambda a: np.repeat(a, G, axis=1))):
            step = np.vectorize(lambda a, b: float(np.float16(
                _f16_floor_bounds(a, b, bits))))(lo, hi)
            step = np.maximum(step, np.vectorize(lambda a, b: _f16_floor_bounds(a, b, bits))(lo, hi))
            step = rep(step) * (1 + 2.0 ** -10)        # rounded up to binary16
            x = x.astype(np.float64)
            assert np.all(np.abs(xhat - x) <= step / 2 + 2.0 ** -20 * np.abs(x))


def test_f16_meta_record_hand_worked():
    """The export_history record of the hand-worked case with fp16 metadata:
    Ks = 1.0 (0x3C00), Kz = +0, Vs = 1.0, Vz = +0 as binary16."""
    d, G, bits, T = 32, 16, 4, 19
    k = np.zeros((1, T, d), np.float16)
    v = np.zeros((1, T, d), np.float16)
    for t in range(T):
        k[0, t, :] = t % 16
        v[0, t, :] = np.arange(d) % 16
    c = oracle.OracleCache(1, d, bits, G, 16, 64, meta=oracle.META_FP16)
    assert c.prefill(k, v) == 0
    r = c.export_history(0)[0]
    assert r.shape == (4 * d + G * (2 * 16 + 4 * 2),)
    assert np.all(r[:2 * d].view(np.uint16) == 0x3C00) and np.all(r[2 * d:4 * d] == 0)
    base = 4 * d
    for t in range(16):
        assert np.all(r[base + 16 * t: base + 16 * t + 16] == t * 0x11)
    vs = r[base + 512: base + 512 + 16 * 2 * 2].view(np.uint16)
    vz = r[base + 576: base + 576 + 16 * 2 * 2].view(np.uint16)
    assert np.all(vs == 0x3C00) and np.all(vz == 0)


# ------------------------------------------------- residual flush policies ---
# "KIVI: ...", "The streaming complication": a completed key group is frozen
# as the window slides (GROUP) versus "4.4 KV Cache quantization", section 3.2:
# the window is quantised in one batch once it is full (WINDOW).

@pytest.mark.parametrize("G,R", [(16, 32), (32, 128), (16, 64)])
def test_group_flush_state_closed_form_and_appends(G, R):
    rng = np.random.default_rng(9000 + G + R)
    P, d = 2, 32
    c = oracle.OracleCache(P, d, 2, G, R, 1024, flush=oracle.FLUSH_GROUP)
    for t in range(1, 400):
        k, v = _rand_kv(rng, P, 1, d)
        assert c.append(k[:, 0], v[:, 0]) == 0
        # one token at a time: the window fills to R, then each arrival at a
        # full window quantises the oldest G tokens
        exp_r = t if t <= R else R - G + 1 + (t - R - 1) % G
        assert (c.n_quant, c.n_resid) == (t - exp_r, exp_r)
        assert c.n_quant % G == 0


@pytest.mark.parametrize("Ns", [0, 5])
def test_group_flush_prefill_equals_appends_and_chunks(Ns):
    rng = np.random.default_rng(9100 + Ns)
    P, d, G, R, T = 2, 64, 16, 64, 333
    k, v = _rand_kv(rng, P, T, d, 2.0)
    mk = lambda: oracle.OracleCache(P, d, 4, G, R, 512, Ns=Ns, flush=oracle.FLUSH_GROUP)
    a, b, c = mk(), mk(), mk()
    assert a.prefill(k, v) == 0
    for t in range(T):
        assert b.append(k[:, t], v[:, t]) == 0
    for x, y in ((0, 7), (7, 100), (100, 101), (101, T)):
        assert c.prefill(k[:, x:y], v[:, x:y]) == 0
    for o in (b, c):
        assert (a.n_sink, a.n_quant, a.n_resid) == (o.n_sink, o.n_quant, o.n_resid)
        for x, y in zip(_state(a), _state(o)):
            assert np.array_equal(x, y)


def test_group_flush_history_is_the_window_history():
    """Key groups depend only on their own G tokens and values only on their
    own token, so the two policies quantise every token they both quantised
    identically; they differ only in how many tokens are still fp16."""
    rng = np.random.default_rng(9200)
    P, d, G, R, T = 2, 64, 32, 128, 1000
    k, v = _rand_kv(rng, P, T, d, 2.0)
    w = oracle.OracleCache(P, d, 2, G, R, 1024)
    g = oracle.OracleCache(P, d, 2, G, R, 1024, flush=oracle.FLUSH_GROUP)
    assert w.prefill(k, v) == 0 and g.prefill(k, v) == 0
    assert (w.n_quant, w.n_resid) == (896, 104) and (g.n_quant, g.n_resid) == (896, 104)
    assert w.append(k[:, 0], v[:, 0]) == 0 and g.append(k[:, 0], v[:, 0]) == 0
    for _ in range(24):                         # fill both windows to 128 + a flush
        assert w.append(k[:, 1], v[:, 1]) == 0 and g.append(k[:, 1], v[:, 1]) == 0
    assert (w.n_quant, w.n_resid) == (1024, 1) and (g.n_quant, g.n_resid) == (928, 97)
    nq = g.n_quant
    for a, b in ((w.kc, g.kc), (w.vc, g.vc), (w.vs, g.vs), (w.vz, g.vz)):
        assert np.array_equal(a[:, :nq], b[:, :nq])
    for a, b in ((w.ks, g.ks), (w.kz, g.kz)):
        assert np.array_equal(a[:, :nq // G], b[:, :nq // G])
    # the group policy's window holds the 97 newest tokens exactly
    seq_k = np.concatenate([k, k[:, :1], np.repeat(k[:, 1:2], 24, axis=1)], axis=1)
    seq_v = np.concatenate([v, v[:, :1], np.repeat(v[:, 1:2], 24, axis=1)], axis=1)
    for p in range(P):
        assert np.array_equal(w.dequant_k(p)[:nq], g.dequant_k(p)[:nq])
        assert np.array_equal(g.dequant_k(p)[nq:], seq_k[p, nq:].astype(np.float64))
        assert np.array_equal(g.dequant_v(p)[nq:], seq_v[p, nq:].astype(np.float64))


# ------------------------------------------------------------------ FP8 KV ---
# "09 -- KV Cache Quantization", "The lazy default: FP8 KV" (E4M3 / E5M2);
# "4.4 KV Cache quantization", section 4.2 (FP8 still needs a scale; 1.0
# uncalibrated).

@pytest.mark.parametrize("fmt,dtype,maxv", [(1, torch.float8_e4m3fn, 448.0),
                                            (2, torch.float8_e5m2, 57344.0)])
def test_fp8_rounding_matches_torch_and_saturates(fmt, dtype, maxv):
    rng = np.random.default_rng(10000 + fmt)
    x = rng.standard_normal(50000) * rng.choice([1e-6, 1e-3, 1, 30, 300, 20000], 50000)
    x = x.astype(np.float32)
    inr = np.abs(x) < maxv
    ref = torch.from_numpy(x[inr]).to(dtype)
    got = np.array([oracle.fp8_round(v, fmt) for v in x[inr]])
    assert np.array_equal(got, ref.float().numpy().astype(np.float64))
    assert np.array_equal(np.array([oracle.fp8_bits(v, fmt) for v in got], np.uint8),
                          ref.view(torch.uint8).numpy())
    # out of range saturates to the largest finite value (no infinity, no NaN)
    for v in (maxv * 1.01, 1e9, -1e9):
        assert oracle.fp8_round(v, fmt) == np.sign(v) * maxv
    # every byte that is a finite value decodes to torch's value
    b = torch.arange(256, dtype=torch.uint8).view(dtype).float().numpy()
    for i in range(256):
        if np.isfinite(b[i]):
            assert oracle.fp8_value(i, fmt) == float(b[i])


@pytest.mark.parametrize("fmt", [1, 2])
def test_fp8_cache_dequant_is_scaled_fp8(fmt):
    rng = np.random.default_rng(11000 + fmt)
    P, d, R, T = 2, 64, 32, 200
    k, v = _rand_kv(rng, P, T, d, 3.0)
    c = oracle.OracleCache(P, d, 8, 32, R, 256, fp8=fmt, fp8_k_scale=0.25, fp8_v_scale=2.0)
    assert c.prefill(k, v) == 0 and (c.n_quant, c.n_resid) == (192, 8)
    for p in range(P):
        K, V = c.dequant_k(p), c.dequant_v(p)
        for t in (0, 57, 191):
            for ch in (0, 13, 63):
                xk = np.float32(np.float32(k[p, t, ch]) / np.float32(0.25))
                xv = np.float32(np.float32(v[p, t, ch]) / np.float32(2.0))
                assert K[t, ch] == float(torch.tensor(xk).to(
                    torch.float8_e4m3fn if fmt == 1 else torch.float8_e5m2).float()) * 0.25
                assert V[t, ch] == float(torch.tensor(xv).to(
                    torch.float8_e4m3fn if fmt == 1 else torch.float8_e5m2).float()) * 2.0
        assert np.array_equal(K[192:], k[p, 192:].astype(np.float64))    # residual exact
    rec = c.export_history(0)
    assert rec.shape == (6, 64 * d)
    assert np.array_equal(rec[1, :32 * d].reshape(32, d), c.kc[0, 32:64])
    assert np.array_equal(rec[1, 32 * d:].reshape(32, d), c.vc[0, 32:64])

"""Pins of the fp64 oracle to facts other than itself (CPU only).

Each test checks the oracle against a closed form, a textbook value, an
invariant, a hand-worked example (tests/golden/) or a brute-force loop, chosen
so that a plausible slip (a dropped term, a wrong sign, index or operand order,
an off-by-one causal position) fails at least one of them.
"""
import cmath
import itertools
import json
import math
import os

import numpy as np
import pytest

import oracle
from workload import GLM, TINY, mla_inputs, dsa_inputs, workload_inputs
from tests._np import to_np

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _rng(seed=0):
    return np.random.default_rng(seed)


# --------------------------------------------------------------------------- RoPE
def test_rope_textbook_values():
    """qk_rope=4, base=10000: pair 0 turns by pos rad, pair 1 by pos/100 rad.

    At pos=100 the angles are 100 rad and 1 rad; the cos/sin constants below
    are textbook values, the products were worked out by hand.
    """
    cos100, sin100 = 0.862318872287684, -0.5063656411097588
    cos1, sin1 = 0.5403023058681398, 0.8414709848078965
    x = np.array([1.0, 2.0, 3.0, 4.0])          # pairs (1,2) and (3,4)
    y = oracle.rope_interleave(x, 100, 10000.0)
    expected = [1 * cos100 - 2 * sin100,        # v[0]      = a0*cs0 - b0*sn0
                3 * cos1 - 4 * sin1,            # v[1]      = a1*cs1 - b1*sn1
                2 * cos100 + 1 * sin100,        # v[half+0] = b0*cs0 + a0*sn0
                4 * cos1 + 3 * sin1]            # v[half+1] = b1*cs1 + a1*sn1
    np.testing.assert_allclose(y, expected, rtol=0, atol=1e-12)
    np.testing.assert_allclose(expected, [1.8750501545072016, -1.7449770216271666,
                                          1.2182721034656092, 4.685622177896248], atol=1e-12)


def test_rope_matches_complex_rotation():
    """Brute force: pair j is the complex number a + ib multiplied by e^{i pos theta_j}."""
    r = _rng(1)
    for d in (2, 8, 64):
        x = r.standard_normal(d)
        for pos in (0, 1, 7, 4095, 65535):
            y = oracle.rope_interleave(x, pos, 10000.0)
            half = d // 2
            for j in range(half):
                z = complex(x[2 * j], x[2 * j + 1]) * cmath.exp(1j * pos * 10000.0 ** (-(2 * j) / d))
                assert abs(y[j] - z.real) < 1e-9 and abs(y[half + j] - z.imag) < 1e-9


def test_rope_identity_at_zero_and_norm():
    r = _rng(2)
    x = r.standard_normal((5, 64))
    y0 = oracle.rope_interleave(x, 0)
    np.testing.assert_allclose(y0[:, :32], x[:, 0::2], atol=0)
    np.testing.assert_allclose(y0[:, 32:], x[:, 1::2], atol=0)
    y = oracle.rope_interleave(x, 123)
    np.testing.assert_allclose(np.linalg.norm(y, axis=-1), np.linalg.norm(x, axis=-1), rtol=1e-12)


def test_rope_relative_position_invariance():
    """RoPE(q,p) . RoPE(k,t) depends only on p - t."""
    r = _rng(3)
    q, k = r.standard_normal(64), r.standard_normal(64)
    d = lambda p, t: float(oracle.rope_interleave(q, p) @ oracle.rope_interleave(k, t))
    for p, t, shift in [(10, 3, 100), (500, 499, 7), (0, 0, 31)]:
        assert abs(d(p, t) - d(p + shift, t + shift)) < 1e-9
    assert abs(d(10, 3) - d(10, 4)) > 1e-6  # and it does depend on the offset


# ------------------------------------------------------------------ geometry pin
def test_glm_geometry_matches_page():
    g = _load("cache_geometry.json")
    assert GLM.H == g["heads"]
    assert GLM.qk_head == g["naive_k_per_head"] and GLM.v_head == g["naive_v_per_head"]
    assert GLM.H * (GLM.qk_head + GLM.v_head) == g["naive_floats_per_token"]
    assert GLM.kv_lora + GLM.qk_rope == g["mla_floats_per_token"]
    assert round(g["naive_floats_per_token"] / g["mla_floats_per_token"]) == g["compression_rounded"]


# ------------------------------------------------------- attention closed forms
def _eye_kvb(n):
    """kv_b for H=1 whose W_UK and W_UV are both the n x n identity."""
    return np.concatenate([np.eye(n), np.eye(n)], axis=0)[None]


def test_two_token_closed_form_latent_part():
    """H=1, qk_nope=qk_rope=kv_lora=v_head=2, scale=1/2.

    q_nope=[1,0] picks Lc[t][0]; Lc = [[2 ln 3, 0], [0, 0]] gives scores
    [ln 3, 0], probabilities [3/4, 1/4], out = [1.5 ln 3, 0].
    """
    q = np.array([[1.0, 0.0, 0.0, 0.0]])
    Lc = np.array([[2 * math.log(3), 0.0], [0.0, 0.0]])
    Rc = np.zeros((2, 2))
    for f in (oracle.attend_dense, oracle.attend_absorbed):
        out = f(q, Lc, Rc, _eye_kvb(2), 2, 1, 0.5)
        np.testing.assert_allclose(out, [[1.5 * math.log(3), 0.0]], atol=1e-14)


def test_two_token_closed_form_rope_part():
    """The rope part alone decides: q_rope=(1,0) at pos=1 rotates to (cos 1, sin 1).

    Rc[0] = 2 ln 3 * (cos 1, sin 1) gives score ln 3 for key 0, 0 for key 1, so
    p = [3/4, 1/4] and out = W_UV (3/4 Lc[0] + 1/4 Lc[1]) = [3/4, 1/4].
    The query position is T - S + s = 1 (T=2, S=1); another position breaks it.
    """
    q = np.array([[[[0.0, 0.0, 1.0, 0.0]]]])                 # [B=1,S=1,H=1,4]
    Lc = np.array([[[1.0, 0.0], [0.0, 1.0]]])
    Rc = np.array([[[2 * math.log(3) * math.cos(1), 2 * math.log(3) * math.sin(1)], [0.0, 0.0]]])
    for f in (oracle.decode_dense, oracle.decode_absorbed):
        out = f(q, Lc, Rc, [2], _eye_kvb(2), 2, 0.5)
        np.testing.assert_allclose(out[0, 0], [[0.75, 0.25]], atol=1e-14)


def test_single_token_returns_its_value():
    """T=1: softmax of one score is 1, so out = W_UV Lc[0] whatever q is."""
    r = _rng(4)
    q = r.standard_normal((TINY.H, TINY.qk_head))
    Lc = r.standard_normal((1, TINY.kv_lora))
    Rc = r.standard_normal((1, TINY.qk_rope))
    kvb = r.standard_normal((TINY.H, TINY.qk_nope + TINY.v_head, TINY.kv_lora))
    W_UV = kvb[:, TINY.qk_nope:, :]
    expect = np.stack([W_UV[h] @ Lc[0] for h in range(TINY.H)])
    for f in (oracle.attend_dense, oracle.attend_absorbed):
        np.testing.assert_allclose(f(q, Lc, Rc, kvb, TINY.qk_nope, 0, 0.3), expect, rtol=1e-12)


def test_zero_query_is_uniform_average():
    """q = 0 makes all scores equal: out = W_UV mean_t Lc[t]."""
    r = _rng(5)
    n = 9
    q = np.zeros((TINY.H, TINY.qk_head))
    Lc = r.standard_normal((n, TINY.kv_lora))
    Rc = r.standard_normal((n, TINY.qk_rope))
    kvb = r.standard_normal((TINY.H, TINY.qk_nope + TINY.v_head, TINY.kv_lora))
    expect = np.stack([kvb[h, TINY.qk_nope:] @ Lc.mean(axis=0) for h in range(TINY.H)])
    for f in (oracle.attend_dense, oracle.attend_absorbed):
        np.testing.assert_allclose(f(q, Lc, Rc, kvb, TINY.qk_nope, n - 1, 0.3), expect, rtol=1e-12)


def test_softmax_rows_sum_to_one():
    r = _rng(6)
    q = r.standard_normal((TINY.H, TINY.qk_head)) * 5
    Lc = r.standard_normal((40, TINY.kv_lora))
    Rc = r.standard_normal((40, TINY.qk_rope))
    kvb = r.standard_normal((TINY.H, TINY.qk_nope + TINY.v_head, TINY.kv_lora))
    _, p = oracle.attend_absorbed(q, Lc, Rc, kvb, TINY.qk_nope, 39, 0.2, return_probs=True)
    assert p.shape == (TINY.H, 40)
    assert np.all(p >= 0)
    np.testing.assert_allclose(p.sum(axis=-1), 1.0, atol=1e-12)


# --------------------------------------------------------------- brute force
def _brute_attention(q, Lc, Rc, kvb, qk_nope, pos, scale, base):
    """Scalar loops written from the definition: rebuild k and v per head and token."""
    H, Dq = len(q), len(q[0])
    Dr = Dq - qk_nope
    v_head = len(kvb[0]) - qk_nope
    out = []
    for h in range(H):
        qr = list(q[h][qk_nope:])
        rot = [0.0] * Dr
        for j in range(Dr // 2):
            ang = pos * base ** (-(2 * j) / Dr)
            a, b = qr[2 * j], qr[2 * j + 1]
            rot[j] = a * math.cos(ang) - b * math.sin(ang)
            rot[Dr // 2 + j] = b * math.cos(ang) + a * math.sin(ang)
        scores, values = [], []
        for t in range(len(Lc)):
            k = [sum(kvb[h][i][l] * Lc[t][l] for l in range(len(Lc[t]))) for i in range(qk_nope)]
            k += list(Rc[t])
            qt = list(q[h][:qk_nope]) + rot
            scores.append(scale * sum(qt[i] * k[i] for i in range(Dq)))
            values.append([sum(kvb[h][qk_nope + j][l] * Lc[t][l] for l in range(len(Lc[t])))
                           for j in range(v_head)])
        m = max(scores)
        e = [math.exp(s - m) for s in scores]
        z = sum(e)
        out.append([sum(e[t] / z * values[t][j] for t in range(len(Lc))) for j in range(v_head)])
    return np.array(out)


@pytest.mark.parametrize("pos", [0, 3, 6])
def test_attention_brute_force(pos):
    r = _rng(7 + pos)
    H, Dn, Dr, Dl, Dv = 2, 3, 4, 5, 3
    q = r.standard_normal((H, Dn + Dr))
    Lc = r.standard_normal((pos + 1, Dl))
    Rc = r.standard_normal((pos + 1, Dr))
    kvb = r.standard_normal((H, Dn + Dv, Dl))
    ref = _brute_attention(q.tolist(), Lc.tolist(), Rc.tolist(), kvb.tolist(), Dn, pos, 0.37, 10000.0)
    for f in (oracle.attend_dense, oracle.attend_absorbed):
        np.testing.assert_allclose(f(q, Lc, Rc, kvb, Dn, pos, 0.37, 10000.0), ref, rtol=1e-12, atol=1e-12)


# --------------------------------------------- absorbed == dense == prefill
def _tiny_inputs(T, S, B=1, seed=11):
    T_list = [T] * B if isinstance(T, int) else list(T)
    x = mla_inputs(TINY, len(T_list), S, T_list, max(T_list), "f32", seed, "cpu")
    return {k: (to_np(v) if k != "T" else v.numpy()) for k, v in x.items()}


def test_absorbed_equals_dense_tiny_workload():
    """The tiny workload (T=64) three ways; the identity is exact up to rounding."""
    x = workload_inputs("tiny")
    q, Lc, Rc, kvb = (to_np(x[k]) for k in ("q", "Lc", "Rc", "kv_b"))
    T = x["T"].numpy()
    sc = TINY.softmax_scale
    a = oracle.decode_absorbed(q, Lc, Rc, T, kvb, TINY.qk_nope, sc)
    d = oracle.decode_dense(q, Lc, Rc, T, kvb, TINY.qk_nope, sc)
    np.testing.assert_allclose(a, d, rtol=1e-12, atol=1e-13)
    p = oracle.prefill_nonabsorbed(q[0], Lc[0], Rc[0], kvb, TINY.qk_nope, sc, pos_base=63)
    np.testing.assert_allclose(p, a[0], rtol=1e-12, atol=1e-13)


def test_prefill_equals_decode_block():
    """S=6 new tokens (a verify-sized block) at pos_base=10: prefill == decode with T=16."""
    x = _tiny_inputs(16, 6)
    sc = TINY.softmax_scale
    dec = oracle.decode_absorbed(x["q"], x["Lc"], x["Rc"], x["T"], x["kv_b"], TINY.qk_nope, sc)
    pre = oracle.prefill_nonabsorbed(x["q"][0], x["Lc"][0], x["Rc"][0], x["kv_b"], TINY.qk_nope, sc, 10)
    np.testing.assert_allclose(pre, dec[0], rtol=1e-12, atol=1e-13)


def test_causal_positions():
    """S=6, T=6: query s sits at pos s; query 0 sees only key 0; each query equals
    a one-token decode over the cache truncated to pos+1 rows."""
    x = _tiny_inputs(6, 6)
    sc = TINY.softmax_scale
    out = oracle.decode_absorbed(x["q"], x["Lc"], x["Rc"], x["T"], x["kv_b"], TINY.qk_nope, sc)
    W_UV = x["kv_b"][:, TINY.qk_nope:]
    np.testing.assert_allclose(out[0, 0], np.stack([W_UV[h] @ x["Lc"][0, 0] for h in range(TINY.H)]),
                               rtol=1e-12)
    for s in range(6):
        one = oracle.decode_absorbed(x["q"][:, s:s + 1], x["Lc"], x["Rc"], [s + 1], x["kv_b"],
                                     TINY.qk_nope, sc)
        np.testing.assert_allclose(out[0, s], one[0, 0], rtol=1e-12)
    assert oracle.query_positions(100, 6) == [94, 95, 96, 97, 98, 99]


def test_decode_ignores_rows_past_length():
    """Cache rows at t >= T[b] are NaN in the generator; the result stays finite."""
    x = _tiny_inputs([20, 33], 2, B=2)
    sc = TINY.softmax_scale
    out = oracle.decode_absorbed(x["q"], x["Lc"], x["Rc"], x["T"], x["kv_b"], TINY.qk_nope, sc)
    assert np.all(np.isfinite(out))


# ------------------------------------------------------------------- indexer
def test_index_scores_hand_example():
    g = _load("indexer_hand_example.json")
    q_idx = np.array(g["q_idx"], dtype=float)[None, None]
    w = np.array(g["w"], dtype=float)[None, None]
    Ic = np.array(g["Ic"], dtype=float)[None]
    got = oracle.index_scores(q_idx, w, Ic, [g["T"]])[0, 0]
    exp = np.array([float(v) for v in g["expected"]])
    assert np.array_equal(got, exp)


def test_index_scores_brute_force():
    r = _rng(12)
    B, S, nh, hd, T_cap = 2, 3, 3, 4, 9
    T = [9, 5]
    q_idx = r.integers(-4, 5, (B, S, nh, hd)).astype(float)
    w = r.integers(-4, 5, (B, S, nh)).astype(float)
    Ic = r.integers(-4, 5, (B, T_cap, hd)).astype(float)
    got = oracle.index_scores(q_idx, w, Ic, T)
    for b, s, t in itertools.product(range(B), range(S), range(T_cap)):
        pos = T[b] - S + s
        if t > pos:
            assert got[b, s, t] == -np.inf
            continue
        ref = 0.0
        for h in range(nh):
            dot = sum(q_idx[b, s, h, d] * Ic[b, t, d] for d in range(hd))
            ref += w[b, s, h] * (dot if dot > 0 else 0.0)
        assert got[b, s, t] == ref


def test_index_scores_exact_integers_dsa_bound():
    """With integers in [-4,4], |q.k| <= hd*16 and |I| <= n_ih*4*hd*16 < 2^24 (exact in fp32)."""
    assert 32 * 4 * 128 * 16 < 2 ** 24
    x = dsa_inputs(1, 1, [300], 300, 32, 128, 99, "cpu")
    I = oracle.index_scores(to_np(x["q_idx"]), to_np(x["w"]), to_np(x["Ic"]), [300])
    assert np.array_equal(I, np.round(I))
    assert np.array_equal(I.astype(np.float32).astype(np.float64), I)


# --------------------------------------------------------------------- top-k
def _parse(v):
    return float(v) if not isinstance(v, str) else float(v.replace("inf", "inf"))


def test_topk_hand_example():
    g = _load("topk_hand_example.json")
    sc = np.array([_parse(v) for v in g["scores"]])[None, None]
    assert math.copysign(1.0, sc[0, 0, 5]) == -1.0  # the fixture really holds -0.0
    for case in g["cases"]:
        sel, nsel = oracle.topk_select(sc, [g["T"]], 1, case["k"])
        n = int(nsel[0, 0])
        assert sel[0, 0, :n].tolist() == case["expected"]
        assert np.all(sel[0, 0, n:] == -1)


def test_topk_brute_force_with_ties():
    """Python sorted() with the comparator (score desc, index asc) on many tied integers."""
    r = _rng(13)
    B, S, T_cap, k = 3, 2, 64, 16
    T = [64, 40, 17]
    sc = r.integers(-3, 4, (B, S, T_cap)).astype(float)
    sc[0, 0, ::5] = -0.0
    sel, nsel = oracle.topk_select(sc, T, S, k)
    for b in range(B):
        for s in range(S):
            pos = T[b] - S + s
            cand = list(range(pos + 1))
            if len(cand) > k:
                cand = sorted(cand, key=lambda t: (-sc[b, s, t], t))[:k]
            exp = sorted(cand)
            n = int(nsel[b, s])
            assert n == len(exp)
            assert sel[b, s, :n].tolist() == exp
            assert max(exp) <= pos


# -------------------------------------------------------------------- sparse
def test_sparse_keep_all_equals_dense():
    x = _tiny_inputs([30, 64], 2, B=2, seed=21)
    sc = TINY.softmax_scale
    T = x["T"]
    k = 64
    scores = np.zeros((2, 2, 64))
    sel, nsel = oracle.topk_select(scores, T, 2, k)
    sp = oracle.sparse_decode(x["q"], x["Lc"], x["Rc"], T, x["kv_b"], sel, nsel, TINY.qk_nope, sc)
    de = oracle.decode_dense(x["q"], x["Lc"], x["Rc"], T, x["kv_b"], TINY.qk_nope, sc)
    np.testing.assert_allclose(sp, de, rtol=1e-12, atol=1e-13)


def test_sparse_subset_equals_dense_on_gathered_rows():
    """A selection is dense attention over the gathered rows at the query's own position."""
    x = _tiny_inputs(40, 1, seed=22)
    sc = TINY.softmax_scale
    idx = np.array([0, 3, 4, 17, 38, 39])
    sel = np.full((1, 1, 8), -1)
    sel[0, 0, :6] = idx
    nsel = np.array([[6]])
    sp = oracle.sparse_decode(x["q"], x["Lc"], x["Rc"], [40], x["kv_b"], sel, nsel, TINY.qk_nope, sc)
    ref = oracle.attend_dense(x["q"][0, 0], x["Lc"][0, idx], x["Rc"][0, idx], x["kv_b"], TINY.qk_nope,
                              39, sc)
    np.testing.assert_allclose(sp[0, 0], ref, rtol=1e-12, atol=1e-13)


def test_sparse_rejects_future_keys():
    x = _tiny_inputs(10, 1, seed=23)
    sel = np.array([[[2, 10]]])
    with pytest.raises(AssertionError):
        oracle.sparse_decode(x["q"], x["Lc"], x["Rc"], [10], x["kv_b"], sel, np.array([[2]]),
                             TINY.qk_nope, TINY.softmax_scale)


# -------------------------------------------------------------- independence
def test_oracle_is_independent_of_the_cuda_path():
    """The oracle imports neither the product package nor any compiled code."""
    here = os.path.join(os.path.dirname(os.path.dirname(__file__)), "oracle")
    for fn in os.listdir(here):
        if fn.endswith(".py"):
            src = open(os.path.join(here, fn)).read()
            assert "mla_latent_kv_06_gb300" not in src
            assert "ctypes" not in src and "import torch" not in src


# --------------------------------------------------------------- cache append ([MLA-KV] §2.1, §2.2)
def test_rms_norm_hand_values_and_invariances():
    """x = (1,-1,1,-1) has mean square 1, so RMSNorm (eps 0) returns x * w exactly;
    a zero vector stays zero; the result does not depend on the scale of x."""
    w = np.array([2.0, 3.0, 4.0, 5.0])
    assert np.array_equal(oracle.rms_norm(np.array([1.0, -1.0, 1.0, -1.0]), w, 0.0), [2.0, -3.0, 4.0, -5.0])
    assert np.array_equal(oracle.rms_norm(np.zeros(4), w, 1e-6), np.zeros(4))
    r = np.random.default_rng(1).standard_normal((3, 16))
    assert np.allclose(oracle.rms_norm(7.5 * r, np.ones(16), 0.0), oracle.rms_norm(r, np.ones(16), 0.0), atol=1e-13)
    y = oracle.rms_norm(r, np.ones(16), 0.0)
    assert np.allclose(np.mean(y * y, axis=-1), 1.0, atol=1e-13)


def test_layer_norm_hand_values_and_moments():
    """(1,2,3): mean 2, variance 2/3, so the normalised values are (-1,0,1)*sqrt(3/2);
    weight 1 and bias 5 shift them by 5.  Normalised rows have mean 0 and variance 1."""
    y = oracle.layer_norm(np.array([1.0, 2.0, 3.0]), np.ones(3), np.full(3, 5.0), 0.0)
    assert np.allclose(y, [5.0 - 1.224744871391589, 5.0, 5.0 + 1.224744871391589], atol=1e-14)
    r = np.random.default_rng(2).standard_normal((4, 128)) * 3.0 + 1.5
    z = oracle.layer_norm(r, np.ones(128), None, 0.0)
    assert np.allclose(z.mean(axis=-1), 0.0, atol=1e-13) and np.allclose(z.var(axis=-1), 1.0, atol=1e-12)


def test_cache_append_rows_and_positions():
    """New tokens land at pos = T[b] - S + s; at pos 0 the rope part is only
    de-interleaved (pairs (x0,x1),(x2,x3) -> x0,x2 | x1,x3)."""
    assert np.array_equal(oracle.new_token_positions([10, 7], 2), [[8, 9], [5, 6]])
    comp = np.arange(1, 13, dtype=np.float64).reshape(1, 1, 12)  # kv_lora 8, qk_rope 4
    lc, rc, pos = oracle.cache_append(comp, np.ones(8), 0.0, [1], 8)
    assert pos.tolist() == [[0]]
    assert np.array_equal(rc[0, 0], [9.0, 11.0, 10.0, 12.0])
    x = comp[0, 0, :8]
    assert np.allclose(lc[0, 0], x / np.sqrt(np.mean(x * x)), atol=1e-14)


def test_index_key_append_layout():
    """rope_dim 0 is LayerNorm alone; with a rotated tail the leading values are untouched
    and the tail keeps its norm pairwise (a rotation)."""
    r = np.random.default_rng(4).standard_normal((2, 3, 16))
    w, b = np.random.default_rng(5).standard_normal(16), np.random.default_rng(6).standard_normal(16)
    plain, _ = oracle.index_key_append(r, w, b, 1e-6, [40, 3], 0)
    assert np.allclose(plain, oracle.layer_norm(r, w, b, 1e-6))
    rot, pos = oracle.index_key_append(r, w, b, 1e-6, [40, 3], 8)
    assert np.array_equal(rot[..., :8], plain[..., :8])
    a0, a1 = plain[..., 8::2], plain[..., 9::2]
    assert np.allclose(rot[..., 8:12] ** 2 + rot[..., 12:16] ** 2, a0 ** 2 + a1 ** 2, atol=1e-12)
    assert pos.tolist() == [[37, 38, 39], [0, 1, 2]]


# --------------------------------------------------------------- paged layout
def test_page_row_hand_example():
    """Pages of 2 rows; sequence 0 uses pages 2 then 0, sequence 1 uses page 1:
    token rows worked out by hand from the block table."""
    table = [[2, 0], [1, -1]]
    assert [oracle.page_row(table, 0, t, 2) for t in range(4)] == [4, 5, 0, 1]
    assert [oracle.page_row(table, 1, t, 2) for t in range(2)] == [2, 3]
    pool = np.arange(3 * 2 * 1, dtype=np.float64).reshape(3, 2, 1)  # row r holds the value r
    out = oracle.unpage(pool, table, [3, 2])
    assert out[0, :3, 0].tolist() == [4.0, 5.0, 0.0] and out[1, :2, 0].tolist() == [2.0, 3.0]
    assert np.isnan(out[1, 2, 0])


def test_identity_block_table_is_the_contiguous_layout():
    """With page b*max_pages + i at table[b, i], the pool read as [B, T_cap, D] is
    the contiguous cache itself."""
    r = np.random.default_rng(7).standard_normal((2, 8, 3))  # B=2, T_cap=8, D=3
    pool = r.reshape(8, 2, 3)                                 # 8 pages of 2 rows
    table = [[0, 1, 2, 3], [4, 5, 6, 7]]
    assert np.array_equal(oracle.unpage(pool, table, [8, 5])[0], r[0])
    assert np.array_equal(oracle.unpage(pool, table, [8, 5])[1, :5], r[1, :5])


# --------------------------------------------------------------- output projection
def test_o_proj_hand_values_and_one_hot():
    """y = x W^T worked by hand for a 2x3 weight; a one-hot row of x returns the
    matching column of W."""
    w = np.array([[1.0, 2.0, 3.0], [-1.0, 0.5, 4.0]])
    x = np.array([[1.0, 1.0, 1.0], [2.0, 0.0, -1.0]])
    assert np.array_equal(oracle.o_proj(x, w), [[6.0, 3.5], [-1.0, -6.0]])
    r = np.random.default_rng(3).standard_normal((5, 7))
    for k in range(7):
        e = np.zeros((1, 7))
        e[0, k] = 1.0
        assert np.array_equal(oracle.o_proj(e, r)[0], r[:, k])


# ------------------------------------------------------------- FP8 latent cache
def test_e4m3_textbook_values():
    """Values fixed by the format: bias 7, three mantissa bits, subnormals
    M * 2^-9, no infinities, S.1111.111 is NaN."""
    table = {0x00: 0.0, 0x01: 2.0 ** -9, 0x07: 7 * 2.0 ** -9, 0x08: 2.0 ** -6, 0x30: 0.5, 0x38: 1.0,
             0x39: 1.125, 0x3F: 1.875, 0x40: 2.0, 0x70: 128.0, 0x78: 256.0, 0x7E: 448.0, 0xB8: -1.0, 0xFE: -448.0}
    for code, val in table.items():
        assert oracle.e4m3_decode(code) == val, hex(code)
    assert np.isnan(oracle.e4m3_decode(0x7F)) and np.isnan(oracle.e4m3_decode(0xFF))
    assert np.signbit(oracle.e4m3_decode(0x80)) and oracle.e4m3_decode(0x80) == 0.0
    pos = oracle.e4m3_decode(np.arange(127))
    assert np.all(np.diff(pos) > 0)                                    # monotone in the code
    np.testing.assert_array_equal(oracle.e4m3_decode(np.arange(128, 255)), -pos)


def test_e4m3_matches_torch_float8():
    """All 256 codes, and a spread of values inside the finite range, against
    torch's float8_e4m3fn (a library routine of the same format)."""
    torch = pytest.importorskip("torch")
    codes = np.arange(256)
    ref = torch.tensor(codes, dtype=torch.uint8).view(torch.float8_e4m3fn).double().numpy()
    got = oracle.e4m3_decode(codes)
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    assert np.array_equal(got[~np.isnan(got)], ref[~np.isnan(ref)])
    r = _rng(11)
    x = np.clip(r.standard_normal(50000) * np.exp(r.uniform(-12, 7, 50000)), -448, 448)
    x = np.concatenate([x, oracle.e4m3_decode(np.arange(126)) * 1.0000001, [0.0, -0.0, 448.0]])
    ref = torch.tensor(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(oracle.e4m3_encode(x), ref)


def test_e4m3_rounding_by_hand():
    """Halfway cases go to the even code; past 448 saturates; NaN stays NaN."""
    cases = {1.0625: 0x38,        # halfway 1.0 (0x38) / 1.125 (0x39) -> even 0x38
             1.1875: 0x3A,        # halfway 1.125 (0x39) / 1.25 (0x3A) -> even 0x3A
             1.07: 0x39, 1.05: 0x38,
             2.0 ** -10: 0x00,    # halfway 0 / 2^-9 -> 0x00
             3 * 2.0 ** -10: 0x02,  # halfway 2^-9 (0x01) / 2^-8 (0x02) -> 0x02
             464.0: 0x7E, 1e6: 0x7E, -1e6: 0xFE, -1.0: 0xB8}
    for x, code in cases.items():
        assert int(oracle.e4m3_encode(x)) == code, x
    assert int(oracle.e4m3_encode(float("nan"))) == 0x7F
    finite = np.array([c for c in range(256) if c not in (0x7F, 0xFF)])
    np.testing.assert_array_equal(oracle.e4m3_encode(oracle.e4m3_decode(finite)), finite)


def test_cache_append_fp8_codes_within_half_a_quantum():
    """The codes decode to the normalised row over lat_scale to within half a
    quantum of E4M3 (2^-4 relative for normal values, 2^-10 absolute below
    2^-6); the rope part is cache_append's."""
    r = _rng(12)
    B, S, Dl, Dr = 2, 3, 32, 8
    comp = r.standard_normal((B, S, Dl + Dr))
    w = r.uniform(0.5, 1.5, Dl)
    lat_scale = math.sqrt(Dl) * 1.5 / 448
    codes, rc, pos = oracle.cache_append_fp8(comp, w, 1e-6, [5, 9], Dl, lat_scale)
    lc, rc0, pos0 = oracle.cache_append(comp, w, 1e-6, [5, 9], Dl)
    y = lc / lat_scale
    d = oracle.e4m3_decode(codes)
    bound = np.maximum(np.abs(y) * 2.0 ** -4, 2.0 ** -10)
    assert np.all(np.abs(d - y) <= bound + 1e-12)
    assert np.max(np.abs(y)) <= 448                       # the RMSNorm bound keeps the row in range
    np.testing.assert_array_equal(rc, rc0)
    np.testing.assert_array_equal(pos, pos0)
    np.testing.assert_allclose(oracle.dequant_latent(codes, lat_scale), lat_scale * d)

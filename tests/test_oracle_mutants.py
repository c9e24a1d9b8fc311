"""Planted mistakes in the oracle must fail its pins (CPU only).

Each case replaces one function of the oracle with a copy that carries one
plausible slip -- a flipped sign, a dropped term, a swapped operand, an
off-by-one position -- and runs the pin tests of test_oracle_pins.py against
the changed oracle.  The pins are only worth something if every such slip
fails at least one of them (an assertion, or an error on an input the slip
cannot handle).  The mistakes live here, in the test, and are
planted with monkeypatch for the duration of one case.
"""
import inspect

import numpy as np
import pytest

import oracle
import oracle.mla as om
from tests import test_oracle_pins as pins

_f64 = om._f64


# ------------------------------------------------------------------ RoPE slips
def _rope(pair, out, theta_num, sign):
    def rope(x, pos, base=10000.0):
        x = _f64(x)
        d = x.shape[-1]
        half = d // 2
        j = np.arange(half, dtype=np.float64)
        ang = _f64(pos)[..., None] * base ** (-theta_num * j / d)
        cs, sn = np.cos(ang), sign * np.sin(ang)
        a, b = (x[..., 0::2], x[..., 1::2]) if pair == "even_odd" else (x[..., :half], x[..., half:])
        y = np.empty_like(x)
        ya, yb = a * cs - b * sn, b * cs + a * sn
        if out == "halves":
            y[..., :half], y[..., half:] = ya, yb
        else:
            y[..., 0::2], y[..., 1::2] = ya, yb
        return y
    return rope


# ------------------------------------------------------------- attention slips
def _absorbed(no_rope=False, unrotated=False, swap_kvb=False, no_scale=False):
    def attend(q, Lc_rows, Rc_rows, kv_b, qk_nope, pos, scale, rope_base=10000.0, return_probs=False):
        q, L, R, kvb = _f64(q), _f64(Lc_rows), _f64(Rc_rows), _f64(kv_b)
        v_head = kvb.shape[1] - qk_nope
        if swap_kvb:   # value rows taken first
            W_UV, W_UK = kvb[:, :v_head], kvb[:, v_head:]
        else:
            W_UK, W_UV = kvb[:, :qk_nope], kvb[:, qk_nope:]
        qabs = np.einsum("hi,hil->hl", q[:, :qk_nope], W_UK)
        q_rot = q[:, qk_nope:] if unrotated else om.rope_interleave(q[:, qk_nope:], pos, rope_base)
        sc = qabs @ L.T + (0.0 if no_rope else q_rot @ R.T)
        p = om.softmax_probs(sc if no_scale else scale * sc)
        clat = p @ L
        out = np.einsum("hjl,hl->hj", W_UV, clat)
        return (out, p) if return_probs else out
    return attend


def _dense_no_rope(q, Lc_rows, Rc_rows, kv_b, qk_nope, pos, scale, rope_base=10000.0):
    q, L = _f64(q), _f64(Lc_rows)
    W_UK, W_UV = om.split_kv_b(kv_b, qk_nope)
    k_nope = np.einsum("hil,tl->thi", W_UK, L)
    v = np.einsum("hjl,tl->thj", W_UV, L)
    p = om.softmax_probs(scale * np.einsum("hi,thi->ht", q[:, :qk_nope], k_nope))
    return np.einsum("ht,thj->hj", p, v)


def _split_swapped(kv_b, qk_nope):
    kv_b = _f64(kv_b)
    v_head = kv_b.shape[1] - qk_nope
    return kv_b[:, v_head:, :], kv_b[:, :v_head, :]


def _softmax_unnormalised(scores):
    s = _f64(scores)
    return np.exp(s - np.max(s, axis=-1, keepdims=True))


def _positions(shift):
    return lambda T_b, S: [T_b - S + s + shift for s in range(S)]


def _prefill_exclusive(q, Lc, Rc, kv_b, qk_nope, scale, pos_base, rope_base=10000.0, queries=None, heads=None):
    """Causal bound t < pos (the query does not see its own key)."""
    q, kvb = _f64(q), _f64(kv_b)
    S, H = q.shape[0], q.shape[1]
    Tk = pos_base + S
    L, R = _f64(Lc)[:Tk], _f64(Rc)[:Tk]
    KV = np.einsum("hjl,tl->thj", kvb, L)
    out = np.full((S, H, kvb.shape[1] - qk_nope), np.nan)
    for s in range(S) if queries is None else queries:
        pos = pos_base + s
        n = max(pos, 1)
        q_rot = om.rope_interleave(q[s, :, qk_nope:], pos, rope_base)
        sc = scale * (np.einsum("hi,thi->ht", q[s, :, :qk_nope], KV[:n, :, :qk_nope]) + q_rot @ R[:n].T)
        out[s] = np.einsum("ht,thj->hj", om.softmax_probs(sc), KV[:n, :, qk_nope:])
    return out


def _prefill(kind):
    """The two-step prefill with one slip: key and value rows swapped, the query
    one position late, or the rotation at the row index instead of the position."""
    def prefill(q, Lc, Rc, kv_b, qk_nope, scale, pos_base, rope_base=10000.0, queries=None, heads=None):
        q, kvb = _f64(q), _f64(kv_b)
        S, H = q.shape[0], q.shape[1]
        Tk = pos_base + S
        L, R = _f64(Lc)[:Tk], _f64(Rc)[:Tk]
        KV = np.einsum("hjl,tl->thj", kvb, L)
        v_head = kvb.shape[1] - qk_nope
        if kind == "swap":
            kn, val = KV[..., v_head:], KV[..., :v_head]
        else:
            kn, val = KV[..., :qk_nope], KV[..., qk_nope:]
        out = np.full((S, H, v_head), np.nan)
        for s in range(S) if queries is None else queries:
            pos = pos_base + s + (1 if kind == "late" else 0)
            n = min(pos + 1, Tk)
            q_rot = om.rope_interleave(q[s, :, qk_nope:], s if kind == "rope_at_row" else pos, rope_base)
            sc = scale * (np.einsum("hi,thi->ht", q[s, :, :qk_nope], kn[:n]) + q_rot @ R[:n].T)
            out[s] = np.einsum("ht,thj->hj", om.softmax_probs(sc), val[:n])
        return out
    return prefill


# ---------------------------------------------------------------- indexer slips
def _index(variant):
    def index_scores(q_idx, w, Ic, T, S_positions=None):
        qi, ww = _f64(q_idx), _f64(w)
        B, S = qi.shape[0], qi.shape[1]
        out = np.full((B, S, np.asarray(Ic).shape[1]), -np.inf)
        for b in range(B):
            for s, pos in enumerate(om.query_positions(int(T[b]), S)):
                dots = qi[b, s] @ _f64(np.asarray(Ic)[b, :pos + 1]).T
                if variant == "no_relu":
                    v = ww[b, s] @ dots
                elif variant == "no_weights":
                    v = np.maximum(dots, 0.0).sum(axis=0)
                elif variant == "relu_after_sum":
                    v = np.maximum(ww[b, s] @ dots, 0.0)
                else:   # "abs": |.| in place of ReLU
                    v = ww[b, s] @ np.abs(dots)
                out[b, s, :pos + 1] = v
        return out
    return index_scores


def _topk(variant):
    def topk_select(scores, T, S, k):
        sc = np.asarray(scores)
        B = sc.shape[0]
        sel = np.full((B, S, k), -1, dtype=np.int64)
        nsel = np.zeros((B, S), dtype=np.int64)
        for b in range(B):
            for s, pos in enumerate(om.query_positions(int(T[b]), S)):
                n = int(T[b]) if variant == "not_causal" else pos + 1
                idx = np.arange(n)
                vals = _f64(sc[b, s, :n])
                vals = np.where(np.isneginf(vals), np.finfo(np.float64).min, vals)
                if variant == "ties_high":
                    order = np.lexsort((-idx, -vals))
                elif variant == "smallest":
                    order = np.lexsort((idx, vals))
                else:
                    order = np.lexsort((idx, -vals))
                keep = np.sort(order[:k])
                sel[b, s, :len(keep)] = keep
                nsel[b, s] = len(keep)
        return sel, nsel
    return topk_select


# ------------------------------------------------------------ norm / layout slips
def _rms(variant):
    def rms_norm(x, w, eps):
        x = _f64(x)
        if variant == "mean_abs":
            return x / (np.mean(np.abs(x), axis=-1, keepdims=True) + eps) * _f64(w)
        if variant == "no_weight":
            return x / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps)
        return x / np.sqrt(np.sum(x * x, axis=-1, keepdims=True) + eps) * _f64(w)   # "sum"
    return rms_norm


def _layer(variant):
    def layer_norm(x, w, b, eps=1e-6):
        x = _f64(x)
        mu = 0.0 if variant == "no_center" else np.mean(x, axis=-1, keepdims=True)
        ddof = 1 if variant == "unbiased" else 0
        var = np.var(x, axis=-1, keepdims=True, ddof=ddof) if variant != "no_center" else \
            np.mean(x * x, axis=-1, keepdims=True)
        y = (x - mu) / np.sqrt(var + eps) * _f64(w)
        return y if b is None or variant == "no_bias" else y + _f64(b)
    return layer_norm


def _sparse_ignores_nsel(q, Lc, Rc, T, kv_b, sel, nsel, qk_nope, scale, rope_base=10000.0, rows=None):
    """Attends to all k entries of the selection, the -1 padding included."""
    q = np.asarray(q)
    B, S, H = q.shape[0], q.shape[1], q.shape[2]
    out = np.full((B, S, H, np.asarray(kv_b).shape[1] - qk_nope), np.nan)
    for b in range(B):
        for s, pos in enumerate(om.query_positions(int(T[b]), S)):
            idx = np.asarray(sel[b, s], dtype=np.int64)
            out[b, s] = om.attend_absorbed(q[b, s], np.asarray(Lc)[b, idx], np.asarray(Rc)[b, idx], kv_b, qk_nope,
                                           pos, scale, rope_base)
    return out


def _unpage_shifted(pool, block_table, T):
    """Reads token t from the row of token t + 1."""
    pool = _f64(pool)
    ps, D = pool.shape[1], pool.shape[2]
    rows = pool.reshape(-1, D)
    out = np.full((len(T), max(T), D), np.nan)
    for b, n in enumerate(T):
        for t in range(n):
            out[b, t] = rows[om.page_row(block_table, b, min(t + 1, n - 1), ps)]
    return out


def _dequant_without_scale(codes, lat_scale):
    return om.e4m3_decode(codes)


def _append_fp8_without_scale(comp, kv_a_ln, eps, T, kv_lora, lat_scale, base=10000.0):
    lc, rc, pos = om.cache_append(comp, kv_a_ln, eps, T, kv_lora, base)
    return om.e4m3_encode(lc), rc, pos


def _page_row_swapped(block_table, b, t, page_size):
    return int(block_table[b][t % page_size]) * page_size + t // page_size


def _page_row_unmapped(block_table, b, t, page_size):
    return (t // page_size) * page_size + t % page_size + b * 0


def _o_proj_untransposed_rows(x, w_o):
    return _f64(x)[::-1] @ _f64(w_o).T


def _key_append_no_rope(k_idx, ln_w, ln_b, eps, T, rope_dim, base=10000.0):
    k = om.layer_norm(k_idx, ln_w, ln_b, eps)
    return k, om.new_token_positions(T, k.shape[1])


def _key_append_head_rope(k_idx, ln_w, ln_b, eps, T, rope_dim, base=10000.0):
    k = om.layer_norm(k_idx, ln_w, ln_b, eps).copy()
    pos = om.new_token_positions(T, k.shape[1])
    if rope_dim > 0:
        k[..., :rope_dim] = om.rope_interleave(k[..., :rope_dim], pos, base)
    return k, pos


def _e4m3_decode(bias=7, subnormal_as_normal=False):
    def decode(codes):
        c = np.asarray(codes, dtype=np.int64)
        sign = np.where(c & 0x80, -1.0, 1.0)
        E, M = (c >> 3) & 0xF, (c & 0x7).astype(np.float64)
        normal = (1.0 + M / 8.0) * 2.0 ** (E - float(bias))
        mag = normal if subnormal_as_normal else np.where(E == 0, M * 2.0 ** (1 - bias - 3), normal)
        return sign * np.where((E == 15) & (M == 7), np.nan, mag)
    return decode


def _e4m3_encode(ties="even", saturate=True):
    def encode(x):
        x = _f64(x)
        grid = om.e4m3_decode(np.arange(127))
        a = np.abs(x) if not saturate else np.minimum(np.abs(x), 448.0)
        hi = np.clip(np.searchsorted(grid, a, side="left"), 0, 126)
        lo = np.maximum(hi - 1, 0)
        dlo, dhi = a - grid[lo], grid[hi] - a
        tie = hi if ties == "up" else lo
        pick = np.where(dlo < dhi, lo, np.where(dhi < dlo, hi, tie))
        code = pick.astype(np.int64) | np.where(np.signbit(x), 0x80, 0)
        code = np.where(a > 448.0, 0x7F, code)
        return np.where(np.isnan(x), 0x7F, code).astype(np.uint8)
    return encode


MUTANTS = {
    "rope_negative_angle": {"rope_interleave": _rope("even_odd", "halves", 2.0, -1.0)},
    "rope_half_split_pairs": {"rope_interleave": _rope("halves", "halves", 2.0, 1.0)},
    "rope_interleaved_output": {"rope_interleave": _rope("even_odd", "interleaved", 2.0, 1.0)},
    "rope_theta_exponent": {"rope_interleave": _rope("even_odd", "halves", 1.0, 1.0)},
    "kv_b_value_rows_first": {"split_kv_b": _split_swapped},
    "absorbed_value_rows_first": {"attend_absorbed": _absorbed(swap_kvb=True)},
    "absorbed_drops_rope_term": {"attend_absorbed": _absorbed(no_rope=True)},
    "absorbed_query_not_rotated": {"attend_absorbed": _absorbed(unrotated=True)},
    "absorbed_no_scale": {"attend_absorbed": _absorbed(no_scale=True)},
    "dense_drops_rope_term": {"attend_dense": _dense_no_rope},
    "softmax_not_normalised": {"softmax_probs": _softmax_unnormalised},
    "query_position_plus_one": {"query_positions": _positions(1)},
    "query_position_minus_one": {"query_positions": _positions(-1)},
    "prefill_excludes_self": {"prefill_nonabsorbed": _prefill_exclusive},
    "prefill_key_value_rows_swapped": {"prefill_nonabsorbed": _prefill("swap")},
    "prefill_query_one_late": {"prefill_nonabsorbed": _prefill("late")},
    "prefill_rope_at_row_index": {"prefill_nonabsorbed": _prefill("rope_at_row")},
    "indexer_no_relu": {"index_scores": _index("no_relu")},
    "indexer_no_head_weights": {"index_scores": _index("no_weights")},
    "indexer_relu_after_sum": {"index_scores": _index("relu_after_sum")},
    "indexer_abs_for_relu": {"index_scores": _index("abs")},
    "topk_ties_to_higher_index": {"topk_select": _topk("ties_high")},
    "topk_keeps_smallest": {"topk_select": _topk("smallest")},
    "topk_not_causal": {"topk_select": _topk("not_causal")},
    "rms_norm_mean_abs": {"rms_norm": _rms("mean_abs")},
    "rms_norm_no_weight": {"rms_norm": _rms("no_weight")},
    "rms_norm_sum_not_mean": {"rms_norm": _rms("sum")},
    "layer_norm_not_centred": {"layer_norm": _layer("no_center")},
    "layer_norm_unbiased_variance": {"layer_norm": _layer("unbiased")},
    "layer_norm_drops_bias": {"layer_norm": _layer("no_bias")},
    "index_key_not_rotated": {"index_key_append": _key_append_no_rope},
    "index_key_rotates_head": {"index_key_append": _key_append_head_rope},
    "sparse_ignores_nsel": {"sparse_decode": _sparse_ignores_nsel},
    "unpage_reads_the_next_token": {"unpage": _unpage_shifted},
    "dequant_drops_the_scale": {"dequant_latent": _dequant_without_scale},
    "fp8_append_drops_the_scale": {"cache_append_fp8": _append_fp8_without_scale},
    "page_row_div_mod_swapped": {"page_row": _page_row_swapped},
    "page_row_ignores_table": {"page_row": _page_row_unmapped},
    "o_proj_rows_reversed": {"o_proj": _o_proj_untransposed_rows},
    "e4m3_bias_8": {"e4m3_decode": _e4m3_decode(bias=8)},
    "e4m3_subnormals_as_normals": {"e4m3_decode": _e4m3_decode(subnormal_as_normal=True)},
    "e4m3_ties_away_from_zero": {"e4m3_encode": _e4m3_encode(ties="up")},
    "e4m3_ties_towards_zero": {"e4m3_encode": _e4m3_encode(ties="down")},
    "e4m3_no_saturation": {"e4m3_encode": _e4m3_encode(saturate=False)},
}


def _pin_cases():
    """Every pin of test_oracle_pins.py as a zero-argument call (parametrised
    pins with each of their parameter values)."""
    cases = []
    for name, fn in inspect.getmembers(pins, inspect.isfunction):
        if not name.startswith("test_") or name == "test_oracle_is_independent_of_the_cuda_path":
            continue
        marks = getattr(fn, "pytestmark", [])
        params = [m for m in marks if m.name == "parametrize"]
        if params:
            argname, values = params[0].args[0], params[0].args[1]
            cases += [(f"{name}[{v}]", lambda fn=fn, a=argname, v=v: fn(**{a: v})) for v in values]
        else:
            cases.append((name, fn))
    return cases


def test_every_pin_passes_on_the_unchanged_oracle():
    for name, call in _pin_cases():
        call()


@pytest.mark.parametrize("mutant", sorted(MUTANTS))
def test_planted_mistake_fails_a_pin(monkeypatch, mutant):
    for attr, fn in MUTANTS[mutant].items():
        assert hasattr(om, attr), attr
        monkeypatch.setattr(om, attr, fn)
        if hasattr(oracle, attr):
            monkeypatch.setattr(oracle, attr, fn)
    caught = []
    for name, call in _pin_cases():
        try:
            with np.errstate(all="ignore"):
                call()
        except Exception:   # a failed assertion, or an input the slip cannot handle
            caught.append(name)
            break
    assert caught, f"no pin fails when the oracle carries the slip '{mutant}'"

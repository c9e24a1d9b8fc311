"""fp64 CPU oracle: definitions of every step of the MLA latent-KV hot path.

TEST INFRASTRUCTURE ONLY (see the package docstring for who may call it).

Notation (the page "MLA 注意力与 KV 缓存", §2): H heads; per head a query of
qk_head = qk_nope + qk_rope values; the cache holds per token a latent
``Lc[t]`` of kv_lora values and a rotated key ``Rc[t]`` of qk_rope values
shared by all heads; ``kv_b [H, qk_nope + v_head, kv_lora]`` reconstructs the
per-head key part ``W_UK[h] = kv_b[h, :qk_nope]`` and value ``W_UV[h] =
kv_b[h, qk_nope:]``.

Readings of points the pages leave open:

* kv_b packing: per head, the qk_nope key rows first, then the v_head value
  rows (from kvb_dim = H*(qk_nope+v_head), §2).
* RoPE: pair j of the rope part is (x[2j], x[2j+1]); it rotates by
  pos * base^(-2j/qk_rope); the results go to y[j] and y[qk_rope/2 + j]
  (§2.1, rope_interleave).  Rc arrives already rotated.
* A call holds S new tokens whose cache rows are already written, so the
  query s of sequence b sits at pos = T[b] - S + s (Tk = pos_base + S, §2) and
  attends to keys t <= pos (causal, self included).
* softmax scale: 1/sqrt(qk_nope + qk_rope) unless given; plain softmax, no sink.
"""
from __future__ import annotations

import numpy as np

NEG_INF = -np.inf


def _f64(x):
    return np.asarray(x, dtype=np.float64)


# ---------------------------------------------------------------------------
# RoPE ([MLA-KV] §2.1: only the qk_rope tail rotates; even/odd pair (a, b)
# becomes v[j] = a*cs - b*sn, v[half+j] = b*cs + a*sn)
# ---------------------------------------------------------------------------
def rope_interleave(x, pos, base: float = 10000.0):
    """Rotate the last axis of ``x`` (length qk_rope, even) to position ``pos``.

    ``pos`` broadcasts against ``x[..., 0]``.  Angle of pair j:
    pos * base ** (-2j / qk_rope).
    """
    x = _f64(x)
    d = x.shape[-1]
    assert d % 2 == 0
    half = d // 2
    j = np.arange(half, dtype=np.float64)
    theta = base ** (-2.0 * j / d)
    ang = _f64(pos)[..., None] * theta
    cs, sn = np.cos(ang), np.sin(ang)
    a = x[..., 0::2]
    b = x[..., 1::2]
    y = np.empty_like(x)
    y[..., :half] = a * cs - b * sn
    y[..., half:] = b * cs + a * sn
    return y


def split_kv_b(kv_b, qk_nope: int):
    """kv_b [H, qk_nope+v_head, kv_lora] -> (W_UK [H,qk_nope,kv_lora], W_UV [H,v_head,kv_lora])."""
    kv_b = _f64(kv_b)
    return kv_b[:, :qk_nope, :], kv_b[:, qk_nope:, :]


def softmax_probs(scores):
    """Plain softmax over the last axis with max subtraction; -inf entries get 0."""
    s = _f64(scores)
    m = np.max(s, axis=-1, keepdims=True)
    e = np.exp(s - m)
    return e / np.sum(e, axis=-1, keepdims=True)


def query_positions(T_b: int, S: int):
    """Positions of the S new query tokens of a sequence whose cache holds T_b rows."""
    return [T_b - S + s for s in range(S)]


# ---------------------------------------------------------------------------
# One query token against a set of cached rows (all given rows are attended)
# ---------------------------------------------------------------------------
def attend_dense(q, Lc_rows, Rc_rows, kv_b, qk_nope: int, pos, scale: float,
                 rope_base: float = 10000.0):
    """Definition: plain multi-head attention over keys/values rebuilt from the latent.

    q [H, qk_nope+qk_rope] (pre-RoPE), Lc_rows [n, kv_lora], Rc_rows [n, qk_rope].
    k[t,h] = [W_UK[h] Lc[t] ; Rc[t]], v[t,h] = W_UV[h] Lc[t] ([MLA-KV] §1: k_nope
    and value are rebuilt from the latent through kv_b at attention time).
    Returns out [H, v_head].
    """
    q = _f64(q)
    L = _f64(Lc_rows)
    R = _f64(Rc_rows)
    W_UK, W_UV = split_kv_b(kv_b, qk_nope)
    k_nope = np.einsum("hil,tl->thi", W_UK, L)          # [n, H, qk_nope]
    v = np.einsum("hjl,tl->thj", W_UV, L)               # [n, H, v_head]
    q_nope = q[:, :qk_nope]
    q_rot = rope_interleave(q[:, qk_nope:], pos, rope_base)
    scores = scale * (np.einsum("hi,thi->ht", q_nope, k_nope) + np.einsum("hr,tr->ht", q_rot, R))
    p = softmax_probs(scores)                            # [H, n]
    return np.einsum("ht,thj->hj", p, v)


def attend_absorbed(q, Lc_rows, Rc_rows, kv_b, qk_nope: int, pos, scale: float,
                    rope_base: float = 10000.0, return_probs: bool = False):
    """Weight-absorbed attention ([MLA-KV] §2.3, absorbed path).

    qabs[h] = sum_i q_nope[h,i] W_UK[h,i,:] (qt_addrow); score_t =
    scale*(qabs . Lc[t] + q_rot . Rc[t]); clat = sum_t p_t Lc[t];
    out[h] = W_UV[h] clat (qt_matvec_rows).
    """
    q = _f64(q)
    L = _f64(Lc_rows)
    R = _f64(Rc_rows)
    W_UK, W_UV = split_kv_b(kv_b, qk_nope)
    qabs = np.einsum("hi,hil->hl", q[:, :qk_nope], W_UK)      # [H, kv_lora]
    q_rot = rope_interleave(q[:, qk_nope:], pos, rope_base)    # [H, qk_rope]
    scores = scale * (qabs @ L.T + q_rot @ R.T)                # [H, n]
    p = softmax_probs(scores)
    clat = p @ L                                               # [H, kv_lora]
    out = np.einsum("hjl,hl->hj", W_UV, clat)
    if return_probs:
        return out, p
    return out


# ---------------------------------------------------------------------------
# Batched decode: causal rule applied per query
# ---------------------------------------------------------------------------
def _decode(attend, q, Lc, Rc, T, kv_b, qk_nope, scale, rope_base, rows=None):
    q = np.asarray(q)
    B, S, H = q.shape[0], q.shape[1], q.shape[2]
    v_head = np.asarray(kv_b).shape[1] - qk_nope
    out = np.full((B, S, H, v_head), np.nan)
    for b in range(B):
        for s, pos in enumerate(query_positions(int(T[b]), S)):
            if rows is not None and (b, s) not in rows:
                continue
            out[b, s] = attend(q[b, s], Lc[b, :pos + 1], Rc[b, :pos + 1], kv_b, qk_nope,
                               pos, scale, rope_base)
    return out


def decode_dense(q, Lc, Rc, T, kv_b, qk_nope, scale, rope_base=10000.0, rows=None):
    """Dense MHA decode for q [B,S,H,qk_head], caches [B,T_cap,.], T [B]."""
    return _decode(attend_dense, q, Lc, Rc, T, kv_b, qk_nope, scale, rope_base, rows)


def decode_absorbed(q, Lc, Rc, T, kv_b, qk_nope, scale, rope_base=10000.0, rows=None):
    """Absorbed decode for q [B,S,H,qk_head]; ``rows`` optionally limits the (b, s) pairs."""
    return _decode(attend_absorbed, q, Lc, Rc, T, kv_b, qk_nope, scale, rope_base, rows)


# ---------------------------------------------------------------------------
# Non-absorbed prefill ([MLA-KV] §2.3, non-absorbed path)
# ---------------------------------------------------------------------------
def prefill_nonabsorbed(q, Lc, Rc, kv_b, qk_nope, scale, pos_base, rope_base=10000.0,
                        queries=None, heads=None):
    """q [S,H,qk_head] at positions pos_base+s against Lc/Rc [Tk,.], Tk = pos_base+S.

    Step 1 (one kv_b matrix product for all Tk keys): KV[t,h,:] = kv_b[h] Lc[t],
    giving k_nope = KV[..., :qk_nope] and value = KV[..., qk_nope:].
    Step 2 (causal attention): score = scale*(q_pass . k_nope[t] + q_rot . Rc[t]) for
    t <= pos, softmax, sum of p * value.
    ``queries``/``heads`` optionally restrict which outputs are computed (the
    rest stay NaN).  Returns out [S,H,v_head].
    """
    q = _f64(q)
    S, H = q.shape[0], q.shape[1]
    kvb = _f64(kv_b)
    Tk = pos_base + S
    L = _f64(Lc)[:Tk]
    R = _f64(Rc)[:Tk]
    heads = list(range(H)) if heads is None else list(heads)
    queries = list(range(S)) if queries is None else list(queries)
    KV = np.einsum("hjl,tl->thj", kvb[heads], L)          # [Tk, |heads|, qk_nope+v_head]
    k_nope = KV[..., :qk_nope]
    value = KV[..., qk_nope:]
    v_head = kvb.shape[1] - qk_nope
    out = np.full((S, H, v_head), np.nan)
    for s in queries:
        pos = pos_base + s
        q_pass = q[s, heads, :qk_nope]
        q_rot = rope_interleave(q[s, heads, qk_nope:], pos, rope_base)
        sc = scale * (np.einsum("hi,thi->ht", q_pass, k_nope[:pos + 1])
                      + q_rot @ R[:pos + 1].T)
        p = softmax_probs(sc)
        out[s, heads] = np.einsum("ht,thj->hj", p, value[:pos + 1])
    return out


# ---------------------------------------------------------------------------
# DSA lightning indexer and causal top-k ([MLA-KV] §2.2)
# ---------------------------------------------------------------------------
def index_scores(q_idx, w, Ic, T, S_positions=None):
    """I[b,s,t] = sum_h w[b,s,h] * max(0, q_idx[b,s,h] . Ic[b,t]) for t <= pos, else -inf.

    q_idx [B,S,n_ih,index_hd], w [B,S,n_ih], Ic [B,T_cap,index_hd] (fp32 per
    token, [FDSA] §二), T [B].  No extra scale (none is printed).
    Returns [B,S,T_cap] float64.
    """
    qi = _f64(q_idx)
    ww = _f64(w)
    B, S = qi.shape[0], qi.shape[1]
    T_cap = np.asarray(Ic).shape[1]
    out = np.full((B, S, T_cap), NEG_INF)
    for b in range(B):
        for s, pos in enumerate(query_positions(int(T[b]), S)):
            K = _f64(np.asarray(Ic)[b, :pos + 1])                  # [n, hd]
            dots = qi[b, s] @ K.T                                   # [n_ih, n]
            out[b, s, :pos + 1] = ww[b, s] @ np.maximum(dots, 0.0)
    return out


def topk_select(scores, T, S: int, k: int):
    """Causal top-k key selection for every (b, s).

    Candidates are t in [0, pos]; with at most k of them all are kept (the
    indexer only prunes once the context exceeds index_topk).  Otherwise keys
    are ordered by (score descending, index ascending) -- the lower index wins
    ties, and -0.0 equals +0.0 -- and the first k are kept.  Output indices are
    ascending, padded with -1: sel [B,S,k] int64, nsel [B,S] int64.
    """
    sc = np.asarray(scores)
    B = sc.shape[0]
    sel = np.full((B, S, k), -1, dtype=np.int64)
    nsel = np.zeros((B, S), dtype=np.int64)
    for b in range(B):
        for s, pos in enumerate(query_positions(int(T[b]), S)):
            n = pos + 1
            idx = np.arange(n)
            if n <= k:
                keep = idx
            else:
                vals = _f64(sc[b, s, :n])
                order = np.lexsort((idx, -vals))   # primary: -score asc; secondary: index asc
                keep = np.sort(order[:k])
            sel[b, s, :len(keep)] = keep
            nsel[b, s] = len(keep)
    return sel, nsel


def sparse_decode(q, Lc, Rc, T, kv_b, sel, nsel, qk_nope, scale, rope_base=10000.0, rows=None):
    """Absorbed decode restricted to the selected keys sel[b,s,:nsel[b,s]].

    The selection of a query is shared by all heads ([MLA-KV] §2.2: later layers
    reuse ``dsa_sel``).  Selected indices must be <= pos.
    """
    q = np.asarray(q)
    B, S, H = q.shape[0], q.shape[1], q.shape[2]
    v_head = np.asarray(kv_b).shape[1] - qk_nope
    out = np.full((B, S, H, v_head), np.nan)
    for b in range(B):
        for s, pos in enumerate(query_positions(int(T[b]), S)):
            if rows is not None and (b, s) not in rows:
                continue
            idx = np.asarray(sel[b, s, :int(nsel[b, s])], dtype=np.int64)
            assert idx.size > 0 and idx.max() <= pos and idx.min() >= 0
            out[b, s] = attend_absorbed(q[b, s], np.asarray(Lc)[b, idx], np.asarray(Rc)[b, idx],
                                        kv_b, qk_nope, pos, scale, rope_base)
    return out


# ---------------------------------------------------------------------------
# Cache append ([MLA-KV] §2.1, KV path: the kv_a output comp[kv_lora + qk_rope]
# of each new token -> the first kv_lora values through RMSNorm(kv_a_ln) into
# Lc[pos], the last qk_rope values through the RoPE shared by all heads into
# Rc[pos]; [MLA-KV] §2.2: the indexer key through LayerNorm (eps 1e-6) and
# RoPE into Ic[pos]).
# ---------------------------------------------------------------------------
def rms_norm(x, w, eps: float):
    """x / sqrt(mean(x^2) + eps) * w over the last axis.  The pages print no
    eps for kv_a_ln: the caller passes it."""
    x = _f64(x)
    return x / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps) * _f64(w)


def layer_norm(x, w, b, eps: float = 1e-6):
    """(x - mean) / sqrt(var + eps) * w + b over the last axis (biased variance).
    Reading: the indexer's "layernorm" has a weight and a bias (b may be None)."""
    x = _f64(x)
    mu = np.mean(x, axis=-1, keepdims=True)
    var = np.mean((x - mu) ** 2, axis=-1, keepdims=True)
    y = (x - mu) / np.sqrt(var + eps) * _f64(w)
    return y if b is None else y + _f64(b)


def new_token_positions(T, S: int):
    """[B, S] cache rows of the S new tokens of each sequence: T[b] - S + s."""
    T = np.asarray(T, dtype=np.int64)
    return T[:, None] - S + np.arange(S)[None, :]


def cache_append(comp, kv_a_ln, eps: float, T, kv_lora: int, base: float = 10000.0):
    """comp [B,S,kv_lora+qk_rope] -> (Lc rows [B,S,kv_lora], Rc rows [B,S,qk_rope],
    positions [B,S]) for the new tokens at pos = T[b] - S + s."""
    comp = _f64(comp)
    S = comp.shape[1]
    pos = new_token_positions(T, S)
    lc = rms_norm(comp[..., :kv_lora], kv_a_ln, eps)
    rc = rope_interleave(comp[..., kv_lora:], pos, base)
    return lc, rc, pos


def index_key_append(k_idx, ln_w, ln_b, eps: float, T, rope_dim: int, base: float = 10000.0):
    """k_idx [B,S,index_hd] -> (Ic rows [B,S,index_hd], positions [B,S]): LayerNorm,
    then the interleaved RoPE on the last rope_dim values (reading: the page
    names LayerNorm and RoPE but not which values rotate; the same tail
    rotation as the attention key is taken)."""
    k = layer_norm(k_idx, ln_w, ln_b, eps)
    S = k.shape[1]
    pos = new_token_positions(T, S)
    if rope_dim > 0:
        k = k.copy()
        k[..., k.shape[-1] - rope_dim:] = rope_interleave(k[..., k.shape[-1] - rope_dim:], pos, base)
    return k, pos


# --------------------------------------------------------------- paged cache layout
def page_row(block_table, b: int, t: int, page_size: int) -> int:
    """Pool row of token t of sequence b: the page that the block table names
    for t // page_size, row t % page_size inside it.  The pages fix no storage
    layout beyond one row per token ([MLA-KV] §1); this is the paged layout's
    own definition."""
    return int(block_table[b][t // page_size]) * page_size + t % page_size


def unpage(pool, block_table, T):
    """[num_pages, page_size, D] pool -> contiguous [B, max(T), D] cache whose
    rows 0..T[b]-1 of sequence b are read through page_row; the rest are NaN."""
    pool = _f64(pool)
    page_size, D = pool.shape[1], pool.shape[2]
    rows = pool.reshape(-1, D)
    out = np.full((len(T), max(T), D), np.nan)
    for b, n in enumerate(T):
        for t in range(n):
            out[b, t] = rows[page_row(block_table, b, t, page_size)]
    return out


# --------------------------------------------------------------- output projection
def o_proj(x, w_o):
    """y[r, n] = sum_k w_o[n, k] x[r, k]: the o output projection that ends both
    attention paths ([MLA-KV] §2.3), x [R, in_dim] (a decode output flattened
    per row), w_o [hidden, in_dim]."""
    return _f64(x) @ _f64(w_o).T


# --------------------------------------------------------------- FP8 latent cache
# The pages fix no cache quantisation (FP8 appears among the weight formats
# only); this is the FP8 cache format's own definition.  The latent part of a
# row is stored as kv_lora E4M3 codes with one dequantisation scale for the
# whole cache, Lc[t] = lat_scale * e4m3(code[t]); the rotated key Rc stays
# 16-bit.  E4M3 here is the OCP 8-bit format without infinities: 1 sign bit,
# 4 exponent bits with bias 7, 3 mantissa bits; exponent field 0 holds the
# subnormals M * 2^-9; S.1111.111 is NaN; the largest finite value is 448.
def e4m3_decode(codes):
    """uint8 codes -> float64 values (NaN for the two NaN codes)."""
    c = np.asarray(codes, dtype=np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    E = (c >> 3) & 0xF
    M = (c & 0x7).astype(np.float64)
    mag = np.where(E == 0, M * 2.0 ** -9, (1.0 + M / 8.0) * 2.0 ** (E - 7.0))
    mag = np.where((E == 15) & (M == 7), np.nan, mag)
    return sign * mag


def e4m3_encode(x):
    """float -> uint8 code of the nearest E4M3 value, ties to the even code,
    magnitudes past 448 saturated to 448, NaN to 0x7F.  The nearest value is
    found among all 127 non-negative finite values, as the definition reads."""
    x = _f64(x)
    grid = e4m3_decode(np.arange(127))             # 0x00 .. 0x7E, increasing
    a = np.minimum(np.abs(x), 448.0)
    hi = np.clip(np.searchsorted(grid, a, side="left"), 0, 126)
    lo = np.maximum(hi - 1, 0)
    dlo, dhi = a - grid[lo], grid[hi] - a
    pick = np.where(dlo < dhi, lo, np.where(dhi < dlo, hi, np.where(lo % 2 == 0, lo, hi)))
    code = pick.astype(np.int64) | np.where(np.signbit(x), 0x80, 0)
    return np.where(np.isnan(x), 0x7F, code).astype(np.uint8)


def dequant_latent(codes, lat_scale: float):
    """Latent rows of an FP8 cache: lat_scale * e4m3(code)."""
    return float(lat_scale) * e4m3_decode(codes)


def cache_append_fp8(comp, kv_a_ln, eps: float, T, kv_lora: int, lat_scale: float, base: float = 10000.0):
    """cache_append into the FP8 format: the RMSNorm output divided by
    lat_scale is rounded to E4M3 codes; Rc as in cache_append.
    Returns (codes [B,S,kv_lora] uint8, rc [B,S,qk_rope], pos [B,S])."""
    lc, rc, pos = cache_append(comp, kv_a_ln, eps, T, kv_lora, base)
    return e4m3_encode(lc / float(lat_scale)), rc, pos

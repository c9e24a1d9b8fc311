"""GPU parity of every C ABI entry point against the fp64 oracle.

Tolerances (normwise max relative error, max|gpu - oracle| / max|oracle|):
fp32 inputs 1e-5, bf16 inputs 2e-2.  DSA scores and the selected index sets
are compared bit for bit.  Inputs come from workload/ (NaN past each
sequence's end, so a read out of range shows up as a NaN output).
"""
import numpy as np
import pytest
import torch

import oracle
from tests._np import check_close, max_rel_err, to_np
from workload import GLM, TINY, WORKLOADS, dsa_inputs, mla_inputs, workload_inputs

pytestmark = pytest.mark.gpu

TOL = {"f32": 1e-5, "bf16": 2e-2}
DEV = "cuda:0"


def _dev(x):
    return {k: (v.to(DEV) if isinstance(v, torch.Tensor) else v) for k, v in x.items()}


def _np_inputs(x):
    return {k: to_np(x[k]) for k in ("q", "Lc", "Rc", "kv_b")}


# --------------------------------------------------------------- absorbed decode
def test_tiny_workload_decode(cuda_lib):
    x = workload_inputs("tiny", "cpu")
    g = _dev(x)
    out = cuda_lib.decode_absorbed(g["q"], g["Lc"], g["Rc"], g["T"], g["kv_b"], TINY)
    n = _np_inputs(x)
    ref = oracle.decode_dense(n["q"], n["Lc"], n["Rc"], x["T_list"], n["kv_b"], TINY.qk_nope,
                              TINY.softmax_scale)
    check_close(to_np(out), ref, TOL["f32"])


@pytest.mark.parametrize("dtype,dims", [("f32", TINY), ("bf16", GLM), ("f32", GLM)])
@pytest.mark.parametrize("T,S", [([1], 1), ([6], 6), ([129, 300, 64], 1), ([130, 257, 6], 6),
                                 ([1000], 2)])
def test_decode_ragged(cuda_lib, dtype, dims, T, S):
    T_cap = max(T) + 37
    x = mla_inputs(dims, len(T), S, T, T_cap, dtype, 100 + sum(T) + S, "cpu")
    g = _dev(x)
    out = cuda_lib.decode_absorbed(g["q"], g["Lc"], g["Rc"], g["T"], g["kv_b"], dims)
    n = _np_inputs(x)
    ref = oracle.decode_absorbed(n["q"], n["Lc"], n["Rc"], T, n["kv_b"], dims.qk_nope, dims.softmax_scale)
    got = to_np(out)
    assert np.all(np.isfinite(got))
    check_close(got, ref, TOL[dtype])
    assert cuda_lib.device_status() == 0


@pytest.mark.parametrize("T,S", [([128 * 152 * 2], 1), ([128 * 152 * 2 + 77], 1), ([40000], 1),
                                 ([3000, 5000, 129, 7000], 2)])
def test_decode_several_tiles_per_cta(cuda_lib, T, S):
    """Long sequences: every persistent CTA runs several key tiles and, for B > 1,
    several sequences, so the split pipeline crosses tile and sequence borders."""
    x = mla_inputs(GLM, len(T), S, T, max(T), "bf16", 11, DEV)
    out = to_np(cuda_lib.decode_absorbed(x["q"], x["Lc"], x["Rc"], x["T"], x["kv_b"], GLM))
    assert cuda_lib.device_status() == 0
    kvb = to_np(x["kv_b"])
    for b in range(len(T)):
        for s in range(S):
            pos = T[b] - S + s
            ref = oracle.attend_absorbed(to_np(x["q"][b, s]), to_np(x["Lc"][b, :pos + 1]),
                                         to_np(x["Rc"][b, :pos + 1]), kvb, GLM.qk_nope, pos, GLM.softmax_scale)
            check_close(out[b, s], ref, TOL["bf16"], (b, s))


def test_decode_glm_t4096_full(cuda_lib):
    """The GLM-5.2 single-sequence workload at full size (B=1, S=1, T=4096), every output."""
    x = workload_inputs("glm_decode_t4096", DEV)
    out = cuda_lib.decode_absorbed(x["q"], x["Lc"], x["Rc"], x["T"], x["kv_b"], GLM)
    n = _np_inputs(x)
    ref = oracle.decode_absorbed(n["q"], n["Lc"], n["Rc"], x["T_list"], n["kv_b"], GLM.qk_nope,
                                 GLM.softmax_scale)
    check_close(to_np(out), ref, TOL["bf16"])


@pytest.mark.parametrize("S", [1, 6])
def test_decode_batched_b32_every_row(cuda_lib, S):
    """B=32, T_b ~ U{1024..32768} at T_cap=32768: every (b, s) row against the
    oracle, the cache of each sequence widened to fp64 once."""
    x = workload_inputs("glm_batched_b32", DEV, S=S)
    out = to_np(cuda_lib.decode_absorbed(x["q"], x["Lc"], x["Rc"], x["T"], x["kv_b"], GLM))
    assert np.all(np.isfinite(out))
    assert cuda_lib.device_status() == 0
    T = x["T_list"]
    kvb = to_np(x["kv_b"])
    for b in range(len(T)):
        L = to_np(x["Lc"][b, :T[b]])
        R = to_np(x["Rc"][b, :T[b]])
        q = to_np(x["q"][b])
        for s in range(S):
            pos = T[b] - S + s
            ref = oracle.attend_absorbed(q[s], L[:pos + 1], R[:pos + 1], kvb, GLM.qk_nope, pos,
                                         GLM.softmax_scale)
            check_close(out[b, s], ref, TOL["bf16"], (b, s))


def test_decode_flags_bad_length(cuda_lib):
    T = [40, 10]
    x = mla_inputs(GLM, 2, 1, T, 40, "bf16", 5, "cpu")
    g = _dev(x)
    g["T"] = torch.tensor([40, 41], dtype=torch.int32, device=DEV)  # 41 > T_cap
    out = cuda_lib.decode_absorbed(g["q"], g["Lc"], g["Rc"], g["T"], g["kv_b"], GLM)
    flags = cuda_lib.device_status()
    assert flags & cuda_lib.MLA_DEV_BAD_LENGTH
    got = to_np(out)
    assert np.all(np.isnan(got[1])) and np.all(np.isfinite(got[0]))
    assert cuda_lib.device_status() == 0  # cleared by the previous read


# --------------------------------------------------------------- DSA
@pytest.mark.parametrize("T,S,nh,hd,k", [([64], 1, 2, 8, 16), ([300, 17, 1000], 2, 4, 32, 64),
                                         ([2048, 2049, 5000], 1, 32, 128, 2048)])
def test_index_and_topk_bit_exact(cuda_lib, T, S, nh, hd, k):
    T_cap = max(T) + 5
    d = dsa_inputs(len(T), S, T, T_cap, nh, hd, 40 + sum(T), "cpu")
    g = _dev(d)
    Tt = torch.tensor(T, dtype=torch.int32, device=DEV)
    sc = cuda_lib.index_scores(g["q_idx"], g["w"], g["Ic"], Tt)
    ref = oracle.index_scores(to_np(d["q_idx"]), to_np(d["w"]), to_np(d["Ic"]), T)
    got = to_np(sc)
    assert np.array_equal(got, ref)
    sel, nsel = cuda_lib.topk_select(sc, Tt, k)
    rsel, rn = oracle.topk_select(ref, T, S, k)
    assert np.array_equal(nsel.cpu().numpy(), rn)
    assert np.array_equal(sel.cpu().numpy(), rsel)


@pytest.mark.parametrize("T,S,nh,hd", [([3000, 517, 129], 2, 32, 128), ([70000], 1, 32, 128), ([1000, 300], 1, 4, 32)])
def test_index_scores_general_floats(cuda_lib, T, S, nh, hd):
    """Non-integer fp32 indexer inputs: scores within 1e-5 (normwise) of the fp64
    definition, -inf exactly past each query's position.  32 heads x 128 run
    on the tensor cores (three tf32 products), other shapes on the CUDA cores."""
    r = np.random.default_rng(11)
    B, T_cap = len(T), max(T) + 45
    q = r.standard_normal((B, S, nh, hd)).astype(np.float32)
    w = r.standard_normal((B, S, nh)).astype(np.float32)
    Ic = r.standard_normal((B, T_cap, hd)).astype(np.float32)
    for b, t in enumerate(T):
        Ic[b, t:] = np.nan
    Tt = torch.tensor(T, dtype=torch.int32, device=DEV)
    sc = to_np(cuda_lib.index_scores(*(torch.from_numpy(x).to(DEV) for x in (q, w, Ic)), Tt))
    ref = oracle.index_scores(q.astype(np.float64), w.astype(np.float64), Ic.astype(np.float64), T)
    fin = np.isfinite(ref)
    assert np.array_equal(np.isneginf(sc), np.isneginf(ref)) and np.all(np.isfinite(sc[fin]))
    assert max_rel_err(sc[fin], ref[fin]) < 1e-5
    assert cuda_lib.device_status() == 0


@pytest.mark.parametrize("frac_q,frac_tiles", [(False, (3, 7)), (True, ()), (True, (0, 5))])
def test_index_scores_mixed_exact_tiles(cuda_lib, frac_q, frac_tiles):
    """Integer-valued keys except for the listed 128-key tiles, whose keys get a
    fraction, and an integer or a fractional query: tiles without low bits skip
    the third tf32 product, an exact query skips the second; every score stays
    within 1e-5 (normwise) of the fp64 definition, and exactly equal where all
    inputs are integers."""
    r = np.random.default_rng(17)
    T, S, nh, hd = [1100, 700], 1, 32, 128
    B, T_cap = len(T), max(T) + 30
    q = r.integers(-4, 5, (B, S, nh, hd)).astype(np.float32)
    if frac_q:
        q += (r.random(q.shape) * 0.5).astype(np.float32)
    w = r.integers(-4, 5, (B, S, nh)).astype(np.float32)
    Ic = r.integers(-4, 5, (B, T_cap, hd)).astype(np.float32)
    for t in frac_tiles:
        Ic[:, 128 * t:128 * (t + 1)] += np.float32(1.0 / 3.0)
    for b, t in enumerate(T):
        Ic[b, t:] = np.nan
    Tt = torch.tensor(T, dtype=torch.int32, device=DEV)
    sc = to_np(cuda_lib.index_scores(*(torch.from_numpy(x).to(DEV) for x in (q, w, Ic)), Tt))
    ref = oracle.index_scores(q.astype(np.float64), w.astype(np.float64), Ic.astype(np.float64), T)
    fin = np.isfinite(ref)
    assert np.array_equal(np.isneginf(sc), np.isneginf(ref)) and np.all(np.isfinite(sc[fin]))
    assert max_rel_err(sc[fin], ref[fin]) < 1e-5
    if not frac_q:  # integer query: the integer tiles are exact
        ints = np.ones(T_cap, dtype=bool)
        for t in frac_tiles:
            ints[128 * t:128 * (t + 1)] = False
        for b, t in enumerate(T):
            m = ints[:t]
            assert np.array_equal(sc[b, 0, :t][m], ref[b, 0, :t][m])
    assert cuda_lib.device_status() == 0


def test_index_scores_unaligned_query(cuda_lib):
    """A query tensor that starts 4 bytes past a 16-byte boundary takes the
    CUDA-core indexer (the tensor-core one loads it in 16-byte vectors): the
    scores stay bit-exact on integer inputs."""
    T, S = [700, 300], 1
    d = dsa_inputs(2, S, T, max(T), 32, 128, 77, "cpu")
    flat = torch.empty(d["q_idx"].numel() + 1, dtype=torch.float32, device=DEV)
    q = flat[1:].view(d["q_idx"].shape)
    q.copy_(d["q_idx"].to(DEV))
    assert q.data_ptr() % 16 == 4
    Tt = torch.tensor(T, dtype=torch.int32, device=DEV)
    sc = cuda_lib.index_scores(q, d["w"].to(DEV), d["Ic"].to(DEV), Tt)
    assert np.array_equal(to_np(sc), oracle.index_scores(to_np(d["q_idx"]), to_np(d["w"]), to_np(d["Ic"]), T))
    assert cuda_lib.device_status() == 0


def test_topk_ties_and_negative_zero(cuda_lib):
    """Many equal scores, +0.0 and -0.0 mixed: the lower index wins."""
    r = np.random.default_rng(3)
    B, S, T_cap, k = 2, 1, 5000, 700
    sc = r.integers(-2, 3, (B, S, T_cap)).astype(np.float32)
    sc[sc == 0] = np.where(r.random(np.sum(sc == 0)) < 0.5, -0.0, 0.0).astype(np.float32)
    T = [5000, 3001]
    g = torch.from_numpy(sc).to(DEV)
    sel, nsel = cuda_lib.topk_select(g, torch.tensor(T, dtype=torch.int32, device=DEV), k)
    rsel, rn = oracle.topk_select(sc.astype(np.float64), T, S, k)
    assert np.array_equal(sel.cpu().numpy(), rsel) and np.array_equal(nsel.cpu().numpy(), rn)


@pytest.mark.parametrize("lo,hi,T", [(1.0, 1.25, [40000, 39000]), (1.0, 1.25, [9000]), (-3.0, 5.0, [65536]),
                                     (1.0, 1.25, [140000, 2500]), (-3.0, 5.0, [140000])])
def test_topk_crowded_and_spread_scores(cuda_lib, lo, hi, T):
    """Scores in [1, 1.25) share their top 11 key bits (crowded radix bins).
    Rows up to 131072 keys run the cluster kernel; the 140000-key cases run
    the single-CTA kernel, whose crowded case overflows its in-smem candidate
    list and takes the fallback passes."""
    r = np.random.default_rng(9)
    T_cap = max(T)
    k = 2048
    sc = r.uniform(lo, hi, (len(T), 1, T_cap)).astype(np.float32)
    sc[0, 0, 100:140] = sc[0, 0, 7]  # exact ties across the threshold region
    g = torch.from_numpy(sc).to(DEV)
    Tt = torch.tensor(T, dtype=torch.int32, device=DEV)
    sel, nsel = cuda_lib.topk_select(g, Tt, k)
    rsel, rn = oracle.topk_select(sc.astype(np.float64), T, 1, k)
    assert np.array_equal(nsel.cpu().numpy(), rn)
    assert np.array_equal(sel.cpu().numpy(), rsel)


def test_dsa_glm_t65536_pipeline(cuda_lib):
    """B=4, T=65536: indexer and top-2048 bit-exact, sparse decode within 2e-2 on every output."""
    x = workload_inputs("glm_dsa_t65536", DEV)
    sc = cuda_lib.index_scores(x["q_idx"], x["w"], x["Ic"], x["T"])
    T = x["T_list"]
    ref_sc = oracle.index_scores(to_np(x["q_idx"]), to_np(x["w"]), to_np(x["Ic"]), T)
    assert np.array_equal(to_np(sc), ref_sc)
    sel, nsel = cuda_lib.topk_select(sc, x["T"], x["topk"])
    rsel, rn = oracle.topk_select(ref_sc, T, 1, x["topk"])
    assert np.array_equal(sel.cpu().numpy(), rsel) and np.array_equal(nsel.cpu().numpy(), rn)
    out = to_np(cuda_lib.sparse_decode(x["q"], x["Lc"], x["Rc"], x["T"], x["kv_b"], sel, nsel, GLM))
    kvb = to_np(x["kv_b"])
    for b in range(4):
        idx = rsel[b, 0]
        pos = T[b] - 1
        ref = oracle.attend_absorbed(to_np(x["q"][b, 0]), to_np(x["Lc"][b, idx]), to_np(x["Rc"][b, idx]),
                                     kvb, GLM.qk_nope, pos, GLM.softmax_scale)
        check_close(out[b, 0], ref, TOL["bf16"], b)


@pytest.mark.parametrize("T,S,nh,hd,k", [([65536, 9000, 2048, 2049], 1, 32, 128, 2048), ([3000, 517, 129], 2, 32, 128, 256),
                                          ([300, 17, 1000], 2, 4, 32, 64), ([130000], 1, 32, 128, 2048)])
def test_fused_select_bit_exact(cuda_lib, T, S, nh, hd, k):
    """dsa_select (indexer histograms feed the top-k's first radix pass) gives the
    oracle's scores and index sets bit for bit, and the same as the two calls."""
    T_cap = max(T) + 3
    d = dsa_inputs(len(T), S, T, T_cap, nh, hd, 200 + S + k, DEV)
    Tt = torch.tensor(T, dtype=torch.int32, device=DEV)
    sc, sel, nsel = cuda_lib.select(d["q_idx"], d["w"], d["Ic"], Tt, k)
    assert cuda_lib.device_status() == 0
    ref_sc = oracle.index_scores(to_np(d["q_idx"]), to_np(d["w"]), to_np(d["Ic"]), T)
    got = to_np(sc)
    for b, t in enumerate(T):  # rows past T_b are not defined by the indexer
        assert np.array_equal(got[b, :, :t], ref_sc[b, :, :t])
    rsel, rn = oracle.topk_select(ref_sc, T, S, k)
    assert np.array_equal(sel.cpu().numpy(), rsel) and np.array_equal(nsel.cpu().numpy(), rn)
    sel2, nsel2 = cuda_lib.topk_select(sc, Tt, k)
    assert torch.equal(sel, sel2) and torch.equal(nsel, nsel2)


def test_fused_select_crowded_scores(cuda_lib):
    """Scores crowded into few first-pass bins (keys and queries in {0, 1}): the
    histograms carry large counts and many ties at the threshold."""
    T, S, k = [40000, 33000], 1, 2048
    g = torch.Generator(device=DEV)
    g.manual_seed(5)
    q = torch.randint(0, 2, (2, S, 32, 128), generator=g, device=DEV, dtype=torch.int32).float()
    w = torch.randint(0, 2, (2, S, 32), generator=g, device=DEV, dtype=torch.int32).float()
    Ic = torch.randint(0, 2, (2, max(T), 128), generator=g, device=DEV, dtype=torch.int32).float()
    Tt = torch.tensor(T, dtype=torch.int32, device=DEV)
    sc, sel, nsel = cuda_lib.select(q, w, Ic, Tt, k)
    assert cuda_lib.device_status() == 0
    ref_sc = oracle.index_scores(to_np(q), to_np(w), to_np(Ic), T)
    rsel, rn = oracle.topk_select(ref_sc, T, S, k)
    assert np.array_equal(sel.cpu().numpy(), rsel) and np.array_equal(nsel.cpu().numpy(), rn)


def test_dsa_selection_shared_by_later_layers(cuda_lib):
    """One indexer pass and top-2048 selection serve the attention of several
    layers ([MLA-KV] §2.2: the shared layers reuse dsa_sel): each layer's
    sparse decode, with its own query, cache and kv_b, equals the oracle over
    the same selected keys."""
    T, S, k = [9000, 20000], 1, 2048
    d = dsa_inputs(2, S, T, max(T), 32, 128, 61, DEV)
    Tt = torch.tensor(T, dtype=torch.int32, device=DEV)
    sc = cuda_lib.index_scores(d["q_idx"], d["w"], d["Ic"], Tt)
    sel, nsel = cuda_lib.topk_select(sc, Tt, k)
    rsel, rn = oracle.topk_select(oracle.index_scores(to_np(d["q_idx"]), to_np(d["w"]), to_np(d["Ic"]), T), T, S, k)
    assert np.array_equal(sel.cpu().numpy(), rsel) and np.array_equal(nsel.cpu().numpy(), rn)
    for layer in range(3):
        x = mla_inputs(GLM, 2, S, T, max(T), "bf16", 70 + layer, DEV)
        out = to_np(cuda_lib.sparse_decode(x["q"], x["Lc"], x["Rc"], x["T"], x["kv_b"], sel, nsel, GLM))
        assert cuda_lib.device_status() == 0
        kvb = to_np(x["kv_b"])
        for b in range(2):
            idx = rsel[b, 0, :rn[b, 0]]
            ref = oracle.attend_absorbed(to_np(x["q"][b, 0]), to_np(x["Lc"][b, idx]), to_np(x["Rc"][b, idx]),
                                         kvb, GLM.qk_nope, T[b] - 1, GLM.softmax_scale)
            check_close(out[b, 0], ref, TOL["bf16"], (layer, b))


@pytest.mark.parametrize("dtype,dims,T,k,L", [("bf16", GLM, [9000, 20000], 2048, 3), ("bf16", GLM, [3000, 129], 512, 1),
                                               ("f32", TINY, [300, 41], 64, 3)])
def test_sparse_decode_layers_over_one_selection(cuda_lib, dtype, dims, T, k, L):
    """One call runs L layers' sparse decodes over one selection ([MLA-KV]
    §2.2): every layer equals the oracle over the selected keys, and equals a
    separate mla_sparse_decode of that layer bit for bit (later layers'
    gathers, launched early into alternating staging buffers, change no
    value)."""
    S = 1
    d = dsa_inputs(2, S, T, max(T), 32, 128, 63, DEV)
    Tt = torch.tensor(T, dtype=torch.int32, device=DEV)
    sel, nsel = cuda_lib.topk_select(cuda_lib.index_scores(d["q_idx"], d["w"], d["Ic"], Tt), Tt, k)
    rsel, rn = sel.cpu().numpy(), nsel.cpu().numpy()
    xs = [mla_inputs(dims, 2, S, T, max(T), dtype, 80 + layer, DEV) for layer in range(L)]
    layers = [(x["q"], x["Lc"], x["Rc"], x["kv_b"]) for x in xs]
    outs = cuda_lib.sparse_decode_layers(layers, Tt, sel, nsel, dims)
    assert cuda_lib.device_status() == 0
    for layer, (x, out) in enumerate(zip(xs, outs)):
        one = cuda_lib.sparse_decode(x["q"], x["Lc"], x["Rc"], Tt, x["kv_b"], sel, nsel, dims)
        assert torch.equal(out, one), layer
        kvb, o = to_np(x["kv_b"]), to_np(out)
        for b in range(2):
            idx = rsel[b, 0, :rn[b, 0]]
            ref = oracle.attend_absorbed(to_np(x["q"][b, 0]), to_np(x["Lc"][b, idx]), to_np(x["Rc"][b, idx]),
                                         kvb, dims.qk_nope, T[b] - 1, dims.softmax_scale)
            check_close(o[b, 0], ref, TOL[dtype], (layer, b))
    # with each layer's output projection ([MLA-KV] §2.3): o_proj of the oracle's sparse decode
    hidden = 640
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    g = torch.Generator(device="cpu").manual_seed(64)
    w_o = [(torch.randn(hidden, dims.H * dims.v_head, generator=g) * 0.02).to(tdt).to(DEV) for _ in range(L)]
    outs2, ys = cuda_lib.sparse_decode_layers(layers, Tt, sel, nsel, dims, w_o=w_o)
    assert cuda_lib.device_status() == 0
    for layer, (x, out2, y) in enumerate(zip(xs, outs2, ys)):
        assert torch.equal(out2, outs[layer]), layer
        att = oracle.sparse_decode(to_np(x["q"]), to_np(x["Lc"]), to_np(x["Rc"]), T, to_np(x["kv_b"]), rsel, rn,
                                   dims.qk_nope, dims.softmax_scale)
        ref = oracle.o_proj(att.reshape(2 * S, -1), to_np(w_o[layer]))
        assert max_rel_err(to_np(y), ref) < (2e-2 if dtype == "bf16" else 1e-5), layer


@pytest.mark.parametrize("dtype,dims", [("f32", TINY), ("bf16", GLM)])
def test_sparse_decode_keep_all_and_subset(cuda_lib, dtype, dims):
    T = [50, 300]
    S, k = 2, 256
    x = mla_inputs(dims, 2, S, T, 320, dtype, 77, "cpu")
    g = _dev(x)
    n = _np_inputs(x)
    r = np.random.default_rng(5)
    sel = np.full((2, S, k), -1, dtype=np.int32)
    nsel = np.zeros((2, S), dtype=np.int32)
    for b in range(2):
        for s in range(S):
            pos = T[b] - S + s
            cnt = min(pos + 1, k)
            sel[b, s, :cnt] = np.sort(r.choice(pos + 1, cnt, replace=False))
            nsel[b, s] = cnt
    out = cuda_lib.sparse_decode(g["q"], g["Lc"], g["Rc"], g["T"], g["kv_b"],
                                 torch.from_numpy(sel).to(DEV), torch.from_numpy(nsel).to(DEV), dims)
    ref = oracle.sparse_decode(n["q"], n["Lc"], n["Rc"], T, n["kv_b"], sel, nsel, dims.qk_nope,
                               dims.softmax_scale)
    check_close(to_np(out), ref, TOL[dtype])
    # keep-all selection reproduces dense decode
    dense = oracle.decode_absorbed(n["q"], n["Lc"], n["Rc"], [50, 300], n["kv_b"], dims.qk_nope,
                                   dims.softmax_scale)
    assert max_rel_err(ref[0], dense[0]) < 1e-12


def test_decode_more_sequences_than_the_in_kernel_plan(cuda_lib):
    """1100 sequences (above the 1024 tile-list rows an attention CTA plans by
    itself, so it reads the absorb kernel's plan), 1..200 keys each; a sample
    of rows against the oracle."""
    B = 1100
    r = np.random.default_rng(21)
    T = [int(t) for t in r.integers(1, 201, B)]
    x = mla_inputs(GLM, B, 1, T, 200, "bf16", 22, "cpu")
    g = _dev(x)
    out = to_np(cuda_lib.decode_absorbed(g["q"], g["Lc"], g["Rc"], g["T"], g["kv_b"], GLM))
    assert cuda_lib.device_status() == 0
    kvb = to_np(x["kv_b"])
    for b in (0, 1, 517, 1023, 1024, 1099):
        ref = oracle.decode_absorbed(to_np(x["q"][b:b + 1]), to_np(x["Lc"][b:b + 1]), to_np(x["Rc"][b:b + 1]), [T[b]],
                                     kvb, GLM.qk_nope, GLM.softmax_scale)
        check_close(out[b], ref[0], TOL["bf16"], b)


def test_sparse_decode_more_rows_than_the_in_kernel_plan(cuda_lib):
    """520 sequences x 2 query tokens = 1040 selection rows (above 1024)."""
    B, S, k = 520, 2, 16
    r = np.random.default_rng(23)
    T = [int(t) for t in r.integers(S, 61, B)]
    x = mla_inputs(GLM, B, S, T, 60, "bf16", 24, "cpu")
    g = _dev(x)
    sel = np.full((B, S, k), -1, dtype=np.int32)
    nsel = np.zeros((B, S), dtype=np.int32)
    for b in range(B):
        for s in range(S):
            pos = T[b] - S + s
            cnt = min(pos + 1, k)
            sel[b, s, :cnt] = np.sort(r.choice(pos + 1, cnt, replace=False))
            nsel[b, s] = cnt
    out = to_np(cuda_lib.sparse_decode(g["q"], g["Lc"], g["Rc"], g["T"], g["kv_b"], torch.from_numpy(sel).to(DEV),
                                       torch.from_numpy(nsel).to(DEV), GLM))
    assert cuda_lib.device_status() == 0
    kvb = to_np(x["kv_b"])
    for b in (0, 300, 511, 512, 519):
        ref = oracle.sparse_decode(to_np(x["q"][b:b + 1]), to_np(x["Lc"][b:b + 1]), to_np(x["Rc"][b:b + 1]), [T[b]],
                                   kvb, sel[b:b + 1], nsel[b:b + 1], GLM.qk_nope, GLM.softmax_scale)
        check_close(out[b], ref[0], TOL["bf16"], b)


def test_sparse_decode_unsorted_ragged_selection(cuda_lib):
    """Selections in any order, with repeated keys, and counts that end
    mid-tile and mid-gather-group (301, 129, 3 of topk 512): each selected
    entry is one key of the softmax, as in the oracle."""
    T, k = [5000, 700, 3], 512
    x = mla_inputs(GLM, 3, 1, T, max(T), "bf16", 90, "cpu")
    g = _dev(x)
    r = np.random.default_rng(91)
    sel = np.zeros((3, 1, k), dtype=np.int32)
    nsel = np.array([[301], [129], [3]], dtype=np.int32)
    for b in range(3):
        n = int(nsel[b, 0])
        sel[b, 0, :n] = r.integers(0, T[b], n)  # unsorted, repeats allowed
    out = to_np(cuda_lib.sparse_decode(g["q"], g["Lc"], g["Rc"], g["T"], g["kv_b"], torch.from_numpy(sel).to(DEV),
                                       torch.from_numpy(nsel).to(DEV), GLM))
    assert cuda_lib.device_status() == 0
    ref = oracle.sparse_decode(to_np(x["q"]), to_np(x["Lc"]), to_np(x["Rc"]), T, to_np(x["kv_b"]), sel, nsel,
                               GLM.qk_nope, GLM.softmax_scale)
    check_close(out, ref, TOL["bf16"])


def test_sparse_decode_flags_future_index(cuda_lib):
    T = [100]
    x = mla_inputs(GLM, 1, 1, T, 100, "bf16", 8, "cpu")
    g = _dev(x)
    sel = torch.tensor([[[0, 5, 100, -1]]], dtype=torch.int32, device=DEV)  # 100 > pos=99
    nsel = torch.tensor([[3]], dtype=torch.int32, device=DEV)
    out = cuda_lib.sparse_decode(g["q"], g["Lc"], g["Rc"], g["T"], g["kv_b"], sel, nsel, GLM)
    assert cuda_lib.device_status() & cuda_lib.MLA_DEV_BAD_INDEX
    assert np.all(np.isnan(to_np(out)))


# --------------------------------------------------------------- prefill
@pytest.mark.parametrize("dtype,dims,S,pos_base", [("f32", TINY, 6, 10), ("f32", TINY, 16, 0),
                                                   ("bf16", GLM, 16, 200), ("bf16", GLM, 130, 77)])
def test_prefill_naive(cuda_lib, dtype, dims, S, pos_base):
    Tk = pos_base + S
    x = mla_inputs(dims, 1, S, [Tk], Tk, dtype, 60 + S, "cpu")
    g = _dev(x)
    out = cuda_lib.prefill_naive(g["q"], g["Lc"], g["Rc"], g["kv_b"], dims, pos_base)
    n = _np_inputs(x)
    ref = oracle.prefill_nonabsorbed(n["q"][0], n["Lc"][0], n["Rc"][0], n["kv_b"], dims.qk_nope,
                                     dims.softmax_scale, pos_base)
    check_close(to_np(out[0]), ref, TOL[dtype])


def test_prefill_glm_full_size_sampled(cuda_lib):
    """The chunked-prefill workload at full size (S=2048 new tokens at pos_base=8192,
    Tk=10240): every output computed on the GPU, sampled (query, head) pairs checked."""
    x = workload_inputs("glm_prefill_s2048", DEV)
    out = to_np(cuda_lib.prefill_naive(x["q"], x["Lc"], x["Rc"], x["kv_b"], GLM, x["pos_base"]))
    assert cuda_lib.device_status() == 0
    assert np.all(np.isfinite(out))
    queries, heads = [0, 1, 127, 128, 1000, 2047], [0, 17, 63]
    ref = oracle.prefill_nonabsorbed(to_np(x["q"][0]), to_np(x["Lc"][0]), to_np(x["Rc"][0]), to_np(x["kv_b"]),
                                     GLM.qk_nope, GLM.softmax_scale, x["pos_base"], queries=queries, heads=heads)
    got = out[0][np.ix_(queries, heads)]
    check_close(got, ref[np.ix_(queries, heads)], TOL["bf16"])
    # every query for eight heads spread over the 64: the absorbed attention at
    # each query's position (the oracle's prefill equals it at every position)
    heads8 = list(range(0, 64, 9))
    q = to_np(x["q"][0])[:, heads8]
    L, R, kvb = to_np(x["Lc"][0]), to_np(x["Rc"][0]), to_np(x["kv_b"])[heads8]
    S, pb = q.shape[0], x["pos_base"]
    ref8 = np.stack([oracle.attend_absorbed(q[s], L[:pb + s + 1], R[:pb + s + 1], kvb, GLM.qk_nope, pb + s,
                                            GLM.softmax_scale) for s in range(S)])
    check_close(out[0][:, heads8], ref8, TOL["bf16"])


def test_prefill_equals_decode_on_gpu(cuda_lib):
    """Absorbed decode and non-absorbed prefill of the same block agree ([MLA-KV] §2.3)."""
    S, pos_base = 6, 500
    x = mla_inputs(GLM, 1, S, [pos_base + S], pos_base + S, "bf16", 61, "cpu")
    g = _dev(x)
    a = to_np(cuda_lib.prefill_naive(g["q"], g["Lc"], g["Rc"], g["kv_b"], GLM, pos_base))
    b = to_np(cuda_lib.decode_absorbed(g["q"], g["Lc"], g["Rc"], g["T"], g["kv_b"], GLM))
    assert max_rel_err(a, b) < 2 * TOL["bf16"]

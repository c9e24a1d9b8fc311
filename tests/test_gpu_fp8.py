"""GPU parity of the FP8 latent cache (mla_decode_fp8, mla_decode_fp8_paged,
mla_cache_append_fp8, mla_cache_append_fp8_paged) against the fp64 oracle.

Decode: the oracle runs its plain absorbed decode over the dequantised cache
lat_scale * e4m3(code).  The kernels feed E4M3 codes to the tensor cores, so
each query row's absorbed latent query and the softmax probabilities are
rounded to E4M3 as well (unit roundoff u = 2^-4 each).  Every output is a
probability-weighted mean, and each probability carries a relative rounding
error of at most u, so the output error stays below u times the mean of the
value magnitudes; on these inputs a CPU model of the two roundings gives a
normwise error of 2-3.5%.  The bound used is u = 0.0625 (normwise); a wrong
descriptor, swizzle, scale or mask gives errors of order 1.

Append: the codes must be the oracle's (round to nearest even of the
normalised row / lat_scale), except where the oracle's value lies within a
relative 1e-5 of a rounding midpoint: there the fp32 kernel may take either
neighbour.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from tests._fp8_model import fp8_row_model
from tests._np import max_rel_err, to_np
from workload import GLM, append_inputs, fp8_latent_codes, mla_inputs, paged_layout, seq_lengths, to_pages

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
U_E4M3 = 2.0 ** -4
LAT_SCALE = 0.05
RMS_EPS = 1e-6


def _inputs(T, S, seed, device="cpu"):
    x = mla_inputs(GLM, len(T), S, T, max(T), "bf16", seed, device)
    x["Lc8"] = fp8_latent_codes(len(T), T, max(T), GLM.kv_lora, seed, device)
    del x["Lc"]
    return x


def _check_rows_against_model(got, x, T, S, lat_scale=LAT_SCALE, rows=None):
    """Each checked (b, s) row: the kernel's normwise error against the exact
    attention over the dequantised cache stays within 1.5x the error of the CPU
    rounding model on the same row (and at least 2e-3, for rows the roundings
    barely touch), and within the stated E4M3 bound."""
    codes = x["Lc8"].cpu().numpy()
    kvb = to_np(x["kv_b"])
    for b in range(len(T)):
        for s in range(S):
            if rows is not None and (b, s) not in rows:
                continue
            pos = T[b] - S + s
            q = to_np(x["q"][b, s])
            x8 = oracle.e4m3_decode(codes[b, :pos + 1])
            R = to_np(x["Rc"][b, :pos + 1])
            ref = oracle.attend_absorbed(q, lat_scale * x8, R, kvb, GLM.qk_nope, pos, GLM.softmax_scale)
            e_model = max_rel_err(fp8_row_model(q, x8, R, kvb, pos + 1, lat_scale), ref)
            e_gpu = max_rel_err(got[b, s], ref)
            assert e_gpu < U_E4M3 and e_gpu <= max(1.5 * e_model, 2e-3), (b, s, e_gpu, e_model)


def _ref(x, T, lat_scale=LAT_SCALE, rows=None):
    return oracle.decode_absorbed(to_np(x["q"]), oracle.dequant_latent(x["Lc8"].cpu().numpy(), lat_scale),
                                  to_np(x["Rc"]), T, to_np(x["kv_b"]), GLM.qk_nope, GLM.softmax_scale, rows=rows)


@pytest.mark.parametrize("T,S", [([1], 1), ([129, 300, 64], 1), ([128, 256], 1), ([130, 257, 6], 6),
                                 ([5000, 700], 2), ([4096], 1), ([33], 3)])
def test_decode_fp8(cuda_lib, T, S):
    x = _inputs(T, S, 500 + sum(T) + S)
    out = cuda_lib.decode_fp8(x["q"].to(DEV), x["Lc8"].to(DEV), x["Rc"].to(DEV), x["T"].to(DEV), x["kv_b"].to(DEV),
                              GLM, LAT_SCALE)
    assert cuda_lib.device_status() == 0
    got = to_np(out)
    assert np.all(np.isfinite(got))
    assert max_rel_err(got, _ref(x, T)) < U_E4M3
    _check_rows_against_model(got, x, T, S)


@pytest.mark.parametrize("T,S", [([40000], 1), ([40000, 39001], 2)])
def test_decode_fp8_streaming_few_rows(cuda_lib, T, S):
    """Few query rows over long caches: every CTA runs two or more key tiles,
    which the streaming form of the FP8 attention serves, with the query rows
    quantised inside the kernel; ragged last tiles and a second sequence."""
    x = _inputs(T, S, 900 + sum(T) + S)
    out = cuda_lib.decode_fp8(x["q"].to(DEV), x["Lc8"].to(DEV), x["Rc"].to(DEV), x["T"].to(DEV), x["kv_b"].to(DEV),
                              GLM, LAT_SCALE)
    assert cuda_lib.device_status() == 0
    got = to_np(out)
    assert np.all(np.isfinite(got))
    assert max_rel_err(got, _ref(x, T)) < U_E4M3
    _check_rows_against_model(got, x, T, S)


@pytest.mark.parametrize("lat_scale", [1.0 / 64, 0.3])
def test_decode_fp8_scale_enters_linearly(cuda_lib, lat_scale):
    """Other cache scales: the same codes describe a cache lat_scale times the codes."""
    T, S = [700, 90], 1
    x = _inputs(T, S, 77)
    out = cuda_lib.decode_fp8(x["q"].to(DEV), x["Lc8"].to(DEV), x["Rc"].to(DEV), x["T"].to(DEV), x["kv_b"].to(DEV),
                              GLM, lat_scale)
    assert cuda_lib.device_status() == 0
    assert max_rel_err(to_np(out), _ref(x, T, lat_scale)) < U_E4M3
    _check_rows_against_model(to_np(out), x, T, S, lat_scale)


def test_decode_fp8_glm_batched_b32_sampled(cuda_lib):
    """32 sequences of 1024..32768 keys (the batched tensor-core path), checked
    on a sample of sequences."""
    T = seq_lengths(32, 1024, 32768, 41)
    x = _inputs(T, 1, 42, DEV)
    out = to_np(cuda_lib.decode_fp8(x["q"], x["Lc8"], x["Rc"], x["T"], x["kv_b"], GLM, LAT_SCALE))
    assert cuda_lib.device_status() == 0
    for b in (0, 13, 31):
        one = {k: (v[b:b + 1].cpu() if k in ("q", "Lc8", "Rc") else v.cpu()) for k, v in x.items()}
        assert max_rel_err(out[b], _ref(one, [T[b]])[0]) < U_E4M3, b
    xc = {k: (v.cpu() if isinstance(v, torch.Tensor) else v) for k, v in x.items()}
    _check_rows_against_model(out, xc, T, 1, rows={(0, 0), (13, 0), (31, 0)})


def test_decode_fp8_more_sequences_than_the_in_kernel_plan(cuda_lib):
    """1100 sequences (the attention CTAs read the absorb kernel's plan), 1..200 keys each."""
    B = 1100
    r = np.random.default_rng(31)
    T = [int(t) for t in r.integers(1, 201, B)]
    x = _inputs(T, 1, 32)
    out = to_np(cuda_lib.decode_fp8(x["q"].to(DEV), x["Lc8"].to(DEV), x["Rc"].to(DEV), x["T"].to(DEV),
                                    x["kv_b"].to(DEV), GLM, LAT_SCALE))
    assert cuda_lib.device_status() == 0
    for b in (0, 777, 1023, 1024, 1099):
        one = {k: (v[b:b + 1] if k in ("q", "Lc8", "Rc") else v) for k, v in x.items()}
        assert max_rel_err(out[b], _ref(one, [T[b]])[0]) < U_E4M3, b


@pytest.mark.parametrize("page_size", [128, 256])
@pytest.mark.parametrize("T,S", [([129, 300, 64], 1), ([130, 257, 6], 6)])
def test_decode_fp8_paged(cuda_lib, page_size, T, S):
    x = _inputs(T, S, 600 + sum(T) + page_size)
    table, num_pages = paged_layout(T, page_size, 7 + S)
    L8p = to_pages(x["Lc8"], table, T, page_size, num_pages, fill=0x7F)
    Rp = to_pages(x["Rc"], table, T, page_size, num_pages)
    out = cuda_lib.decode_fp8_paged(x["q"].to(DEV), L8p.to(DEV), Rp.to(DEV), table.to(DEV), x["T"].to(DEV),
                                    x["kv_b"].to(DEV), GLM, LAT_SCALE)
    assert cuda_lib.device_status() == 0
    assert max_rel_err(to_np(out), _ref(x, T)) < U_E4M3


def test_decode_fp8_flags_bad_length(cuda_lib):
    T = [300, 200]
    x = _inputs(T, 1, 9)
    Tbad = torch.tensor([300, 400], dtype=torch.int32, device=DEV)  # 400 > T_cap = 300
    out = cuda_lib.decode_fp8(x["q"].to(DEV), x["Lc8"].to(DEV), x["Rc"].to(DEV), Tbad, x["kv_b"].to(DEV), GLM,
                              LAT_SCALE)
    assert cuda_lib.device_status() & cuda_lib.MLA_DEV_BAD_LENGTH
    assert cuda_lib.device_status() == 0
    ref = _ref(x, [300, 200])
    assert max_rel_err(to_np(out)[0], ref[0]) < U_E4M3


def _codes_match(got, y):
    """got: kernel codes; y: the oracle's value before rounding (normalised / lat_scale)."""
    want = oracle.e4m3_encode(y)
    same = oracle.e4m3_decode(got) == oracle.e4m3_decode(want)   # -0 and +0 alike
    # values within 1e-5 (relative) of a midpoint between two neighbours may round either way
    lo = oracle.e4m3_decode(oracle.e4m3_encode(y * (1 - 1e-5)))
    hi = oracle.e4m3_decode(oracle.e4m3_encode(y * (1 + 1e-5)))
    either = (oracle.e4m3_decode(got) == lo) | (oracle.e4m3_decode(got) == hi)
    return np.all(same | either), int(np.sum(~same))


@pytest.mark.parametrize("T,S", [([1], 1), ([129, 300, 64], 1), ([130, 257, 6], 6), ([70000], 2)])
def test_cache_append_fp8_rows(cuda_lib, T, S):
    B, T_cap = len(T), max(T) + 5
    x = append_inputs(GLM, B, S, "bf16", 11 + sum(T) + S, "cpu")
    lat_scale = math.sqrt(GLM.kv_lora) * float(x["kv_a_ln"].float().abs().max()) / 448
    g = torch.Generator().manual_seed(12)
    Lc8 = torch.randint(0, 256, (B, T_cap, GLM.kv_lora), generator=g, dtype=torch.uint8).to(DEV)
    Rc = torch.randn(B, T_cap, GLM.qk_rope, generator=g).bfloat16().to(DEV)
    L0, R0 = Lc8.clone(), Rc.clone()
    Tt = torch.tensor(T, dtype=torch.int32, device=DEV)
    cuda_lib.cache_append_fp8(x["comp"].to(DEV), x["kv_a_ln"].to(DEV), Tt, Lc8, Rc, GLM, RMS_EPS, lat_scale)
    assert cuda_lib.device_status() == 0
    lc, rc, pos = oracle.cache_append(to_np(x["comp"]), to_np(x["kv_a_ln"]), RMS_EPS, T, GLM.kv_lora)
    got = np.stack([Lc8[b, t - S:t].cpu().numpy() for b, t in enumerate(T)])
    ok, differ = _codes_match(got, lc / lat_scale)
    assert ok, differ
    got_r = np.stack([to_np(Rc[b, t - S:t]) for b, t in enumerate(T)])
    assert np.all(np.abs(got_r - rc) <= 2.0 ** -8 * np.abs(rc) + 1e-5 * np.max(np.abs(rc)))
    keep = torch.ones(B, T_cap, dtype=torch.bool, device=DEV)
    for b, t in enumerate(T):
        keep[b, t - S:t] = False
    assert torch.equal(Lc8[keep], L0[keep])
    assert torch.equal(Rc[keep].view(torch.uint8), R0[keep].view(torch.uint8))


def test_cache_append_fp8_paged_rows(cuda_lib):
    T, S, page_size = [130, 257, 6], 6, 128
    table, num_pages = paged_layout(T, page_size, 29)
    x = append_inputs(GLM, 3, S, "bf16", 31, "cpu")
    lat_scale = 0.05
    L8p = torch.zeros(num_pages, page_size, GLM.kv_lora, dtype=torch.uint8, device=DEV)
    Rp = torch.zeros(num_pages, page_size, GLM.qk_rope, dtype=torch.bfloat16, device=DEV)
    cuda_lib.cache_append_fp8_paged(x["comp"].to(DEV), x["kv_a_ln"].to(DEV), table.to(DEV),
                                    torch.tensor(T, dtype=torch.int32, device=DEV), L8p, Rp, GLM, RMS_EPS, lat_scale)
    assert cuda_lib.device_status() == 0
    lc, rc, pos = oracle.cache_append(to_np(x["comp"]), to_np(x["kv_a_ln"]), RMS_EPS, T, GLM.kv_lora)
    tbl = table.tolist()
    flat = L8p.view(-1, GLM.kv_lora).cpu().numpy()
    got = np.stack([[flat[oracle.page_row(tbl, b, int(pos[b, s]), page_size)] for s in range(S)] for b in range(3)])
    ok, differ = _codes_match(got, lc / lat_scale)
    assert ok, differ
    assert int((L8p.view(-1, GLM.kv_lora) != 0).any(dim=1).sum()) == 3 * S  # no other pool row touched


def test_append_fp8_then_decode_fp8(cuda_lib):
    """Rows written by the FP8 append and read by the FP8 decode give the
    oracle's decode of the oracle-written FP8 cache (within the decode bound)."""
    T, S = [300, 45], 2
    x = _inputs(T, S, 90)
    a = append_inputs(GLM, 2, S, "bf16", 91, "cpu")
    lat_scale = math.sqrt(GLM.kv_lora) * float(a["kv_a_ln"].float().abs().max()) / 448
    Lc8, Rc = x["Lc8"].clone().to(DEV), x["Rc"].clone().to(DEV)
    Tt = x["T"].to(DEV)
    cuda_lib.cache_append_fp8(a["comp"].to(DEV), a["kv_a_ln"].to(DEV), Tt, Lc8, Rc, GLM, RMS_EPS, lat_scale)
    out = cuda_lib.decode_fp8(x["q"].to(DEV), Lc8, Rc, Tt, x["kv_b"].to(DEV), GLM, lat_scale)
    assert cuda_lib.device_status() == 0
    codes, rc, _ = oracle.cache_append_fp8(to_np(a["comp"]), to_np(a["kv_a_ln"]), RMS_EPS, T, GLM.kv_lora, lat_scale)
    L8 = x["Lc8"].numpy().copy()
    R = to_np(x["Rc"]).copy()
    for b, t in enumerate(T):
        L8[b, t - S:t] = codes[b]
        R[b, t - S:t] = rc[b]
    ref = oracle.decode_absorbed(to_np(x["q"]), oracle.dequant_latent(L8, lat_scale), R, T, to_np(x["kv_b"]),
                                 GLM.qk_nope, GLM.softmax_scale)
    assert max_rel_err(to_np(out), ref) < U_E4M3

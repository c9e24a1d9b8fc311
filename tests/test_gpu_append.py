"""GPU parity of the cache writers (mla_cache_append, dsa_index_key_append)
against the fp64 oracle.

The new rows are compared element by element: fp32 caches within 1e-5 of the
oracle relative to the row's largest value, bf16 caches within one bf16 ulp
(2^-8 relative) of the oracle value, since the kernel rounds once from fp32.
Every other row of the caches must come back bit-identical.
"""
import numpy as np
import pytest
import torch

import oracle
from tests._np import to_np
from workload import GLM, TINY, Dims, append_inputs, seq_lengths

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
RMS_EPS = 1e-6


def _fill(shape, dtype, seed):
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    return torch.randn(*shape, generator=g).to(dtype).to(DEV)


def _check_rows(got, ref, dtype):
    """got, ref: [B, S, D] new rows; ref in fp64; the fp32 bound is relative to the row's largest value."""
    scale = np.max(np.abs(ref), axis=-1, keepdims=True) + 1e-30
    if dtype == "f32":
        assert np.max(np.abs(got - ref) / scale) < 1e-5
    else:  # one rounding to bf16 (half an ulp <= 2^-8 |x|) after fp32 arithmetic
        assert np.all(np.abs(got - ref) <= 2.0 ** -8 * np.abs(ref) + 1e-5 * scale)


def _untouched_equal(after, before, T, S):
    keep = torch.ones(after.shape[:2], dtype=torch.bool, device=after.device)
    for b, t in enumerate(T):
        keep[b, t - S:t] = False
    return torch.equal(after[keep].view(torch.uint8) if after.dtype == torch.bfloat16 else after[keep],
                       before[keep].view(torch.uint8) if before.dtype == torch.bfloat16 else before[keep])


def _new_rows(cache, T, S):
    return np.stack([to_np(cache[b, t - S:t]) for b, t in enumerate(T)])


WIDE = Dims(H=2, qk_nope=8, qk_rope=200, kv_lora=1000, v_head=8)  # more than 4 latent values per thread


@pytest.mark.parametrize("dtype,dims", [("f32", TINY), ("f32", GLM), ("bf16", GLM), ("bf16", WIDE)])
@pytest.mark.parametrize("T,S", [([1], 1), ([6], 6), ([129, 300, 64], 1), ([130, 257, 6], 6), ([70000], 2)])
def test_cache_append_rows(cuda_lib, dtype, dims, T, S):
    B, T_cap = len(T), max(T) + 5
    x = append_inputs(dims, B, S, dtype, 7 + sum(T) + S, "cpu")
    tdt = torch.float32 if dtype == "f32" else torch.bfloat16
    Lc = _fill((B, T_cap, dims.kv_lora), tdt, 1)
    Rc = _fill((B, T_cap, dims.qk_rope), tdt, 2)
    Lc0, Rc0 = Lc.clone(), Rc.clone()
    Tt = torch.tensor(T, dtype=torch.int32, device=DEV)
    cuda_lib.cache_append(x["comp"].to(DEV), x["kv_a_ln"].to(DEV), Tt, Lc, Rc, dims, RMS_EPS)
    assert cuda_lib.device_status() == 0
    lc, rc, pos = oracle.cache_append(to_np(x["comp"]), to_np(x["kv_a_ln"]), RMS_EPS, T, dims.kv_lora)
    assert pos[0, -1] == T[0] - 1
    _check_rows(_new_rows(Lc, T, S), lc, dtype)
    _check_rows(_new_rows(Rc, T, S), rc, dtype)
    assert _untouched_equal(Lc, Lc0, T, S) and _untouched_equal(Rc, Rc0, T, S)


def test_cache_append_glm_batched_b32_s6(cuda_lib):
    """The batched GLM-5.2 shape: 32 sequences of 1024..32768 cached tokens in a
    32768-row cache, 6 new tokens each (the speculative-decode step)."""
    B, S, T_cap = 32, 6, 32768
    T = seq_lengths(B, 1024, 32768, 99)
    x = append_inputs(GLM, B, S, "bf16", 21, DEV)
    Lc = torch.zeros(B, T_cap, GLM.kv_lora, dtype=torch.bfloat16, device=DEV)
    Rc = torch.zeros(B, T_cap, GLM.qk_rope, dtype=torch.bfloat16, device=DEV)
    Tt = torch.tensor(T, dtype=torch.int32, device=DEV)
    cuda_lib.cache_append(x["comp"], x["kv_a_ln"], Tt, Lc, Rc, GLM, RMS_EPS)
    assert cuda_lib.device_status() == 0
    lc, rc, _ = oracle.cache_append(to_np(x["comp"]), to_np(x["kv_a_ln"]), RMS_EPS, T, GLM.kv_lora)
    _check_rows(_new_rows(Lc, T, S), lc, "bf16")
    _check_rows(_new_rows(Rc, T, S), rc, "bf16")
    written = torch.zeros(B, T_cap, dtype=torch.bool, device=DEV)
    for b, t in enumerate(T):
        written[b, t - S:t] = True
    assert not torch.any(Lc[~written] != 0) and not torch.any(Rc[~written] != 0)


def test_cache_append_flags_bad_length(cuda_lib):
    S, T_cap = 2, 40
    x = append_inputs(GLM, 3, S, "bf16", 3, DEV)
    Lc = _fill((3, T_cap, GLM.kv_lora), torch.bfloat16, 4)
    Rc = _fill((3, T_cap, GLM.qk_rope), torch.bfloat16, 5)
    Lc0, Rc0 = Lc.clone(), Rc.clone()
    Tt = torch.tensor([40, 41, 1], dtype=torch.int32, device=DEV)  # 41 > T_cap, 1 < S
    cuda_lib.cache_append(x["comp"], x["kv_a_ln"], Tt, Lc, Rc, GLM, RMS_EPS)
    assert cuda_lib.device_status() & cuda_lib.MLA_DEV_BAD_LENGTH
    assert torch.equal(Lc[1:].view(torch.uint8), Lc0[1:].view(torch.uint8))
    assert torch.equal(Rc[1:].view(torch.uint8), Rc0[1:].view(torch.uint8))
    lc, rc, _ = oracle.cache_append(to_np(x["comp"][:1]), to_np(x["kv_a_ln"]), RMS_EPS, [40], GLM.kv_lora)
    _check_rows(_new_rows(Lc[:1], [40], S), lc, "bf16")
    assert cuda_lib.device_status() == 0


@pytest.mark.parametrize("hd,rope_dim,bias", [(128, 64, True), (128, 0, True), (128, 128, False),
                                              (8, 4, True), (300, 64, True)])
@pytest.mark.parametrize("T,S", [([1], 1), ([130, 257, 6], 6), ([65536, 9], 1)])
def test_index_key_append_rows(cuda_lib, hd, rope_dim, bias, T, S):
    B, T_cap = len(T), max(T) + 3
    x = append_inputs(GLM, B, S, "f32", 13 + hd + rope_dim + S, "cpu", index_hd=hd)
    ln_b = x["ln_b"] if bias else None
    Ic = _fill((B, T_cap, hd), torch.float32, 6)
    Ic0 = Ic.clone()
    Tt = torch.tensor(T, dtype=torch.int32, device=DEV)
    cuda_lib.index_key_append(x["k_idx"].to(DEV), x["ln_w"].to(DEV), None if ln_b is None else ln_b.to(DEV),
                              Tt, Ic, rope_dim)
    assert cuda_lib.device_status() == 0
    ref, _ = oracle.index_key_append(to_np(x["k_idx"]), to_np(x["ln_w"]), None if ln_b is None else to_np(ln_b),
                                     1e-6, T, rope_dim)
    _check_rows(_new_rows(Ic, T, S), ref, "f32")
    assert _untouched_equal(Ic, Ic0, T, S)


def test_append_then_decode_matches_oracle(cuda_lib):
    """A cache written by the append kernels and read by the absorbed decode
    gives the oracle's decode of the oracle-written cache."""
    T, S, T_cap = [300, 45], 1, 320
    dims = GLM
    x = append_inputs(dims, 2, S, "f32", 31, "cpu")
    Lc = _fill((2, T_cap, dims.kv_lora), torch.float32, 8) / 8.0
    Rc = _fill((2, T_cap, dims.qk_rope), torch.float32, 9) / 8.0
    g = torch.Generator(device="cpu")
    g.manual_seed(10)
    q = torch.randn(2, S, dims.H, dims.qk_head, generator=g) / 8.0
    kv_b = torch.randn(dims.H, dims.qk_nope + dims.v_head, dims.kv_lora, generator=g) * 0.02
    Lc_np, Rc_np = to_np(Lc).copy(), to_np(Rc).copy()
    Tt = torch.tensor(T, dtype=torch.int32, device=DEV)
    cuda_lib.cache_append(x["comp"].to(DEV), x["kv_a_ln"].to(DEV), Tt, Lc, Rc, dims, RMS_EPS)
    out = cuda_lib.decode_absorbed(q.to(DEV), Lc, Rc, Tt, kv_b.to(DEV), dims)
    assert cuda_lib.device_status() == 0
    lc, rc, _ = oracle.cache_append(to_np(x["comp"]), to_np(x["kv_a_ln"]), RMS_EPS, T, dims.kv_lora)
    for b, t in enumerate(T):
        Lc_np[b, t - S:t] = lc[b]
        Rc_np[b, t - S:t] = rc[b]
    ref = oracle.decode_absorbed(to_np(q), Lc_np, Rc_np, T, to_np(kv_b), dims.qk_nope, dims.softmax_scale)
    got = to_np(out)
    assert np.max(np.abs(got - ref)) / np.max(np.abs(ref)) < 1e-5

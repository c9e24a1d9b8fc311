"""Bounded device waits, made to run out on unchanged kernels.

Every wait inside the tensor-core kernels (a TMA copy landing, an MMA
retiring, a partner warp's hand-over) gives up after the library's wait
limit, raises MLA_DEV_TIMEOUT in the device status word and lets the kernel
drain its copies and MMAs, free its tensor memory and return.  With the limit
at 1 ns every wait on data still in flight gives up at once, so each call
below must (1) return, (2) leave MLA_DEV_TIMEOUT in the status word, and (3)
leave nothing behind: the same call at the default limit right after it
matches the oracle and raises no flag.
"""
import numpy as np
import pytest
import torch

import oracle
from tests._np import check_close, max_rel_err, to_np
from workload import GLM, dsa_inputs, fp8_latent_codes, mla_inputs

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
DEFAULT_LIMIT_NS = 2_000_000_000  # the library's default wait limit
TOL_BF16 = 2e-2


def _dev(x):
    return {k: (v.to(DEV) if isinstance(v, torch.Tensor) else v) for k, v in x.items()}


def _timed_out_then_recovers(cuda_lib, call):
    """Runs call() at a 1 ns limit (expects MLA_DEV_TIMEOUT), then at the
    default limit (expects a clean status); returns the second result."""
    assert cuda_lib.device_status() == 0
    cuda_lib.set_wait_limit_ns(1)
    try:
        call()
        flags = cuda_lib.device_status()
    finally:
        cuda_lib.set_wait_limit_ns(DEFAULT_LIMIT_NS)
    assert flags & cuda_lib.MLA_DEV_TIMEOUT, f"flags {flags:#x}: no wait ran out"
    out = call()
    assert cuda_lib.device_status() == 0
    return out


@pytest.mark.parametrize("B,T", [(1, [512]), (16, None)])
def test_decode_timeout_then_recovers(cuda_lib, B, T):
    """B=1: absorb, attention and combine kernels; B=16: the tensor-core GEMMs
    of the many-row path as well."""
    T = T or [int(t) for t in np.random.default_rng(41).integers(100, 700, B)]
    x = mla_inputs(GLM, B, 1, T, max(T), "bf16", 700 + B, "cpu")
    g = _dev(x)
    out = _timed_out_then_recovers(
        cuda_lib, lambda: cuda_lib.decode_absorbed(g["q"], g["Lc"], g["Rc"], g["T"], g["kv_b"], GLM))
    ref = oracle.decode_absorbed(to_np(x["q"]), to_np(x["Lc"]), to_np(x["Rc"]), T, to_np(x["kv_b"]), GLM.qk_nope,
                                 GLM.softmax_scale)
    check_close(to_np(out), ref, TOL_BF16)


def test_dsa_select_timeout_then_recovers(cuda_lib):
    """The tensor-core indexer (32 index heads x 128) feeding the cluster top-k."""
    T = [3000, 2049]
    d = dsa_inputs(2, 1, T, max(T), 32, 128, 43, "cpu")
    gd = _dev(d)
    Tg = torch.tensor(T, dtype=torch.int32, device=DEV)
    sc, sel, nsel = _timed_out_then_recovers(
        cuda_lib, lambda: cuda_lib.select(gd["q_idx"], gd["w"], gd["Ic"], Tg, 2048))
    ref_sc = oracle.index_scores(to_np(d["q_idx"]), to_np(d["w"]), to_np(d["Ic"]), T)
    ref_sel, ref_n = oracle.topk_select(ref_sc, T, 1, 2048)
    assert np.array_equal(to_np(sc)[np.isfinite(ref_sc)], ref_sc[np.isfinite(ref_sc)])
    assert np.array_equal(sel.cpu().numpy(), ref_sel) and np.array_equal(nsel.cpu().numpy(), ref_n)


def test_prefill_timeout_then_recovers(cuda_lib):
    """The tensor-core prefill: kv_b GEMM and flash attention."""
    S, pos_base = 200, 300
    x = mla_inputs(GLM, 1, S, [pos_base + S], pos_base + S, "bf16", 45, "cpu")
    g = _dev(x)
    out = _timed_out_then_recovers(
        cuda_lib, lambda: cuda_lib.prefill_naive(g["q"], g["Lc"], g["Rc"], g["kv_b"], GLM, pos_base))
    queries, heads = [0, 57, 199], [0, 31, 63]
    ref = oracle.prefill_nonabsorbed(to_np(x["q"][0]), to_np(x["Lc"][0]), to_np(x["Rc"][0]), to_np(x["kv_b"]),
                                     GLM.qk_nope, GLM.softmax_scale, pos_base, queries=queries, heads=heads)
    check_close(to_np(out)[0][np.ix_(queries, heads)], ref[np.ix_(queries, heads)], TOL_BF16)


def test_fp8_decode_timeout_then_recovers(cuda_lib):
    """The FP8 path: query quantiser and the kind::f8f6f4 attention kernel."""
    T = [700, 129]
    x = mla_inputs(GLM, 2, 1, T, max(T), "bf16", 47, "cpu")
    L8 = fp8_latent_codes(2, T, max(T), GLM.kv_lora, 47, "cpu")
    g = _dev(x)
    L8d = L8.to(DEV)
    out = _timed_out_then_recovers(
        cuda_lib, lambda: cuda_lib.decode_fp8(g["q"], L8d, g["Rc"], g["T"], g["kv_b"], GLM, 0.05))
    ref = oracle.decode_absorbed(to_np(x["q"]), oracle.dequant_latent(L8.numpy(), 0.05), to_np(x["Rc"]), T,
                                 to_np(x["kv_b"]), GLM.qk_nope, GLM.softmax_scale)
    check_close(to_np(out), ref, 2.0 ** -4)


@pytest.mark.parametrize("B", [1, 4])
def test_decode_oproj_timeout_then_recovers(cuda_lib, B):
    """Decode, then the projection: the ring of W_O rows (bulk copies into shared memory) for B=1, the
    register GEMV after the many-row decode chain for B=4."""
    T, hidden = [700, 300, 129, 512][:B], 640
    x = mla_inputs(GLM, B, 1, T, 700, "bf16", 49, "cpu")
    g = _dev(x)
    gen = torch.Generator().manual_seed(50)
    w = (torch.randn(hidden, GLM.H * GLM.v_head, generator=gen) * 0.02).to(torch.bfloat16)
    wd = w.to(DEV)
    y = _timed_out_then_recovers(
        cuda_lib, lambda: cuda_lib.decode_oproj(g["q"], g["Lc"], g["Rc"], g["T"], g["kv_b"], wd, GLM))
    att = oracle.decode_absorbed(to_np(x["q"]), to_np(x["Lc"]), to_np(x["Rc"]), T, to_np(x["kv_b"]), GLM.qk_nope,
                                 GLM.softmax_scale)
    ref = oracle.o_proj(att.reshape(B, -1), to_np(w)).reshape(B, 1, hidden)
    assert max_rel_err(to_np(y), ref) < TOL_BF16

"""mla_prefill_naive_noalloc: the prefill entry point that allocates nothing.

It serves callers that may not allocate device memory (their GPU memory is
owned by a host framework's pool, or they cannot afford the synchronisation a
cudaMalloc may cause, or they are plain C programs without an allocator).
Its scratch is a static device array inside the library, so these tests check
that two calls in a row -- each reusing the array the previous call left
behind -- match the workspace-taking mla_prefill_naive within the usual
tolerances, and that requests larger than the array are refused up front.

This file is named to be collected last, so a run that stops at the first
failure has already run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

import mla_latent_kv_06_gb300 as mla
from tests._np import check_close, max_rel_err, to_np
from workload import GLM, TINY, mla_inputs

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
TOL = {"f32": 1e-5, "bf16": 2e-2}


def _noalloc(lib, dims, x, pos_base, out):
    q = x["q"]
    B, S = q.shape[0], q.shape[1]
    d = mla.make_dims(dims)
    code = mla.MLA_F32 if q.dtype == torch.float32 else mla.MLA_BF16
    return lib.mla_prefill_naive_noalloc(ctypes.byref(d), code, B, S, pos_base, q.data_ptr(),
                                         x["Lc"].data_ptr(), x["Rc"].data_ptr(), x["kv_b"].data_ptr(),
                                         out.data_ptr(), torch.cuda.current_stream().cuda_stream)


def _case(dims, dtype, S, pos_base, seed):
    Tk = pos_base + S
    x = mla_inputs(dims, 1, S, [Tk], Tk, dtype, seed, "cpu")
    return {k: v.to(DEV) for k, v in x.items()}


def test_noalloc_matches_prefill_on_two_calls_in_a_row(cuda_lib):
    lib = cuda_lib.lib()
    cases = [(GLM, "bf16", 16, 200, 501), (TINY, "f32", 6, 10, 502)]
    for dims, dtype, S, pos_base, seed in cases:  # two calls in a row, different sizes
        x = _case(dims, dtype, S, pos_base, seed)
        got = torch.full((1, S, dims.H, dims.v_head), float("nan"), device=DEV)
        rc = _noalloc(lib, dims, x, pos_base, got)
        assert rc == mla.MLA_OK, lib.mla_last_error()
        ref = cuda_lib.prefill_naive(x["q"], x["Lc"], x["Rc"], x["kv_b"], dims, pos_base)
        torch.cuda.synchronize()
        g, r = to_np(got), to_np(ref)
        assert np.all(np.isfinite(g))
        check_close(g, r, TOL[dtype])


def test_noalloc_repeated_call_same_inputs(cuda_lib):
    lib = cuda_lib.lib()
    x = _case(GLM, "bf16", 8, 120, 503)
    outs = []
    for _ in range(2):
        o = torch.empty(1, 8, GLM.H, GLM.v_head, device=DEV)
        assert _noalloc(lib, GLM, x, 120, o) == mla.MLA_OK, lib.mla_last_error()
        outs.append(o)
    ref = cuda_lib.prefill_naive(x["q"], x["Lc"], x["Rc"], x["kv_b"], GLM, 120)
    torch.cuda.synchronize()
    for o in outs:
        check_close(to_np(o), to_np(ref), TOL["bf16"])


def test_noalloc_refuses_requests_beyond_its_scratch(cuda_lib):
    """GLM bf16 needs 57,344 bytes of rebuilt KV per key: 2,016 keys exceed 32 MiB."""
    lib = cuda_lib.lib()
    x = _case(GLM, "bf16", 16, 16, 504)  # small real tensors; the size check fires first
    d = mla.make_dims(GLM)
    out = torch.empty(1, 16, GLM.H, GLM.v_head, device=DEV)
    rc = lib.mla_prefill_naive_noalloc(ctypes.byref(d), mla.MLA_BF16, 1, 16, 2000, x["q"].data_ptr(),
                                       x["Lc"].data_ptr(), x["Rc"].data_ptr(), x["kv_b"].data_ptr(),
                                       out.data_ptr(), None)
    assert rc == mla.MLA_ERR_INVALID
    assert b"static scratch" in lib.mla_last_error()

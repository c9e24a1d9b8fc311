"""mla_prefill_naive_noalloc: the prefill entry point that allocates nothing.

It serves callers that may not allocate device memory (their GPU memory is
owned by a host framework's pool, or they cannot afford the synchronisation a
cudaMalloc may cause, or they are plain C programs without an allocator).
Its scratch is a static device array inside the library, so these tests check
that calls in a row -- each reusing the array the previous call left behind --
agree with the oracle and give the very outputs of the workspace-taking
mla_prefill_naive (the same kernels), including a request that fills the
array to within 8 KB, and that requests larger than the array are refused up
front.

This file is named to be collected last, so a run that stops at the first
failure has already run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

import mla_latent_kv_06_gb300 as mla
import oracle
from tests._np import check_close, to_np
from workload import GLM, TINY, mla_inputs

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
TOL = {"f32": 1e-5, "bf16": 2e-2}
SCRATCH = 32 << 20
GLM_KEY_BYTES = GLM.H * (GLM.qk_nope + GLM.v_head) * 2  # rebuilt KV bytes per key, bf16


def _noalloc(lib, dims, x, pos_base, out, stream=None):
    q = x["q"]
    B, S = q.shape[0], q.shape[1]
    d = mla.make_dims(dims)
    code = mla.MLA_F32 if q.dtype == torch.float32 else mla.MLA_BF16
    st = torch.cuda.current_stream().cuda_stream if stream is None else stream
    return lib.mla_prefill_naive_noalloc(ctypes.byref(d), code, B, S, pos_base, q.data_ptr(),
                                         x["Lc"].data_ptr(), x["Rc"].data_ptr(), x["kv_b"].data_ptr(),
                                         out.data_ptr(), st)


def _case(dims, dtype, S, pos_base, seed):
    Tk = pos_base + S
    x = mla_inputs(dims, 1, S, [Tk], Tk, dtype, seed, "cpu")
    return x, {k: v.to(DEV) for k, v in x.items()}


def _oracle(x, dims, pos_base, queries, heads):
    return oracle.prefill_nonabsorbed(to_np(x["q"][0]), to_np(x["Lc"][0]), to_np(x["Rc"][0]), to_np(x["kv_b"]),
                                      dims.qk_nope, dims.softmax_scale, pos_base, queries=queries, heads=heads)


@pytest.mark.parametrize("dims,dtype,S,pos_base", [(GLM, "bf16", 16, 200), (TINY, "f32", 6, 10),
                                                   (GLM, "bf16", 64, 585 - 64)])
def test_noalloc_matches_oracle_and_prefill(cuda_lib, dims, dtype, S, pos_base):
    """The last case needs 585 * 57,344 = 33,546,240 of the 33,554,432 bytes."""
    lib = cuda_lib.lib()
    x, g = _case(dims, dtype, S, pos_base, 500 + S + pos_base)
    got = torch.full((1, S, dims.H, dims.v_head), float("nan"), device=DEV)
    rc = _noalloc(lib, dims, g, pos_base, got)
    assert rc == mla.MLA_OK, lib.mla_last_error()
    ref = cuda_lib.prefill_naive(g["q"], g["Lc"], g["Rc"], g["kv_b"], dims, pos_base)
    torch.cuda.synchronize()
    assert cuda_lib.device_status() == 0
    assert torch.equal(got, ref), "the same kernels on the same inputs give the same outputs"
    queries = sorted({0, S // 2, S - 1})
    heads = sorted({0, dims.H // 2, dims.H - 1})
    want = _oracle(x, dims, pos_base, queries, heads)
    check_close(to_np(got)[0][np.ix_(queries, heads)], want[np.ix_(queries, heads)], TOL[dtype])


def test_noalloc_calls_in_a_row_reuse_the_array(cuda_lib):
    """A large request, then a small one, then the large one again: each
    against the oracle, the array holding the previous call's contents."""
    lib = cuda_lib.lib()
    cases = [(GLM, "bf16", 32, 500), (GLM, "bf16", 8, 120), (GLM, "bf16", 32, 500)]
    for i, (dims, dtype, S, pos_base) in enumerate(cases):
        x, g = _case(dims, dtype, S, pos_base, 600 + i)
        got = torch.empty(1, S, dims.H, dims.v_head, device=DEV)
        assert _noalloc(lib, dims, g, pos_base, got) == mla.MLA_OK, lib.mla_last_error()
        torch.cuda.synchronize()
        assert cuda_lib.device_status() == 0
        queries, heads = [0, S - 1], [0, 63]
        want = _oracle(x, dims, pos_base, queries, heads)
        check_close(to_np(got)[0][np.ix_(queries, heads)], want[np.ix_(queries, heads)], TOL[dtype])


def test_noalloc_refuses_requests_beyond_its_scratch(cuda_lib):
    """586 GLM bf16 keys need 33,603,584 bytes: refused before any launch."""
    assert 585 * GLM_KEY_BYTES <= SCRATCH < 586 * GLM_KEY_BYTES
    lib = cuda_lib.lib()
    _, g = _case(GLM, "bf16", 16, 16, 504)  # small real tensors; the size check fires first
    d = mla.make_dims(GLM)
    out = torch.empty(1, 16, GLM.H, GLM.v_head, device=DEV)
    rc = lib.mla_prefill_naive_noalloc(ctypes.byref(d), mla.MLA_BF16, 1, 16, 586 - 16, g["q"].data_ptr(),
                                       g["Lc"].data_ptr(), g["Rc"].data_ptr(), g["kv_b"].data_ptr(),
                                       out.data_ptr(), None)
    assert rc == mla.MLA_ERR_INVALID
    assert b"static scratch" in lib.mla_last_error()
    # sizes whose product overflows are refused the same way
    rc = lib.mla_prefill_naive_noalloc(ctypes.byref(d), mla.MLA_BF16, 1 << 30, 16, (1 << 31) - 17,
                                       g["q"].data_ptr(), g["Lc"].data_ptr(), g["Rc"].data_ptr(),
                                       g["kv_b"].data_ptr(), out.data_ptr(), None)
    assert rc == mla.MLA_ERR_INVALID

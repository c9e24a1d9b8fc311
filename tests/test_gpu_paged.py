"""GPU parity of the paged-cache entry points (mla_decode_paged,
mla_sparse_decode_paged, mla_cache_append_paged) against the fp64 oracle.

The oracle reads the pool back into a contiguous cache through the block
table (oracle.unpage) and runs its plain decode.  Tolerances as for the
contiguous layout: 1e-5 for fp32 inputs, 2e-2 for bf16 (normwise).  Pool rows
that no sequence owns are NaN, so a read through a wrong page shows up.
"""
import numpy as np
import pytest
import torch

import oracle
from tests._np import check_close, max_rel_err, to_np
from workload import GLM, TINY, append_inputs, mla_inputs, paged_layout, to_pages

pytestmark = pytest.mark.gpu

TOL = {"f32": 1e-5, "bf16": 2e-2}
DEV = "cuda:0"


def _paged(x, T, page_size, seed):
    table, num_pages = paged_layout(T, page_size, seed)
    Lp = to_pages(x["Lc"], table, T, page_size, num_pages)
    Rp = to_pages(x["Rc"], table, T, page_size, num_pages)
    return table, Lp, Rp


@pytest.mark.parametrize("dtype,dims,page_size", [("f32", TINY, 16), ("bf16", GLM, 128), ("bf16", GLM, 256),
                                                  ("bf16", GLM, 64), ("f32", GLM, 128)])
@pytest.mark.parametrize("T,S", [([1], 1), ([129, 300, 64], 1), ([130, 257, 6], 6), ([5000, 700], 2)])
def test_decode_paged(cuda_lib, dtype, dims, page_size, T, S):
    x = mla_inputs(dims, len(T), S, T, max(T), dtype, 300 + sum(T) + S, "cpu")
    table, Lp, Rp = _paged(x, T, page_size, 5 + S)
    out = cuda_lib.decode_paged(x["q"].to(DEV), Lp.to(DEV), Rp.to(DEV), table.to(DEV), x["T"].to(DEV),
                                x["kv_b"].to(DEV), dims)
    assert cuda_lib.device_status() == 0
    tbl = table.tolist()
    ref = oracle.decode_absorbed(to_np(x["q"]), oracle.unpage(to_np(Lp), tbl, T), oracle.unpage(to_np(Rp), tbl, T),
                                 T, to_np(x["kv_b"]), dims.qk_nope, dims.softmax_scale)
    got = to_np(out)
    assert np.all(np.isfinite(got))
    check_close(got, ref, TOL[dtype])


def test_decode_paged_glm_b32_sampled(cuda_lib):
    """Batched GLM-5.2 decode (32 sequences of 1024..32768 keys) over a shuffled
    128-row page pool, checked on a sample of query rows."""
    from workload import seq_lengths
    T = seq_lengths(32, 1024, 32768, 41)
    x = mla_inputs(GLM, 32, 1, T, max(T), "bf16", 42, DEV)
    table, Lp, Rp = _paged(x, T, 128, 43)
    del x["Lc"], x["Rc"]
    out = to_np(cuda_lib.decode_paged(x["q"], Lp, Rp, table.to(DEV), x["T"], x["kv_b"], GLM))
    assert cuda_lib.device_status() == 0
    kvb = to_np(x["kv_b"])
    tbl = table.tolist()
    for b in (0, 7, 31):
        pos = T[b] - 1
        rows = [oracle.page_row(tbl, b, t, 128) for t in range(pos + 1)]
        Lb = to_np(Lp.view(-1, GLM.kv_lora)[rows])
        Rb = to_np(Rp.view(-1, GLM.qk_rope)[rows])
        ref = oracle.attend_absorbed(to_np(x["q"][b, 0]), Lb, Rb, kvb, GLM.qk_nope, pos, GLM.softmax_scale)
        check_close(out[b, 0], ref, TOL["bf16"], b)


@pytest.mark.parametrize("dtype,dims,page_size", [("f32", TINY, 8), ("bf16", GLM, 128)])
def test_sparse_decode_paged(cuda_lib, dtype, dims, page_size):
    T, S, k = [300, 1000], 2, 64
    x = mla_inputs(dims, 2, S, T, max(T), dtype, 17, "cpu")
    table, Lp, Rp = _paged(x, T, page_size, 18)
    g = torch.Generator().manual_seed(19)
    sel = torch.full((2, S, k), -1, dtype=torch.int32)
    nsel = torch.zeros(2, S, dtype=torch.int32)
    for b in range(2):
        for s in range(S):
            pos = T[b] - S + s
            n = min(k, pos + 1)
            idx = torch.randperm(pos + 1, generator=g)[:n].sort().values
            sel[b, s, :n] = idx.to(torch.int32)
            nsel[b, s] = n
    out = cuda_lib.sparse_decode_paged(x["q"].to(DEV), Lp.to(DEV), Rp.to(DEV), table.to(DEV), x["T"].to(DEV),
                                       x["kv_b"].to(DEV), sel.to(DEV), nsel.to(DEV), dims)
    assert cuda_lib.device_status() == 0
    tbl = table.tolist()
    ref = oracle.sparse_decode(to_np(x["q"]), oracle.unpage(to_np(Lp), tbl, T), oracle.unpage(to_np(Rp), tbl, T), T,
                               to_np(x["kv_b"]), sel.numpy(), nsel.numpy(), dims.qk_nope, dims.softmax_scale)
    check_close(to_np(out), ref, TOL[dtype])


def test_decode_paged_flags_bad_page(cuda_lib):
    T, page_size = [300, 200], 128
    x = mla_inputs(GLM, 2, 1, T, max(T), "bf16", 23, "cpu")
    table, Lp, Rp = _paged(x, T, page_size, 24)
    table[1, 1] = Lp.shape[0] + 5  # past the pool
    cuda_lib.decode_paged(x["q"].to(DEV), Lp.to(DEV), Rp.to(DEV), table.to(DEV), x["T"].to(DEV),
                          x["kv_b"].to(DEV), GLM)
    assert cuda_lib.device_status() & cuda_lib.MLA_DEV_BAD_INDEX
    assert cuda_lib.device_status() == 0


@pytest.mark.parametrize("dtype,dims,page_size", [("f32", TINY, 4), ("bf16", GLM, 128)])
def test_cache_append_paged(cuda_lib, dtype, dims, page_size):
    T, S = [130, 257, 6], 6
    table, num_pages = paged_layout(T, page_size, 29)
    tdt = torch.float32 if dtype == "f32" else torch.bfloat16
    gen = torch.Generator().manual_seed(30)
    Lp = torch.randn(num_pages, page_size, dims.kv_lora, generator=gen).to(tdt).to(DEV)
    Rp = torch.randn(num_pages, page_size, dims.qk_rope, generator=gen).to(tdt).to(DEV)
    Lp0, Rp0 = Lp.clone(), Rp.clone()
    x = append_inputs(dims, 3, S, dtype, 31, "cpu")
    cuda_lib.cache_append_paged(x["comp"].to(DEV), x["kv_a_ln"].to(DEV), table.to(DEV),
                                torch.tensor(T, dtype=torch.int32, device=DEV), Lp, Rp, dims, 1e-6)
    assert cuda_lib.device_status() == 0
    lc, rc, pos = oracle.cache_append(to_np(x["comp"]), to_np(x["kv_a_ln"]), 1e-6, T, dims.kv_lora)
    tbl = table.tolist()
    rows = [[oracle.page_row(tbl, b, int(pos[b, s]), page_size) for s in range(S)] for b in range(3)]
    Lflat, Rflat = Lp.view(-1, dims.kv_lora), Rp.view(-1, dims.qk_rope)
    got_l = np.stack([to_np(Lflat[r]) for r in rows])
    got_r = np.stack([to_np(Rflat[r]) for r in rows])
    tol = 1e-5 if dtype == "f32" else 2.0 ** -8
    assert np.all(np.abs(got_l - lc) <= tol * np.max(np.abs(lc), axis=-1, keepdims=True))
    assert np.all(np.abs(got_r - rc) <= tol * np.max(np.abs(rc), axis=-1, keepdims=True))
    keep = torch.ones(Lflat.shape[0], dtype=torch.bool, device=DEV)
    keep[[r for rr in rows for r in rr]] = False
    same = lambda a, b: torch.equal(a.view(torch.uint8) if a.dtype == torch.bfloat16 else a,
                                    b.view(torch.uint8) if b.dtype == torch.bfloat16 else b)
    assert same(Lflat[keep], Lp0.view(-1, dims.kv_lora)[keep])
    assert same(Rflat[keep], Rp0.view(-1, dims.qk_rope)[keep])

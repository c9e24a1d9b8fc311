"""GPU parity of the output projection (mla_o_proj, mla_decode_oproj)
against the fp64 oracle.

fp32 weights: within 1e-5 of the oracle (normwise).  bf16 weights: the
streaming path computes in fp32 (1e-5 as well); the tensor-core path for more
than 8 rows rounds x to bf16 first, so it is held to the bf16 bound 2e-2.
"""
import numpy as np
import pytest
import torch

import oracle
from tests._np import max_rel_err, to_np
from workload import GLM, TINY, mla_inputs

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


def _w(hidden, in_dim, dtype, seed):
    g = torch.Generator().manual_seed(seed)
    w = torch.randn(hidden, in_dim, generator=g) * 0.02
    return w.to(torch.bfloat16 if dtype == "bf16" else torch.float32)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
# (1 | 2 rows, in_dim a multiple of 2048, bf16) take the ring of whole W_O rows, other shapes the register
# GEMV; the 70000-row cases need more CTAs than there are SMs
@pytest.mark.parametrize("R,in_dim,hidden", [(1, 16384, 6144), (2, 16384, 777), (1, 4096, 100), (2, 2048, 70000),
                                             (3, 16384, 1000), (4, 16384, 6144), (8, 16384, 777), (5, 8192, 300),
                                             (6, 4096, 50), (7, 32768, 129), (4, 4096, 70000),
                                             (8, 64, 77), (5, 200, 64), (1, 8, 1), (2, 64, 30000)])
def test_o_proj_streaming(cuda_lib, dtype, R, in_dim, hidden):
    g = torch.Generator().manual_seed(R + in_dim + hidden)
    x = torch.randn(R, in_dim, generator=g)
    w = _w(hidden, in_dim, dtype, 2)
    y = cuda_lib.o_proj(x.to(DEV), w.to(DEV))
    ref = oracle.o_proj(to_np(x), to_np(w))
    assert max_rel_err(to_np(y), ref) < 1e-5


@pytest.mark.parametrize("R,dtype,tol", [(32, "bf16", 2e-2), (17, "bf16", 2e-2), (32, "f32", 1e-5)])
def test_o_proj_many_rows(cuda_lib, R, dtype, tol):
    """More than 8 rows: tensor-core GEMM for bf16 weights, 8-row passes for fp32."""
    in_dim, hidden = 16384, 6144
    g = torch.Generator().manual_seed(R)
    x = torch.randn(R, in_dim, generator=g)
    w = _w(hidden, in_dim, dtype, 3)
    y = cuda_lib.o_proj(x.to(DEV), w.to(DEV))
    assert cuda_lib.device_status() == 0
    ref = oracle.o_proj(to_np(x), to_np(w))
    assert max_rel_err(to_np(y), ref) < tol


@pytest.mark.parametrize("dtype,dims,T,S,hidden", [("bf16", GLM, [4096], 1, 6144), ("bf16", GLM, [300, 1000], 2, 640),
                                                   ("f32", TINY, [64, 9], 1, 40)])
def test_decode_then_o_proj(cuda_lib, dtype, dims, T, S, hidden):
    """mla_decode_oproj equals the oracle's decode followed by its projection."""
    x = mla_inputs(dims, len(T), S, T, max(T), dtype, 90 + S, "cpu")
    w = _w(hidden, dims.H * dims.v_head, dtype, 4)
    y = cuda_lib.decode_oproj(x["q"].to(DEV), x["Lc"].to(DEV), x["Rc"].to(DEV), x["T"].to(DEV),
                              x["kv_b"].to(DEV), w.to(DEV), dims)
    assert cuda_lib.device_status() == 0
    att = oracle.decode_absorbed(to_np(x["q"]), to_np(x["Lc"]), to_np(x["Rc"]), T, to_np(x["kv_b"]), dims.qk_nope,
                                 dims.softmax_scale)
    ref = oracle.o_proj(att.reshape(len(T) * S, -1), to_np(w)).reshape(len(T), S, hidden)
    assert max_rel_err(to_np(y), ref) < (2e-2 if dtype == "bf16" else 1e-5)

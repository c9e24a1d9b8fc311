"""CPU model of the FP8 decode's roundings (test helper, float64).

The FP8 path computes with three values rounded to E4M3: the cache codes (the
input), each query row's absorbed latent query (scale = its largest magnitude
/ 448), and the softmax probabilities (the value-product operand; row sums
stay fp32, and the running max moves only when it grows by more than 2^8, as
the kernel's lazy rescale does).  fp8_row_model() repeats those roundings
around the exact arithmetic for one query row; its distance from the oracle's
exact attention over the dequantised cache is the error the roundings alone
produce, which the GPU tests compare the kernels' error with.
"""
import math

import numpy as np
import pytest

import oracle
from workload import GLM

def _e4m3(x):
    return oracle.e4m3_decode(oracle.e4m3_encode(x))


def _bf16(x):
    torch = pytest.importorskip("torch")
    return torch.tensor(np.asarray(x, np.float32)).bfloat16().double().numpy()


def fp8_row_model(q, x8, R, kvb, T, lat_scale, tau=8.0, tile=128):
    """Absorbed decode of one query row at position T - 1 over the E4M3 values
    x8 [T, kv_lora] (codes decoded, before lat_scale) and rope keys R [T, 64],
    with the FP8 kernel's roundings."""
    Dn = GLM.qk_nope
    qabs = _bf16(np.einsum("hi,hil->hl", q[:, :Dn], kvb[:, :Dn]))       # the absorb kernel's bf16 output
    qrot = _bf16(oracle.rope_interleave(q[:, Dn:], T - 1))
    sq = np.max(np.abs(qabs), axis=1) / 448.0
    q8 = _e4m3(qabs / sq[:, None])
    qr = _bf16(qrot / (lat_scale * sq[:, None]))
    f = GLM.softmax_scale / math.log(2.0) * lat_scale * sq             # score factor (log2 units)
    S = (q8 @ x8.T + qr @ R.T) * f[:, None]
    H = S.shape[0]
    m = np.full(H, -np.inf)
    l = np.zeros(H)
    O = np.zeros((H, x8.shape[1]))
    for t0 in range(0, T, tile):
        st = S[:, t0:t0 + tile]
        tm = st.max(axis=1)
        mn = np.where(tm > m + tau, tm, m)
        al = np.where(np.isfinite(m), 2.0 ** (m - mn), 0.0)
        O *= al[:, None]
        l *= al
        m = mn
        p = 2.0 ** (st - m[:, None])
        l += p.sum(axis=1)
        O += _e4m3(p) @ x8[t0:t0 + tile]
    return np.einsum("hjl,hl->hj", kvb[:, Dn:], lat_scale * O / l[:, None])

"""The FP8 decode's tolerance, checked on a CPU model of its roundings (CPU only).

The FP8 path computes with three values rounded to E4M3: the cache codes (the
input), each query row's absorbed latent query (scale = its largest magnitude /
448), and the softmax probabilities (the value-product operand; row sums stay
fp32, and the running max moves only when it grows by more than 2^8, as the
kernel's lazy rescale does).  This model repeats those roundings in float64
around the exact arithmetic and compares with the oracle's exact attention over
the dequantised cache.  The GPU parity tests hold the kernels to u = 2^-4
(normwise); here the model must stay below u on the same kind of inputs, and
the error must be of the order the roundings predict, far above fp32 noise.
"""
import math

import numpy as np
import pytest

import oracle
from tests._np import max_rel_err, to_np
from workload import GLM, fp8_latent_codes, mla_inputs

U_E4M3 = 2.0 ** -4
LAT_SCALE = 0.05


def _e4m3(x):
    return oracle.e4m3_decode(oracle.e4m3_encode(x))


def _bf16(x):
    torch = pytest.importorskip("torch")
    return torch.tensor(np.asarray(x, np.float32)).bfloat16().double().numpy()


def _model(q, x8, R, kvb, T, lat_scale, tau=8.0, tile=128):
    """Absorbed decode of one query row with the FP8 kernel's roundings."""
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


@pytest.mark.parametrize("T,seed", [(4096, 1), (1000, 2), (300, 3), (33, 4)])
def test_fp8_model_within_the_stated_bound(T, seed):
    x = mla_inputs(GLM, 1, 1, [T], T, "bf16", seed, "cpu")
    q, R, kvb = to_np(x["q"])[0, 0], to_np(x["Rc"])[0], to_np(x["kv_b"])
    codes = fp8_latent_codes(1, [T], T, GLM.kv_lora, seed, "cpu").numpy()[0]
    x8 = oracle.e4m3_decode(codes)
    ref = oracle.decode_absorbed(q[None, None], (LAT_SCALE * x8)[None], R[None], [T], kvb, GLM.qk_nope,
                                 GLM.softmax_scale)[0, 0]
    err = max_rel_err(_model(q, x8, R, kvb, T, LAT_SCALE), ref)
    assert 1e-3 < err < U_E4M3, err

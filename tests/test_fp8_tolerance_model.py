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
import oracle
import pytest
from tests._fp8_model import fp8_row_model
from tests._np import max_rel_err, to_np
from workload import GLM, fp8_latent_codes, mla_inputs

U_E4M3 = 2.0 ** -4
LAT_SCALE = 0.05


@pytest.mark.parametrize("T,seed", [(4096, 1), (1000, 2), (300, 3), (33, 4)])
def test_fp8_model_within_the_stated_bound(T, seed):
    x = mla_inputs(GLM, 1, 1, [T], T, "bf16", seed, "cpu")
    q, R, kvb = to_np(x["q"])[0, 0], to_np(x["Rc"])[0], to_np(x["kv_b"])
    codes = fp8_latent_codes(1, [T], T, GLM.kv_lora, seed, "cpu").numpy()[0]
    x8 = oracle.e4m3_decode(codes)
    ref = oracle.decode_absorbed(q[None, None], (LAT_SCALE * x8)[None], R[None], [T], kvb, GLM.qk_nope,
                                 GLM.softmax_scale)[0, 0]
    err = max_rel_err(fp8_row_model(q, x8, R, kvb, T, LAT_SCALE), ref)
    assert 1e-3 < err < U_E4M3, err

"""The seeded input generators (CPU only): the same seed gives the same tensors,
rows past each sequence's length are poisoned, and the shapes and value ranges
are the ones the tests and the bench rely on."""
import numpy as np
import torch

import oracle
from workload import (GLM, TINY, E4M3_NAN, append_inputs, dsa_inputs, fp8_latent_codes, mla_inputs, paged_layout,
                      seq_lengths, to_pages)


def test_same_seed_same_inputs():
    a = mla_inputs(TINY, 2, 2, [9, 5], 12, "f32", 3)
    b = mla_inputs(TINY, 2, 2, [9, 5], 12, "f32", 3)
    c = mla_inputs(TINY, 2, 2, [9, 5], 12, "f32", 4)
    for k in a:
        assert torch.equal(torch.nan_to_num(a[k]), torch.nan_to_num(b[k])), k
    assert not torch.equal(a["q"], c["q"])


def test_rows_past_the_length_are_nan_and_the_rest_finite():
    T = [9, 5]
    x = mla_inputs(TINY, 2, 1, T, 12, "f32", 5)
    for b, t in enumerate(T):
        assert torch.isnan(x["Lc"][b, t:]).all() and torch.isnan(x["Rc"][b, t:]).all()
        assert torch.isfinite(x["Lc"][b, :t]).all() and torch.isfinite(x["Rc"][b, :t]).all()
    assert x["T"].dtype == torch.int32 and x["T"].tolist() == T
    assert x["kv_b"].shape == (TINY.H, TINY.qk_nope + TINY.v_head, TINY.kv_lora)


def test_fp8_codes_are_finite_before_the_length_and_nan_after():
    T = [7, 3]
    c = fp8_latent_codes(2, T, 10, 32, 6)
    assert c.dtype == torch.uint8 and c.shape == (2, 10, 32)
    vals = oracle.e4m3_decode(c.numpy())
    for b, t in enumerate(T):
        assert np.all(np.isfinite(vals[b, :t]))
        assert np.all(c[b, t:].numpy() == E4M3_NAN)
    mags = np.abs(vals[0, :7])
    assert mags.min() >= 2.0 ** -3 and mags.max() <= 1.875 * 2.0 ** 4   # exponent field 4..11
    assert fp8_latent_codes(2, T, 10, 32, 6).equal(c)


def test_dsa_inputs_are_small_integers():
    d = dsa_inputs(1, 1, [40], 48, 2, 8, 7)
    for k in ("q_idx", "w"):
        v = d[k].numpy()
        assert np.all(v == np.round(v)) and np.abs(v).max() <= 4
    ic = d["Ic"].numpy()[0, :40]
    assert np.all(ic == np.round(ic)) and np.abs(ic).max() <= 4
    assert np.isnan(d["Ic"].numpy()[0, 40:]).all()


def test_seq_lengths_and_paged_layout():
    T = seq_lengths(32, 1024, 32768, 41)
    assert len(T) == 32 and min(T) >= 1024 and max(T) <= 32768 and T == seq_lengths(32, 1024, 32768, 41)
    table, num_pages = paged_layout([130, 257, 6], 128, 9)
    used = [p for row in table.tolist() for p in row if p >= 0]
    assert len(used) == len(set(used)) == 2 + 3 + 1 and num_pages >= len(used)
    x = torch.arange(3 * 257 * 2, dtype=torch.float32).view(3, 257, 2)
    pool = to_pages(x, table, [130, 257, 6], 128, num_pages)
    back = oracle.unpage(pool.numpy(), table.tolist(), [130, 257, 6])
    for b, t in enumerate([130, 257, 6]):
        np.testing.assert_array_equal(back[b, :t], x[b, :t].numpy())


def test_append_inputs_shapes():
    a = append_inputs(GLM, 2, 3, "bf16", 8, index_hd=16)
    assert a["comp"].shape == (2, 3, GLM.kv_lora + GLM.qk_rope) and a["comp"].dtype == torch.bfloat16
    assert a["kv_a_ln"].shape == (GLM.kv_lora,)
    assert a["k_idx"].shape == (2, 3, 16) and a["ln_w"].shape == (16,) and a["ln_b"].shape == (16,)

"""The C ABI library builds, loads and exports every symbol of include/mla.h (CPU only).

No compute call is made here; host-side argument checks that return before
any CUDA call are exercised with null pointers.
"""
import ctypes
import os
import re

import pytest

import mla_latent_kv_06_gb300 as mla
from mla_latent_kv_06_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return mla.load()


def _header_symbols():
    src = open(os.path.join(ROOT, "include", "mla.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"\b([a-z_][a-z0-9_]*)\s*\(", src)
    return sorted({n for n in names if n.startswith(("mla_", "dsa_"))})


def test_header_lists_match_binding():
    assert sorted(mla.EXPORTS) == _header_symbols()


def test_library_exports_every_header_symbol(lib):
    for name in _header_symbols():
        assert hasattr(lib, name), name
    assert lib.mla_abi_version() == 1


def test_built_for_sm103a_only():
    assert _build.ARCH == ["-gencode", "arch=compute_103a,code=sm_103a"]


def test_host_rejects_bad_arguments_without_a_gpu(lib):
    d = mla.MlaDims(64, 192, 64, 512, 256, 0.0, 0.0)
    # null tensors
    rc = lib.mla_decode_absorbed(ctypes.byref(d), mla.MLA_BF16, 1, 1, None, None, None, 16, None, None,
                                 None, None, 0, None)
    assert rc == mla.MLA_ERR_INVALID
    assert b"null" in lib.mla_last_error()
    # odd rotary width
    bad = mla.MlaDims(64, 192, 63, 512, 256, 0.0, 0.0)
    assert lib.mla_decode_absorbed(ctypes.byref(bad), 1, 1, 1, None, None, None, 16, None, None, None,
                                   None, 0, None) == mla.MLA_ERR_INVALID
    # unknown dtype, S > T_cap, non-positive topk
    assert lib.mla_decode_absorbed(ctypes.byref(d), 7, 1, 1, None, None, None, 16, None, None, None,
                                   None, 0, None) == mla.MLA_ERR_INVALID
    assert lib.mla_decode_absorbed(ctypes.byref(d), 1, 1, 6, None, None, None, 5, None, None, None,
                                   None, 0, None) == mla.MLA_ERR_INVALID
    assert lib.mla_sparse_decode(ctypes.byref(d), 1, 1, 1, None, None, None, 16, None, None, None, None,
                                 0, None, None, 0, None) == mla.MLA_ERR_INVALID
    assert lib.dsa_topk_select(1, 1, None, 16, None, 0, None, None, None, 0, None) == mla.MLA_ERR_INVALID
    assert lib.dsa_index_scores(0, 1, 32, 128, None, None, None, 16, None, None, None) == mla.MLA_ERR_INVALID
    assert lib.mla_prefill_naive(ctypes.byref(d), 1, 1, 4, -1, None, None, None, None, None, None, 0,
                                 None) == mla.MLA_ERR_INVALID
    # cache writers: null tensors, S > T_cap, negative eps, odd / too wide rotary part
    p = ctypes.c_void_p(16)
    assert lib.mla_cache_append(ctypes.byref(d), 1, 1, 1, None, p, 1e-6, 8, p, p, p, None) == mla.MLA_ERR_INVALID
    assert lib.mla_cache_append(ctypes.byref(d), 1, 1, 9, p, p, 1e-6, 8, p, p, p, None) == mla.MLA_ERR_INVALID
    assert lib.mla_cache_append(ctypes.byref(d), 1, 1, 1, p, p, -1.0, 8, p, p, p, None) == mla.MLA_ERR_INVALID
    wide = mla.MlaDims(64, 192, 258, 512, 256, 0.0, 0.0)
    assert lib.mla_cache_append(ctypes.byref(wide), 1, 1, 1, p, p, 1e-6, 8, p, p, p,
                                None) == mla.MLA_ERR_UNSUPPORTED
    assert lib.dsa_index_key_append(1, 1, 128, 63, p, p, None, 1e-6, 1e4, 8, p, p, None) == mla.MLA_ERR_INVALID
    assert lib.dsa_index_key_append(1, 1, 128, 130, p, p, None, 1e-6, 1e4, 8, p, p, None) == mla.MLA_ERR_INVALID
    assert lib.dsa_index_key_append(1, 1, 600, 300, p, p, None, 1e-6, 1e4, 8, p, p,
                                    None) == mla.MLA_ERR_UNSUPPORTED
    assert lib.dsa_index_key_append(1, 1, 128, 64, None, p, None, 1e-6, 1e4, 8, p, p, None) == mla.MLA_ERR_INVALID
    # paged entries: null block table, zero page size, capacity below S, pool of 2^31 rows
    assert lib.mla_decode_paged(ctypes.byref(d), 1, 1, 1, p, p, p, 4, 128, None, 2, p, p, p, None, 0,
                                None) == mla.MLA_ERR_INVALID
    assert lib.mla_decode_paged(ctypes.byref(d), 1, 1, 1, p, p, p, 4, 0, p, 2, p, p, p, None, 0,
                                None) == mla.MLA_ERR_INVALID
    assert lib.mla_decode_paged(ctypes.byref(d), 1, 1, 9, p, p, p, 4, 2, p, 2, p, p, p, None, 0,
                                None) == mla.MLA_ERR_INVALID
    assert lib.mla_decode_paged(ctypes.byref(d), 1, 1, 1, p, p, p, 1 << 24, 1 << 8, p, 2, p, p, p, None, 0,
                                None) == mla.MLA_ERR_UNSUPPORTED
    assert lib.mla_sparse_decode_paged(ctypes.byref(d), 1, 1, 1, p, p, p, 4, 128, p, 2, p, p, p, p, 0, p, None, 0,
                                       None) == mla.MLA_ERR_INVALID
    assert lib.mla_cache_append_paged(ctypes.byref(d), 1, 1, 1, p, p, 1e-6, p, p, 4, 128, None, 2, p,
                                      None) == mla.MLA_ERR_INVALID
    assert lib.mla_decode_paged_workspace_size(ctypes.byref(d), 1, 1, 1, 2, 64) == 0  # not a multiple of 128
    assert lib.mla_decode_paged_workspace_size(ctypes.byref(d), 1, 1, 1, 2, 128) > 0
    # FP8 cache: scale not positive / not finite, other geometries, page sizes off 128
    tiny = mla.MlaDims(4, 16, 8, 32, 16, 0.0, 0.0)
    for sc in (0.0, -1.0, float("inf"), float("nan")):
        assert lib.mla_decode_fp8(ctypes.byref(d), 1, 1, p, p, p, sc, 16, p, p, p, None, 0,
                                  None) == mla.MLA_ERR_INVALID
        assert lib.mla_cache_append_fp8(ctypes.byref(d), 1, 1, p, p, 1e-6, sc, 8, p, p, p,
                                        None) == mla.MLA_ERR_INVALID
    assert lib.mla_cache_append_fp8(ctypes.byref(d), 1, 1, p, p, 1e-6, 1e-39, 8, p, p, p,
                                    None) == mla.MLA_ERR_INVALID  # 1 / lat_scale overflows
    assert lib.mla_decode_fp8(ctypes.byref(tiny), 1, 1, p, p, p, 0.01, 16, p, p, p, None, 0,
                              None) == mla.MLA_ERR_UNSUPPORTED
    assert lib.mla_decode_fp8(ctypes.byref(d), 1, 1, None, p, p, 0.01, 16, p, p, p, None, 0,
                              None) == mla.MLA_ERR_INVALID
    assert lib.mla_decode_fp8_paged(ctypes.byref(d), 1, 1, p, p, p, 0.01, 4, 64, p, 2, p, p, p, None, 0,
                                    None) == mla.MLA_ERR_UNSUPPORTED
    assert lib.mla_cache_append_fp8_paged(ctypes.byref(d), 1, 1, p, p, 1e-6, 0.01, p, p, 4, 128, None, 2, p,
                                          None) == mla.MLA_ERR_INVALID
    assert lib.mla_decode_fp8_workspace_size(ctypes.byref(tiny), 1, 1, 16) == 0
    assert lib.mla_decode_fp8_workspace_size(ctypes.byref(d), 1, 1, 16) > 0


def test_workspace_sizes_are_host_only(lib):
    d = mla.MlaDims(4, 16, 8, 32, 16, 0.0, 0.0)
    assert lib.mla_decode_absorbed_workspace_size(ctypes.byref(d), mla.MLA_F32, 1, 1, 64) == 0
    n = lib.mla_prefill_naive_workspace_size(ctypes.byref(d), mla.MLA_F32, 2, 3, 5)
    assert n >= 2 * 8 * 4 * 32 * 4 and n % 256 == 0


def test_product_path_does_not_use_the_oracle():
    pkg = os.path.join(ROOT, "mla_latent_kv_06_gb300")
    for dirpath, _, files in os.walk(pkg):
        for fn in files:
            if fn.endswith((".py", ".cu", ".cuh", ".h")):
                src = open(os.path.join(dirpath, fn)).read()
                assert "import oracle" not in src and "from oracle" not in src, fn

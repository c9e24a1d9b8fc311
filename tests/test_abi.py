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


def test_host_rejects_bad_arguments_of_the_fused_and_projection_calls(lib):
    d = mla.MlaDims(64, 192, 64, 512, 256, 0.0, 0.0)
    p = ctypes.c_void_p(256)
    # fused selection: sizes, null tensors, a query block too large for one CTA, missing workspace
    assert lib.dsa_select(0, 1, 32, 128, p, p, p, 16, p, 8, p, p, p, None, 0, None) == mla.MLA_ERR_INVALID
    assert lib.dsa_select(1, 1, 32, 128, None, p, p, 16, p, 8, p, p, p, None, 0, None) == mla.MLA_ERR_INVALID
    assert lib.dsa_select(1, 1, 512, 512, p, p, p, 16, p, 8, p, p, p, None, 0, None) == mla.MLA_ERR_UNSUPPORTED
    assert lib.dsa_select(1, 1, 32, 128, p, p, p, 16, p, 8, p, p, p, None, 0, None) == mla.MLA_ERR_INVALID
    assert b"workspace" in lib.mla_last_error()
    # output projection: sizes, in_dim not a multiple of 8, dtype, null and misaligned pointers
    assert lib.mla_o_proj(0, 64, 8, mla.MLA_BF16, p, p, p, None, 0, None) == mla.MLA_ERR_INVALID
    assert lib.mla_o_proj(1, 60, 8, mla.MLA_BF16, p, p, p, None, 0, None) == mla.MLA_ERR_INVALID
    assert lib.mla_o_proj(1, 64, 8, 7, p, p, p, None, 0, None) == mla.MLA_ERR_INVALID
    assert lib.mla_o_proj(1, 64, 8, mla.MLA_BF16, None, p, p, None, 0, None) == mla.MLA_ERR_INVALID
    assert lib.mla_o_proj(1, 64, 8, mla.MLA_BF16, ctypes.c_void_p(8), p, p, None, 0, None) == mla.MLA_ERR_INVALID
    # decode + projection: S > T_cap, null workspace (the attention output lives there)
    assert lib.mla_decode_oproj(ctypes.byref(d), 1, 1, 4, p, p, p, 2, p, p, p, 8, p, p, 1 << 30,
                                None) == mla.MLA_ERR_INVALID
    assert lib.mla_decode_oproj(ctypes.byref(d), 1, 1, 1, p, p, p, 16, p, p, p, 8, p, None, 0,
                                None) == mla.MLA_ERR_INVALID
    # sparse decode of several layers: L < 1, null pointer arrays, a null entry in one,
    # projection weights without outputs, a misaligned projection weight
    arr = (ctypes.c_void_p * 2)(256, 256)
    hole = (ctypes.c_void_p * 2)(256, None)
    odd = (ctypes.c_void_p * 2)(256, 8)

    def layers(L, q, rc, w_o, y):
        return lib.mla_sparse_decode_layers(ctypes.byref(d), 1, L, 1, 1, q, arr, rc, 16, p, arr, p, p, 8, arr, w_o,
                                            64, y, p, 1 << 30, None)
    assert layers(0, arr, arr, None, None) == mla.MLA_ERR_INVALID
    assert layers(2, None, arr, None, None) == mla.MLA_ERR_INVALID
    assert layers(2, arr, hole, None, None) == mla.MLA_ERR_INVALID
    assert b"layer 1" in lib.mla_last_error()
    assert layers(2, arr, arr, arr, None) == mla.MLA_ERR_INVALID
    assert layers(2, arr, arr, odd, arr) == mla.MLA_ERR_INVALID
    assert b"aligned" in lib.mla_last_error()
    # prefill without caller workspace: negative pos_base, rebuilt KV above the static scratch
    assert lib.mla_prefill_naive_noalloc(ctypes.byref(d), 1, 1, 4, -1, p, p, p, p, p, None) == mla.MLA_ERR_INVALID
    assert lib.mla_prefill_naive_noalloc(ctypes.byref(d), 1, 1, 2048, 8192, p, p, p, p, p,
                                         None) == mla.MLA_ERR_INVALID


def test_host_only_sizes_and_counts(lib):
    d = mla.MlaDims(64, 192, 64, 512, 256, 0.0, 0.0)
    tiny = mla.MlaDims(4, 16, 8, 32, 16, 0.0, 0.0)
    assert lib.dsa_select_workspace_size(0, 1, 32, 128, 16, 8) == 0
    assert lib.dsa_select_workspace_size(1, 1, 32, 128, 1024, 64) > 0      # tensor-core indexer histograms
    assert lib.dsa_select_workspace_size(1, 1, 4, 32, 1024, 64) == 0       # CUDA-core indexer: none
    assert lib.dsa_topk_select_workspace_size(1, 1, 16, 0) == 0
    assert lib.mla_sparse_decode_workspace_size(ctypes.byref(d), mla.MLA_BF16, 1, 1, 0) == 0
    assert lib.mla_sparse_decode_workspace_size(ctypes.byref(d), mla.MLA_BF16, 1, 1, 2048) > 0
    assert lib.mla_o_proj_workspace_size(0, 64, 8, mla.MLA_BF16) == 0
    assert lib.mla_decode_oproj_workspace_size(ctypes.byref(d), mla.MLA_BF16, 1, 1, 4096, 6144) > 0
    assert lib.mla_decode_oproj_workspace_size(ctypes.byref(d), mla.MLA_BF16, 1, 2, 1, 6144) == 0
    # kernels per tensor-core decode call: absorb, attention, combine; five for more than 8 rows;
    # one more (the gather) for the sparse path; one kernel on the CUDA cores
    assert lib.mla_decode_launch_count(ctypes.byref(d), mla.MLA_BF16, 1, 1, 0) == 3
    assert lib.mla_decode_launch_count(ctypes.byref(d), mla.MLA_BF16, 32, 1, 0) == 5
    assert lib.mla_decode_launch_count(ctypes.byref(d), mla.MLA_BF16, 4, 1, 1) == 4
    assert lib.mla_decode_launch_count(ctypes.byref(tiny), mla.MLA_F32, 1, 1, 0) == 1


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


def test_header_is_c_and_the_library_links_from_c(tmp_path, lib):
    """include/mla.h compiles as C99 with warnings as errors, and a C program
    linked against libmla.so calls host-only entry points (no GPU needed)."""
    import shutil
    import subprocess
    if shutil.which("gcc") is None:
        pytest.skip("no C compiler")
    prog = tmp_path / "abi.c"
    prog.write_text(r"""
#include <stdio.h>
#include "mla.h"
int main(void) {
  mla_dims d = {64, 192, 64, 512, 256, 0.0f, 0.0f};
  size_t ws = mla_decode_absorbed_workspace_size(&d, MLA_BF16, 1, 1, 4096);
  int bad = mla_decode_absorbed(&d, MLA_BF16, 1, 1, NULL, NULL, NULL, 16, NULL, NULL, NULL, NULL, 0, NULL);
  printf("%d %zu %d %d\n", mla_abi_version(), ws, bad, mla_last_error()[0] != 0);
  return 0;
}
""")
    libdir = os.path.dirname(mla.LIB_PATH)
    exe = tmp_path / "abi"
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"), str(prog), "-o",
                    str(exe), "-L", libdir, "-lmla", "-Wl,-rpath," + libdir], check=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.split()
    assert out[0] == "1" and int(out[1]) > 0 and int(out[2]) == mla.MLA_ERR_INVALID and out[3] == "1"


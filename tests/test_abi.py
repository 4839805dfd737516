"""The C-ABI library loads and exports every symbol include/dsa.h declares; host
validation rejects bad arguments before anything reaches the GPU (no GPU needed)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def header_functions():
    text = open(os.path.join(ROOT, "include", "dsa.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(dsa_[a-z_0-9]+)\s*\(", text)))


@pytest.fixture(scope="module")
def dsa():
    import __graft_entry__
    __graft_entry__.build()
    import dsa_indexed_sparse_gb300 as m
    return m


def test_every_declared_function_is_exported(dsa):
    names = header_functions()
    assert len(names) >= 11
    lib = ctypes.CDLL(dsa.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), n
    assert sorted(dsa.EXPORTED) == names


def test_version_and_status_strings(dsa):
    assert dsa.abi_version() == 1
    for code, name in dsa.STATUS_NAMES.items():
        assert dsa._lib.dsa_status_string(code).decode() == name


def test_host_validation_rejects_bad_arguments(dsa):
    lib = dsa._lib
    # NULL descriptors
    assert lib.dsa_indexer_scores(None, None, None, 0, None) == 1
    assert lib.dsa_topk(None, None, 0, 1, None, None) == 1
    assert "NULL" in dsa.last_error()
    # T = B * q_per_seq violated
    s = dsa.SeqDesc(B=2, T=3, max_ctx=128, q_per_seq=1, q_seq=16, q_pos=16, block_table=16,
                    bt_stride=2, page_size=64, cache_rows=256)
    assert lib.dsa_topk(ctypes.byref(s), 16, 128, 8, 16, None) == 1
    assert "q_per_seq" in dsa.last_error()
    # page table too narrow for max_ctx
    s = dsa.SeqDesc(B=1, T=1, max_ctx=1000, q_per_seq=1, q_seq=16, q_pos=16, block_table=16,
                    bt_stride=2, page_size=64, cache_rows=4096)
    assert lib.dsa_topk(ctypes.byref(s), 16, 1024, 8, 16, None) == 1
    assert "bt_stride" in dsa.last_error()
    # K = 0
    s.bt_stride = 16
    assert lib.dsa_topk(ctypes.byref(s), 16, 1024, 0, 16, None) == 1
    # FP8 latent rows only for 512 + 64 dims
    m = dsa.MlaDesc(H=4, d_latent=64, d_rope=16, dtype=dsa.DSA_E4M3, q=16, kv_cache=16, row_bytes=656,
                    softmax_scale=0.1)
    assert lib.dsa_sparse_mla_attn_workspace_size(ctypes.byref(s), ctypes.byref(m), 32) == 0
    assert lib.dsa_sparse_mla_attn(ctypes.byref(s), ctypes.byref(m), 16, 32, 16, None, None, 0, None) == 2
    # misaligned score buffer for the indexer
    x = dsa.IndexerDesc(H_I=4, D_I=32, dtype=dsa.DSA_F32, q=16, q_scale=None, w=16, k_cache=16, k_scale=None)
    assert lib.dsa_indexer_scores(ctypes.byref(s), ctypes.byref(x), 20, 1024, None) == 1
    # decode step without a workspace
    assert lib.dsa_decode_step(ctypes.byref(s), ctypes.byref(x), ctypes.byref(m), 32, 16, None, None,
                               None, 0, None) == 3
    # MXFP8 index keys: D_I a multiple of 32, both scale arrays required
    x = dsa.IndexerDesc(H_I=4, D_I=48, dtype=dsa.DSA_MXFP8_E4M3, q=16, q_scale=16, w=16, k_cache=16, k_scale=16)
    assert lib.dsa_indexer_scores(ctypes.byref(s), ctypes.byref(x), 16, 1024, None) == 2
    assert "multiple of 32" in dsa.last_error()
    x = dsa.IndexerDesc(H_I=4, D_I=64, dtype=dsa.DSA_MXFP8_E4M3, q=16, q_scale=None, w=16, k_cache=16, k_scale=16)
    assert lib.dsa_indexer_scores(ctypes.byref(s), ctypes.byref(x), 16, 1024, None) == 1
    # per-128-tile FP8 rows: 512 + 64 dims only; the latent writer does not produce them
    m = dsa.MlaDesc(H=4, d_latent=64, d_rope=16, dtype=dsa.DSA_E4M3_T128, q=16, kv_cache=16, row_bytes=656,
                    softmax_scale=0.1)
    assert lib.dsa_sparse_mla_attn(ctypes.byref(s), ctypes.byref(m), 16, 32, 16, None, None, 0, None) == 2
    m = dsa.MlaDesc(H=128, d_latent=512, d_rope=64, dtype=dsa.DSA_E4M3_T128, q=16, kv_cache=16, row_bytes=656,
                    softmax_scale=0.1)
    # (the tile-128 writer exists; D_I rules for the MXFP8 key writer)
    assert lib.dsa_index_cache_append_mx(ctypes.byref(s), 48, dsa.DSA_F32, 16, 16, 16, None) == 2


def test_host_validation_of_writers_prolog_and_debug_switch(dsa):
    """Each rejection below returns before the library's first CUDA call."""
    lib = dsa._lib
    s = dsa.SeqDesc(B=1, T=1, max_ctx=1000, q_per_seq=1, q_seq=16, q_pos=16, block_table=16,
                    bt_stride=16, page_size=64, cache_rows=4096)
    # index-key writer: D_I in [4, 1024] and a multiple of 4, fp32 or bf16 sources, pointers non-NULL and aligned
    assert lib.dsa_index_cache_append(ctypes.byref(s), 6, dsa.DSA_F32, 16, 16, 16, None) == 2
    assert lib.dsa_index_cache_append(ctypes.byref(s), 64, dsa.DSA_E4M3, 16, 16, 16, None) == 2
    assert lib.dsa_index_cache_append(ctypes.byref(s), 64, dsa.DSA_F32, None, 16, 16, None) == 1
    assert lib.dsa_index_cache_append(ctypes.byref(s), 64, dsa.DSA_BF16, 16, 24, 16, None) == 1
    assert "aligned" in dsa.last_error()
    # latent writer: copied rows move 16-byte vectors; pointers non-NULL and aligned
    m = dsa.MlaDesc(H=4, d_latent=60, d_rope=2, dtype=dsa.DSA_BF16, q=16, kv_cache=16, row_bytes=128,
                    softmax_scale=0.1)
    assert lib.dsa_latent_cache_append(ctypes.byref(s), ctypes.byref(m), 16, 16, None) == 2
    m = dsa.MlaDesc(H=4, d_latent=64, d_rope=16, dtype=dsa.DSA_BF16, q=16, kv_cache=16, row_bytes=160,
                    softmax_scale=0.1)
    assert lib.dsa_latent_cache_append(ctypes.byref(s), ctypes.byref(m), None, 16, None) == 1
    assert lib.dsa_latent_cache_append(ctypes.byref(s), ctypes.byref(m), 16, 8, None) == 1
    # prolog: D_I == 128, 1 <= H_I <= 128, d_model and d_q positive multiples of 64
    ok = dict(d_model=256, d_q=128, H_I=8, D_I=128, x=16, x_q=16, w_q=16, w_k=16, w_w=16, gamma=16, beta=16)
    for bad in (dict(D_I=64), dict(H_I=0), dict(H_I=129), dict(d_model=100), dict(d_q=0)):
        pd = dsa.PrologDesc(**{**ok, **bad})
        assert lib.dsa_indexer_prolog_workspace_size(ctypes.byref(s), ctypes.byref(pd)) == 0, bad
        assert lib.dsa_indexer_prolog(ctypes.byref(s), ctypes.byref(pd), 16, 16, 16, 16, 16, 16, 1 << 20,
                                      None) == 2, bad
    assert lib.dsa_indexer_prolog(ctypes.byref(s), None, 16, 16, 16, 16, 16, 16, 1 << 20, None) == 1
    pd = dsa.PrologDesc(**{**ok, "x": None})
    assert lib.dsa_indexer_prolog(ctypes.byref(s), ctypes.byref(pd), 16, 16, 16, 16, 16, 16, 1 << 20, None) == 1
    pd = dsa.PrologDesc(**ok)
    assert lib.dsa_indexer_prolog(ctypes.byref(s), ctypes.byref(pd), 8, 16, 16, 16, 16, 16, 1 << 20, None) == 1
    # K outside [1, 16384]: no workspace size, and the static-workspace step says unsupported
    m = dsa.MlaDesc(H=128, d_latent=512, d_rope=64, dtype=dsa.DSA_BF16, q=16, kv_cache=16, row_bytes=1152,
                    softmax_scale=0.1)
    x = dsa.IndexerDesc(H_I=64, D_I=128, dtype=dsa.DSA_E4M3, q=16, q_scale=16, w=16, k_cache=16, k_scale=16)
    for K in (0, 16385):
        assert lib.dsa_decode_workspace_size(ctypes.byref(s), ctypes.byref(x), ctypes.byref(m), K) == 0
        assert lib.dsa_decode_step_static_ws(ctypes.byref(s), ctypes.byref(x), ctypes.byref(m), K, 16, None, None,
                                             None) == 2
    # failure-detection switch: the wait bound must lie in [1 us, 1 s]; switching off always succeeds
    assert lib.dsa_debug_withhold_arrival(1, 999) == 1
    assert lib.dsa_debug_withhold_arrival(1, 2_000_000_000) == 1
    assert lib.dsa_debug_withhold_arrival(0, 0) == 0


C_CALLER = r"""
#include <stdio.h>
#include <string.h>
#include "dsa.h"
int main(void) {
  if (dsa_abi_version() != 1) return 1;
  /* a NULL descriptor is rejected on the host, before any CUDA call */
  if (dsa_topk(NULL, NULL, 0, 1, NULL, NULL) != DSA_ERR_INVALID_ARG) return 2;
  if (strcmp(dsa_status_string(DSA_ERR_TIMEOUT), "DSA_ERR_TIMEOUT") != 0) return 3;
  if (strstr(dsa_last_error(), "NULL") == NULL) return 4;
  printf("ok\n");
  return 0;
}
"""


def test_header_is_plain_c_and_a_c_program_links(dsa, tmp_path):
    """include/dsa.h compiles as strict C99, and a C program links against libdsa.so and calls it."""
    import shutil
    import subprocess
    if shutil.which("gcc") is None:
        pytest.skip("gcc not found")
    src = tmp_path / "caller.c"
    src.write_text(C_CALLER)
    exe = tmp_path / "caller"
    libdir = os.path.dirname(dsa.LIB_PATH)
    libname = os.path.basename(dsa.LIB_PATH)
    assert libname.startswith("lib") and libname.endswith(".so")
    cc = subprocess.run(["gcc", "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror", "-I",
                         os.path.join(ROOT, "include"), str(src), "-L", libdir, "-l" + libname[3:-3],
                         "-Wl,-rpath," + libdir, "-o", str(exe)], capture_output=True, text=True)
    assert cc.returncode == 0, cc.stderr
    run = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert run.returncode == 0 and run.stdout.strip() == "ok", (run.returncode, run.stdout, run.stderr)


def test_product_package_does_not_touch_the_oracle():
    pkg = os.path.join(ROOT, "dsa_indexed_sparse_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, f)).read()
                assert "oracle" not in text.lower(), f

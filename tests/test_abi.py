"""Host-side checks of the C ABI (no GPU needed): the library loads, it
exports every function include/bq.h declares, host-only queries give the
expected sizes, and the product package never imports the oracle."""
import ctypes
import os
import re
import shutil
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "bq.h")
PKG = os.path.join(ROOT, "block_quantized_moe_gather_gb300")


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"\b(bq_[a-z0-9_]+)\s*\(", text)
    return sorted(set(names))


@pytest.fixture(scope="module")
def bq():
    if not os.path.exists(os.path.join(PKG, "libbq.so")):
        import __graft_entry__
        __graft_entry__.build()
    import block_quantized_moe_gather_gb300 as m
    return m


def test_header_declares_the_boundary():
    names = _declared_functions()
    for must in ("bq_gguf_dequant_q8_0", "bq_gguf_dequant_q2_k", "bq_qmm", "bq_moe_gather_qmm",
                 "bq_moe_route", "bq_moe_permute", "bq_repack_q8_0", "bq_repack_q2_k", "bq_repack_int4",
                 "bq_dequant_mxfp4", "bq_repack_mxfp4"):
        assert must in names


def test_library_exports_every_declared_symbol(bq):
    lib = ctypes.CDLL(bq.LIB_PATH)
    missing = [n for n in _declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_status_strings(bq):
    for code, name in bq.STATUS_NAMES.items():
        assert bq.status_string(code).startswith(name)


def test_qweight_bytes_match_format_density(bq):
    # bytes per weight equal the on-disk formats: 34/32, 84/256, 9/16, 17/32
    assert bq.qweight_bytes(bq.FMT_Q8_0, 1, 256, 2048) == 256 * 2048 * 34 // 32
    assert bq.qweight_bytes(bq.FMT_Q2_K, 1, 4096, 4096) == 4096 * 4096 * 84 // 256
    assert bq.qweight_bytes(bq.FMT_INT4_G64, 128, 1536, 2048) == 128 * 1536 * 2048 * 9 // 16
    assert bq.qweight_bytes(bq.FMT_MXFP4, 128, 1536, 2048) == 128 * 1536 * 2048 * 17 // 32
    assert bq.qweight_bytes(bq.FMT_MXFP4, 1, 128, 64) == 0       # k not a multiple of 128
    assert bq.qweight_bytes(bq.FMT_Q2_K, 1, 100, 4096) == 0      # n not a multiple of 128
    assert bq.qweight_bytes(bq.FMT_Q2_K, 1, 128, 200) == 0       # k not a multiple of 256
    assert bq.qweight_bytes(9, 1, 128, 256) == 0                 # unknown format


def test_permute_workspace_query(bq):
    assert bq.moe_permute_workspace_bytes(2048, 8, 128) >= 64 * 128 * 4
    assert bq.moe_permute_workspace_bytes(1, 9, 16) == 0          # k > 8
    assert bq.moe_permute_workspace_bytes(1, 2, 2000) == 0        # E > 1024


def test_struct_layout_matches_header(bq):
    assert ctypes.sizeof(bq.QWeightC) == 32
    assert bq.MoEDescC.w_gate_up.offset == 24
    assert ctypes.sizeof(bq.MoEDescC) == 24 + 32 + 32 + 16 + 8
    assert bq.MoEDescC.route_scale.offset == 104


def test_host_validation_rejects_before_launch(bq):
    # shape checks run before the device is touched, so they work without a GPU
    lib = bq._lib
    assert lib.bq_moe_route(None, None, 4, 2000, 2, None, None, None) == 2        # E > 1024
    assert lib.bq_moe_route(None, None, 4, 16, 9, None, None, None) == 2          # k > 8
    assert lib.bq_moe_route_scored(None, None, 4, 16, 2, 3, 1.0, None, None, None) == 2   # unknown rule
    assert lib.bq_gguf_dequant_q8_0(None, -1, None, None) == 2
    assert lib.bq_gguf_dequant_q8_0(None, 5, None, None) == 1
    assert lib.bq_gguf_dequant_q2_k(ctypes.c_void_p(8), 5, ctypes.c_void_p(16), None) == 3   # misaligned
    assert "aligned" in bq.last_error()


def test_product_never_imports_the_oracle():
    for dirpath, _, files in os.walk(PKG):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, f)).read()
                assert not re.search(r"^\s*(import|from)\s+oracle\b", text, re.M), f
                assert "bq_oracle" not in text, f


def test_import_fails_loudly_without_the_library(tmp_path):
    dst = tmp_path / "block_quantized_moe_gather_gb300"
    shutil.copytree(PKG, dst, ignore=shutil.ignore_patterns("*.so", "_build", "__pycache__"))
    r = subprocess.run([sys.executable, "-c", "import block_quantized_moe_gather_gb300"], cwd=tmp_path,
                       capture_output=True, text=True)
    assert r.returncode != 0 and "ImportError" in r.stderr


def test_host_validation_of_the_block_format_and_norm_entry_points(bq):
    # MXFP4 / FP8 dequant, FP8 repack shapes and the RMSNorm calls, all rejected on the host
    lib = bq._lib
    assert lib.bq_dequant_mxfp4(None, -1, None, None) == 2
    assert lib.bq_dequant_mxfp4(None, 3, None, None) == 1
    assert lib.bq_dequant_mxfp4(None, 0, None, None) == 0                       # empty is a no-op
    assert lib.bq_dequant_fp8_b128(None, None, -1, 4, None, None) == 2
    assert lib.bq_dequant_fp8_b128(None, None, 4, 0, None, None) == 0
    assert lib.bq_dequant_fp8_b128(None, None, 4, 4, None, None) == 1
    assert lib.bq_dequant_fp8_b128(ctypes.c_void_p(16), ctypes.c_void_p(2), 4, 4, ctypes.c_void_p(16), None) == 3
    # FP8 weights need k a multiple of 128, and fused gate/up halves on the 128-row scale grid
    assert bq.qweight_bytes(bq.FMT_FP8_B128, 1, 128, 64) == 0
    assert bq.qweight_bytes(bq.FMT_FP8_B128, 2, 256, 256) == 2 * 2 * 4 * 8208
    w = bq.QWeightC(bq.FMT_FP8_B128, 1, 384, 128, 1, 0, 4096)
    assert lib.bq_repack_fp8_b128(ctypes.c_void_p(16), ctypes.c_void_p(16), ctypes.byref(w), None) == 2
    w = bq.QWeightC(bq.FMT_MXFP4, 1, 128, 128, 0, 0, 4096)
    assert lib.bq_repack_mxfp4(None, ctypes.byref(w), None) == 1
    assert lib.bq_rmsnorm(None, 2, 12, None, 1e-6, None, None) == 2              # H not a multiple of 8
    assert lib.bq_rmsnorm(None, 2, 16, None, -1.0, None, None) == 2              # eps < 0
    assert lib.bq_rmsnorm(None, 0, 16, None, 1e-6, None, None) == 0              # T == 0 is a no-op
    assert lib.bq_rmsnorm(None, 2, 16, None, 1e-6, None, None) == 1
    q = bq.QWeightC(bq.FMT_Q8_0, 1, 128, 64, 1, 0, 4096)                         # fused gate/up: rejected
    assert lib.bq_rmsnorm_qmm(None, 1, None, 1e-6, ctypes.byref(q), None, None, None) == 4


def test_hidden_layer_workspace_query(bq):
    gu = bq.QWeightC(bq.FMT_INT4_G64, 128, 256, 256, 1, 0, 4096)
    dn = bq.QWeightC(bq.FMT_INT4_G64, 128, 256, 128, 0, 0, 4096)
    d = bq.MoEDescC(4, 256, 128, 128, 4, 0, gu, dn, None, None, 1.0, 0)
    base = bq._lib.bq_moe_workspace_bytes(ctypes.byref(d))
    hidden = bq._lib.bq_moe_hidden_workspace_bytes(ctypes.byref(d))
    assert base > 0 and hidden >= base + 4 * 256 * 2 + 4 * 128 * 4
    # a descriptor whose weights have no valid format has no workspace size
    bad = bq.MoEDescC(4, 256, 128, 128, 4, 0, bq.QWeightC(), bq.QWeightC(), None, None, 1.0, 0)
    assert bq._lib.bq_moe_workspace_bytes(ctypes.byref(bad)) == 0
    assert bq._lib.bq_moe_hidden_workspace_bytes(ctypes.byref(bad)) == 0


def test_host_validation_of_the_layer_and_matmul_entry_points(bq):
    lib = bq._lib
    assert lib.bq_qmm(None, 1, None, None, None) == 1                                   # w NULL
    q = bq.QWeightC(bq.FMT_Q8_0, 1, 128, 64, 0, 0, 4096)
    assert lib.bq_qmm(None, -1, ctypes.byref(q), None, None) == 2                       # m < 0
    bad = bq.QWeightC(7, 1, 128, 64, 0, 0, 4096)
    assert lib.bq_qmm(None, 1, ctypes.byref(bad), None, None) == 4                      # unknown format
    assert lib.bq_moe_gather_qmm(None, None, None, None, None, None, 0, None) == 1       # desc NULL
    gu = bq.QWeightC(bq.FMT_INT4_G64, 8, 256, 256, 1, 0, 4096)
    dn = bq.QWeightC(bq.FMT_INT4_G64, 8, 256, 128, 0, 0, 4096)
    d = bq.MoEDescC(4, 256, 128, 8, 4, 9, gu, dn, None, None, 1.0, 0)                   # scoring 9
    assert lib.bq_moe_gather_qmm(ctypes.byref(d), None, None, None, None, None, 0, None) == 2
    d = bq.MoEDescC(4, 256, 128, 8, 9, 0, gu, dn, None, None, 1.0, 0)                   # top-k 9 > 8
    assert lib.bq_moe_gather_qmm(ctypes.byref(d), None, None, None, None, None, 0, None) == 2
    d = bq.MoEDescC(4, 256, 128, 8, 4, 0, gu, dn, None, None, 1.0, 0)
    assert lib.bq_moe_gather_qmm(ctypes.byref(d), None, None, None, None, None, 0, None) == 1   # NULL x
    x = ctypes.c_void_p(4096)
    assert lib.bq_moe_gather_qmm(ctypes.byref(d), x, x, None, x, None, 0, None) == 5    # no workspace
    assert lib.bq_set_stage_events(6, None, None) == 2                                  # unknown stage
    assert lib.bq_set_stage_events(5, None, None) == 0                                  # norm + router stage


def test_host_validation_of_pair_counts_and_the_wait_probe(bq):
    lib = bq._lib
    # T * k must fit an int: 2^29 + 1 tokens x top-8 is rejected before anything runs
    big = (1 << 29) + 1
    assert lib.bq_moe_route(None, None, big, 16, 8, None, None, None) == 2
    assert lib.bq_moe_permute_workspace_bytes(big, 8, 16) == 0
    assert lib.bq_moe_permute_noalloc(None, big, 8, 16, None, None, None, None, None, None) == 2
    assert "pairs" in bq.last_error()
    # the wait probe takes 0/1 and a limit in [1 ms, 2 s] (0 = default)
    assert lib.bq_test_set_wait_probe(2, 0) == 2
    assert lib.bq_test_set_wait_probe(0, 1000) == 2
    assert lib.bq_test_set_wait_probe(0, 3_000_000_000) == 2
    assert lib.bq_test_set_wait_probe(0, 0) == 0

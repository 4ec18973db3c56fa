"""CPU-side checks of the C-ABI library: it builds for sm_103a, loads without a GPU, exports
exactly the functions include/mosaic.h declares, and the binding agrees with the header's
status codes. No compute call is made here (that needs a GB300)."""
import ctypes
import os
import re
import subprocess

import pytest

from masked_token_lm_gb300 import build as mbuild
from masked_token_lm_gb300 import mosaic

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "mosaic.h")


@pytest.fixture(scope="module")
def lib_path():
    if not os.path.exists(mbuild.LIB):
        mbuild.build()
    return mbuild.LIB


def declared_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"MOSAIC_API\s+[\w\s\*]+?\b(mosaic_\w+)\s*\(", text)))


def test_header_declares_the_api():
    assert declared_functions() == sorted([
        "mosaic_check", "mosaic_create", "mosaic_destroy", "mosaic_last_error_string",
        "mosaic_launch_count", "mosaic_masked_logits", "mosaic_masked_logits_fp8",
        "mosaic_masked_logits_noalloc", "mosaic_quantize_masked_rows_e4m3",
        "mosaic_quantize_rows_e4m3",
        "mosaic_masked_sample", "mosaic_masked_sample_workspace_bytes", "mosaic_min_chunk_rows",
        "mosaic_set_wait_timeout", "mosaic_workspace_bind", "mosaic_workspace_bound_bytes",
        "mosaic_workspace_create", "mosaic_workspace_destroy", "mosaic_workspace_reserved_bytes",
        "mosaic_workspace_trim"])


def test_library_loads_and_exports_every_declared_symbol(lib_path):
    lib = ctypes.CDLL(lib_path)
    for name in declared_functions():
        assert hasattr(lib, name), name
    out = subprocess.run(["nm", "-D", "--defined-only", lib_path], capture_output=True, text=True).stdout
    exported = sorted(set(re.findall(r" T (mosaic_\w+)", out)))
    assert exported == declared_functions()


def test_status_codes_match_header():
    text = open(HEADER).read()
    for name, val in re.findall(r"(MOSAIC_(?:OK|ERR_\w+))\s*=\s*(\d+)", text):
        assert getattr(mosaic, name) == int(val), name
    for name, val in re.findall(r"(MOSAIC_(?:BF16|F32))\s*=\s*(\d+)", text):
        assert getattr(mosaic, name) == int(val), name


def test_null_handle_is_rejected_without_a_gpu(lib_path):
    mosaic.load_library()
    st = mosaic.mosaic_masked_logits(None, None, 1, 8, None, 0, None, None, 0, None, 8, None,
                                     0, 0, None, None, None)
    assert st == mosaic.MOSAIC_ERR_INVALID_ARG
    assert "handle" in mosaic.mosaic_last_error_string()
    assert mosaic.mosaic_check(None, None) == mosaic.MOSAIC_ERR_INVALID_ARG
    assert mosaic.mosaic_launch_count(None) == -1
    assert mosaic.mosaic_destroy(None) == mosaic.MOSAIC_OK


def test_create_without_gpu_fails_cleanly(lib_path):
    import torch

    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    st, h = mosaic.mosaic_create(0)
    assert st in (mosaic.MOSAIC_ERR_CUDA, mosaic.MOSAIC_ERR_UNSUPPORTED)
    assert not h.value


def test_product_package_does_not_import_the_oracle():
    pkg = os.path.join(ROOT, "masked_token_lm_gb300")
    for dp, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                src = open(os.path.join(dp, f), encoding="utf-8").read()
                assert not re.search(r"^\s*(from\s+oracle|import\s+oracle)", src, re.M), f
                assert not re.search(r'#include\s+"[^"]*oracle', src), f


def _brute_min_chunks(M, V, elt, budget):
    if M * V * elt <= budget:
        return 0, (1 if M > 0 else 0)
    for n in range(1, M + 1):
        rows = -(-M // n)
        if rows * V * elt <= budget:
            return rows, -(-M // rows)
    return None


def test_min_chunk_rows_matches_brute_force(lib_path):
    import itertools
    mosaic.load_library()
    for M, V, dt, budget in itertools.product([0, 1, 7, 100, 1000, 4097], [1, 8, 1024],
                                              [mosaic.MOSAIC_BF16, mosaic.MOSAIC_F32],
                                              [0, 15, 16, 17, 1000, 4096, 10 ** 5, 10 ** 7]):
        elt = 4 if dt == mosaic.MOSAIC_F32 else 2
        st, cr, nc = mosaic.mosaic_min_chunk_rows(M, V, dt, budget)
        want = _brute_min_chunks(M, V, elt, budget)
        if want is None:
            assert st == mosaic.MOSAIC_ERR_UNSUPPORTED, (M, V, dt, budget)
            continue
        assert st == mosaic.MOSAIC_OK, (M, V, dt, budget, mosaic.mosaic_last_error_string())
        assert (cr, nc) == want, (M, V, dt, budget, cr, nc, want)
        if cr:
            assert cr * V * elt <= budget and nc == -(-M // cr)


def test_min_chunk_rows_long_context_budget(lib_path):
    # 117,965 rows x 126,464 bf16 = 29.8 GB; a 1.036 GB budget (4096 rows) needs 29 chunks
    st, cr, nc = mosaic.mosaic_min_chunk_rows(117965, 126464, mosaic.MOSAIC_BF16, 4096 * 126464 * 2)
    assert st == mosaic.MOSAIC_OK and nc == 29 and cr <= 4096 and cr * 29 >= 117965
    st, cr, nc = mosaic.mosaic_min_chunk_rows(2048, 126464, mosaic.MOSAIC_BF16, 10 ** 12)
    assert (st, cr, nc) == (mosaic.MOSAIC_OK, 0, 1)  # lazy: off when it fits
    assert mosaic.mosaic_min_chunk_rows(-1, 8, 0, 10)[0] == mosaic.MOSAIC_ERR_INVALID_ARG


def test_sample_workspace_bytes(lib_path):
    mosaic.load_library()
    # 3 arrays (max, sum, arg) x rows x N tiles of 256 columns (rounded up to 4) x 4 bytes
    assert mosaic.mosaic_masked_sample_workspace_bytes(3686, 126464, 0) == 3 * 3686 * 496 * 4
    assert mosaic.mosaic_masked_sample_workspace_bytes(10000, 1000, 4096) == 3 * 4096 * 4 * 4
    assert mosaic.mosaic_masked_sample_workspace_bytes(-1, 10, 0) == -1


def test_workspace_without_gpu_fails_cleanly(lib_path):
    import torch

    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    st, ws = mosaic.mosaic_workspace_create(0, 1 << 30)
    assert st == mosaic.MOSAIC_ERR_CUDA and not ws.value
    assert mosaic.mosaic_workspace_bound_bytes(None) == -1
    assert mosaic.mosaic_workspace_destroy(None) == mosaic.MOSAIC_OK

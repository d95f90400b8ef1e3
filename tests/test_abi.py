"""CPU checks of the C ABI: the library builds for sm_103a, loads without a GPU, exports
every function include/gemm.h declares, and rejects bad arguments before touching CUDA."""
import os
import re
import subprocess

import pytest
import torch

import tensor_core_gemm_tcgen05_gb300 as g
from tensor_core_gemm_tcgen05_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gemm.h")


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return g.lib()


def header_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(gemm_\w+)\s*\(", text)))


def header_constants():
    text = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    return {k: int(v) for k, v in re.findall(r"\b(GEMM_[A-Z_0-9]+)\s*=\s*(-?\d+)", text)}


def test_exports_match_header(lib):
    funcs = header_functions()
    assert len(funcs) == 16
    assert sorted(g.EXPORTS) == funcs
    out = subprocess.run(["nm", "-D", "--defined-only", g.LIB_PATH], capture_output=True, text=True,
                         check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if line.strip()}
    for f in funcs:
        assert f in exported, f
        assert hasattr(lib, f)


def test_constants_match_header():
    consts = header_constants()
    for name, value in consts.items():
        assert getattr(g, name) == value, name
    assert consts["GEMM_EPI_GELU"] == g.EPI_GELU and consts["GEMM_EPI_RELU"] == g.EPI_RELU


def test_library_is_sm103a_only(lib):
    assert "compute_103a,code=sm_103a" in " ".join(_build.NVCC_FLAGS)
    # statically linked runtime: loads on a machine without libcudart.so in the path
    out = subprocess.run(["ldd", g.LIB_PATH], capture_output=True, text=True).stdout
    assert "libcudart" not in out


def test_status_strings(lib):
    for code in (0, -1, -2, -3, -4, -5, -6):
        assert g.gemm_status_string(code).startswith("GEMM_")
    assert "unknown" in g.gemm_status_string(42)


def test_null_context_is_rejected(lib):
    assert lib.gemm_run(None, 8, 8, 8, 16, 16, None, 16, 0, None) == g.GEMM_ERR_ARG
    assert lib.gemm_run_host(None, 8, 8, 8, 16, 16, None, 16, 0, None) == g.GEMM_ERR_ARG
    assert lib.gemm_last_device_error(None, None) == g.GEMM_ERR_ARG
    assert lib.gemm_set_debug(None, 0) == g.GEMM_ERR_ARG
    assert lib.gemm_set_timeout_ns(None, 5) == g.GEMM_ERR_ARG
    assert lib.gemm_destroy(None) == g.GEMM_OK
    assert lib.gemm_num_sms(None) == 0
    assert lib.gemm_num_pairs(None) == 0
    assert lib.gemm_row_softmax(None, 4, 8, 16, 16, None) == g.GEMM_ERR_ARG
    assert lib.gemm_attention_fwd(None, 1, 128, 128, 128, 16, 16, 16, 16, 0.1, 0, None) == g.GEMM_ERR_ARG
    assert lib.gemm_create(None, 0) == g.GEMM_ERR_ARG
    import ctypes
    buf = ctypes.create_string_buffer(64)
    assert lib.gemm_describe(None, 8, 8, 8, 0, buf, 64) == g.GEMM_ERR_ARG
    assert lib.gemm_describe(None, 8, 8, 8, 0, None, 64) == g.GEMM_ERR_ARG
    assert lib.gemm_clock_trace(None, 16, 8, 100000, 1000000, None) == g.GEMM_ERR_ARG
    # the allocation-free variant rejects bad sizes before touching CUDA
    assert lib.gemm_run_noalloc(-1, 8, 8, 16, 16, None, 16, 0, None) == g.GEMM_ERR_ARG
    assert lib.gemm_run_noalloc(8, 8, 2 ** 31, 16, 16, None, 16, 0, None) == g.GEMM_ERR_ARG
    assert lib.gemm_run_noalloc(8, 8, 8, 16, 16, None, 16, 5, None) == g.GEMM_ERR_ARG


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-GPU path")
def test_create_without_gpu_fails_cleanly(lib):
    with pytest.raises(g.GemmError) as e:
        g.gemm_create(0)
    assert e.value.status == g.GEMM_ERR_DEVICE


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    monkeypatch.setattr(g, "_lib", None)
    monkeypatch.setattr(g, "LIB_PATH", str(tmp_path / "absent.so"))
    with pytest.raises(RuntimeError, match="no CPU fallback"):
        g.lib()

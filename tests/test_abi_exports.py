"""The C-ABI library builds for sm_103a, loads without a GPU, and exports every
entry point include/nvfp4.h declares (no compute call is made here)."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "nvfp4.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"\b(nvfp4_[a-z0-9_]+)\s*\(", text)
    return sorted(set(names))


@pytest.fixture(scope="module")
def libpath():
    from nvfp4_precision_rl_gb300 import _build
    return _build.build()


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ["nvfp4_quantize_per_token", "nvfp4_gemm", "nvfp4_grouped_gemm",
                     "nvfp4_moe_permute", "nvfp4_swiglu_quantize", "nvfp4_get_device_status"]:
        assert required in names


def test_library_exports_every_declared_symbol(libpath):
    lib = ctypes.CDLL(libpath)
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_library_exports_nothing_else(libpath):
    out = subprocess.run(["nm", "-D", "--defined-only", libpath], capture_output=True, text=True,
                         check=True).stdout
    exported = {ln.split()[-1] for ln in out.splitlines() if " T " in ln}
    ours = {n for n in exported if n.startswith("nvfp4_")}
    assert ours == set(declared_functions())


def test_size_helpers_without_gpu(libpath):
    lib = ctypes.CDLL(libpath)
    lib.nvfp4_sf_bytes.restype = ctypes.c_size_t
    lib.nvfp4_sf_bytes.argtypes = [ctypes.c_int64, ctypes.c_int64]
    lib.nvfp4_packed_bytes.restype = ctypes.c_size_t
    lib.nvfp4_packed_bytes.argtypes = [ctypes.c_int64, ctypes.c_int64]
    lib.nvfp4_moe_capacity.restype = ctypes.c_int64
    lib.nvfp4_moe_capacity.argtypes = [ctypes.c_int64, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32]
    assert lib.nvfp4_sf_bytes(300, 160) == 384 * 12
    lib.nvfp4_mxfp8_sf_bytes.restype = ctypes.c_size_t
    lib.nvfp4_mxfp8_sf_bytes.argtypes = [ctypes.c_int64, ctypes.c_int64]
    assert lib.nvfp4_mxfp8_sf_bytes(300, 160) == 384 * 8
    assert lib.nvfp4_mxfp8_sf_bytes(130, 2080) == 256 * 68
    assert lib.nvfp4_packed_bytes(300, 160) == 300 * 80
    cap = lib.nvfp4_moe_capacity(4096, 8, 128, 128)
    assert cap % 128 == 0 and cap >= 4096 * 8 + 128 * 127


def test_binding_names_match_the_header():
    from nvfp4_precision_rl_gb300 import ops
    for n in declared_functions():
        assert hasattr(ops, n), n


def test_sm103a_only_and_no_fast_math():
    from nvfp4_precision_rl_gb300 import _build
    assert _build.ARCH == ["-gencode", "arch=compute_103a,code=sm_103a"]
    assert not any("fast" in f for f in _build.FLAGS)

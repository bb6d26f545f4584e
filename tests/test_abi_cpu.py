"""CPU checks of the C ABI: the library builds, loads without a GPU, exports
every function include/fa_gb300.h declares, and rejects bad arguments on the
host before touching CUDA.  No kernel is launched here."""
import ctypes
import os
import re
import shutil

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fa_gb300.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fa_[a-z0-9_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    import exact_io_aware_15_gb300 as fa
    from exact_io_aware_15_gb300 import build as b
    if not os.path.exists(fa.LIB_PATH):
        if not (shutil.which("nvcc") or os.path.exists("/usr/local/cuda/bin/nvcc")):
            pytest.skip("library not built and nvcc unavailable")
        b.build()
    return fa.load_library()


def test_header_declares_the_boundary():
    fns = declared_functions()
    for name in ["fa_fwd", "fa_fwd_f32", "fa_fwd_ex", "fa_fwd_varlen",
                 "fa_decode_workspace_bytes", "fa_decode_splitkv", "fa_combine_states",
                 "fa_check_device_status", "fa_status_string", "fa_last_cuda_error"]:
        assert name in fns


def test_every_declared_symbol_is_exported(lib):
    import exact_io_aware_15_gb300 as fa
    for name in declared_functions():
        assert hasattr(lib, name), name
        assert name in fa.SIGNATURES, f"binding lacks {name}"


def test_status_strings(lib):
    import exact_io_aware_15_gb300 as fa
    assert fa.fa_status_string(0) == "ok"
    for code in range(-8, 0):
        assert fa.fa_status_string(code) != "unknown status code"


def test_workspace_bytes(lib):
    assert lib.fa_decode_workspace_bytes(64, 32, 128, 16) == 64 * 32 * 16 * 4 * (2 + 128)
    assert lib.fa_decode_workspace_bytes(1, 1, 96, 16) == 0
    assert lib.fa_decode_workspace_bytes(1, 1, 64, 0) == 0


def test_host_validation_without_gpu(lib):
    """Bad arguments are refused on the host, before any CUDA call."""
    null = None
    buf = ctypes.create_string_buffer(4096 + 16)
    p = (ctypes.addressof(buf) + 15) // 16 * 16
    assert lib.fa_fwd(null, p, p, p, p, 1, 1, 16, 64, 0.125, 0, null) == -1
    assert lib.fa_fwd(p, p, p, p, p, 1, 1, 16, 96, 0.125, 0, null) == -1      # D
    assert lib.fa_fwd(p, p, p, p, p, 1, 1, 16, 64, -0.5, 0, null) == -1      # scale
    assert lib.fa_fwd(p, p, p, p, p, 1, 1, 16, 64, float("nan"), 0, null) == -1
    assert lib.fa_fwd(p + 2, p, p, p, p, 1, 1, 16, 64, 0.1, 0, null) == -1   # alignment
    assert lib.fa_fwd(p, p, p, p, p, -1, 1, 16, 64, 0.1, 0, null) == -1      # B < 0
    assert lib.fa_fwd_ex(p, p, p, p, p, 1, 1, 16, 64, 0.1, 0, 5, 0, null) == -1  # dtype
    assert lib.fa_fwd_varlen(p, p, p, p, p, null, 1, 16, 16, 1, 64, 0.1, 1, null) == -1
    assert lib.fa_decode_splitkv(p, p, p, p, 16, 1, 1, 128, 0, 0.1, p, p, p, null) == -1
    assert lib.fa_decode_splitkv(p, p, p, p, 16, 1, 1, 128, 300, 0.1, p, p, p, null) == -1
    assert lib.fa_combine_states(p, p, p, 1, 16, 128, p, 7, p, null) == -1
    # paged decode: page size not a power of two, H not a multiple of H_kv
    assert lib.fa_decode_paged_splitkv(p, p, p, p, p, 4, 24, 4, 1, 8, 2, 128, 4, 0.1,
                                       p, p, p, null) == -1
    assert lib.fa_decode_paged_splitkv(p, p, p, p, p, 4, 16, 4, 1, 8, 3, 128, 4, 0.1,
                                       p, p, p, null) == -1
    assert lib.fa_fwd_window(p, p, p, p, p, 1, 1, 16, 64, 0.1, 0, null) == -1
    # the failure-path test hook: a tile index >= 0 and a limit in [1 us, 2 s]
    assert lib.fa_fwd_fault_inject(p, p, p, p, p, 1, 1, 16, 64, 0.1, 0, -1, 1000, null) == -1
    assert lib.fa_fwd_fault_inject(p, p, p, p, p, 1, 1, 16, 64, 0.1, 0, 1, 0, null) == -1
    assert lib.fa_fwd_fault_inject(p, p, p, p, p, 1, 1, 16, 64, 0.1, 0, 1, 2000001, null) == -1


def test_binding_exports_exist():
    """Every name the binding exports is defined (no GPU needed)."""
    import exact_io_aware_15_gb300 as fa
    for name in fa.__all__:
        assert hasattr(fa, name), name

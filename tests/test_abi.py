"""The C ABI library loads and exports every symbol include/nc_api.h declares,
and rejects bad arguments on the host before touching a GPU."""

import ctypes
import os
import re

import pytest

from pretraining_step_03_b300 import _lib as L

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "nc_api.h")


def _declared():
    txt = open(HEADER).read()
    return sorted(set(re.findall(r"^NC_API[^(]*?\b(nc_\w+)\(", txt, flags=re.M)))


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(L.LIB_PATH):
        from pretraining_step_03_b300 import build
        build.build()
    return L.lib()


def test_every_declared_symbol_is_exported(lib):
    names = _declared()
    assert len(names) >= 20
    for n in names:
        assert hasattr(lib, n), n
    # and the binding declares a signature for each of them
    assert set(names) == set(L.SIGNATURES), set(names) ^ set(L.SIGNATURES)


def test_arena_size_and_argument_checks(lib):
    b = L.nc_arena_bytes(20, 1280, 10, 65536, 32, 2048, L.NC_BF16)
    # parameters, optimizer state and the activation stash of a d20 step fit a B300
    assert 40e9 < b < 200e9
    small = L.nc_arena_bytes(2, 128, 2, 512, 4, 64, L.NC_FP32)
    assert 0 < small < b
    for bad in [(0, 128, 2, 512), (2, 100, 2, 512), (2, 128, 3, 512), (2, 128, 2, 500), (2, 512, 2, 512)]:
        with pytest.raises(L.NcError) as e:
            L.nc_arena_bytes(*bad, 4, 64, L.NC_BF16)
        assert e.value.code == L.NC_ERR_ARG
    with pytest.raises(L.NcError) as e:
        L.nc_arena_bytes(2, 128, 2, 512, 4, 64, 7)
    assert e.value.code == L.NC_ERR_ARG


def test_null_handles_are_rejected(lib):
    out = ctypes.c_void_p()
    rc = lib.nc_init_model(2, 128, 2, 512, 0, None, 0, L.NC_BF16, 4, 64, None, ctypes.byref(out))
    assert rc == L.NC_ERR_ARG
    assert lib.nc_forward_backward(None, None, None, None, 1, 1, 0, 1.0, None) == L.NC_ERR_ARG
    assert lib.nc_muon_step(None, 0.02, 0.95, 1, 5, None) == L.NC_ERR_ARG
    assert lib.nc_adamw_step(None, 0.1, 0.1, 0.9, 0.95, 1e-8, 0.0, 1) == L.NC_ERR_ARG
    assert lib.nc_gemm_bf16(0, 1, 1, 1, None, 1, 0, 0, None, 1, 0, 0, None, 1, 0, 0, 1.0, 0.0, None, 0,
                            None) == L.NC_ERR_ARG
    assert "null" in L.nc_last_error()


def test_arena_shortfall_is_reported_before_any_launch(lib):
    """The library never allocates: an arena smaller than nc_arena_bytes is its allocation
    failure, reported as NC_ERR_OOM on the host (the pointer is only checked for alignment,
    never dereferenced, so no GPU is needed)."""
    out = ctypes.c_void_p()
    need = L.nc_arena_bytes(2, 128, 2, 512, 4, 64, L.NC_BF16)
    rc = lib.nc_init_model(2, 128, 2, 512, 0, ctypes.c_void_p(1 << 20), need - 256, L.NC_BF16, 4, 64, None,
                           ctypes.byref(out))
    assert rc == L.NC_ERR_OOM
    assert "arena" in L.nc_last_error()
    rc = lib.nc_init_model(2, 128, 2, 512, 0, ctypes.c_void_p((1 << 20) + 8), need, L.NC_BF16, 4, 64, None,
                           ctypes.byref(out))
    assert rc == L.NC_ERR_ARG   # not 256-byte aligned

"""The C-ABI library builds, loads and exports every symbol include/spectra.h
declares; host-side helpers and argument validation behave as documented.
CPU only: no call here launches GPU work."""
import ctypes as C
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def spx():
    from kv_cache_transform_encode_b300 import build
    build.build()
    import kv_cache_transform_encode_b300 as spx
    spx.lib()
    return spx


def header_functions():
    src = open(os.path.join(ROOT, "include", "spectra.h")).read()
    return sorted(set(re.findall(r"SPECTRA_API\s+[\w\s\*]+?\b(spectra_\w+)\s*\(", src)))


def test_header_declares_the_boundary():
    names = header_functions()
    for want in ("spectra_calibrate", "spectra_alloc_bits", "spectra_encode", "spectra_decode",
                 "spectra_attn_decode"):
        assert want in names


def test_every_declared_symbol_is_exported(spx):
    lib = C.CDLL(spx.library_path())
    for name in header_functions():
        assert hasattr(lib, name), name
    assert set(header_functions()) == set(spx.EXPORTS)


def test_version_and_status_strings(spx):
    assert spx.spectra_version() >= 100
    for st, name in spx.STATUS_NAMES.items():
        assert spx.spectra_status_string(st) == name


def test_stream_bytes_matches_layout(spx, orc):
    for R in (0, 1, 3, 170, 256, 512, 1024):
        for T in (0, 1, 31, 32, 33, 128, 1000, 32768):
            assert spx.spectra_stream_bytes(R, T) == (orc.stream_bytes(T, R) if R and T else 0)


def test_workspace_sizes(spx):
    assert spx.spectra_plan_derived_bytes(8, 128) % 256 == 0
    assert spx.spectra_plan_derived_bytes(8, 96) == 0
    assert spx.spectra_calibrate_workspace_bytes(8, 128, 2048) >= 8 * 128 * 128 * 4
    assert spx.spectra_attn_workspace_bytes(16, 32, 128, 65536) > 16 * 32 * 128 * 4
    assert spx.spectra_attn_workspace_bytes(0, 32, 128, 10) == 0


def _plan_struct(spx, **kw):
    p = spx.spectra_plan(8, 128, 0, 0, 256, 0, 16, 16, 16, 16, 16, 256, 16)
    for k, v in kw.items():
        setattr(p, k, v)
    return p


def test_invalid_arguments_rejected_before_launch(spx):
    """Bad sizes, enums, pointers and strides return an error status from the
    host-side checks (nothing reaches the GPU)."""
    lib = spx.lib()
    null = None
    bad = [
        lib.spectra_encode(None, C.c_void_p(16), 0, 10, 1024, C.c_void_p(16), 4096, null, 0, null),
        lib.spectra_encode(C.byref(_plan_struct(spx, head_dim=96)), C.c_void_p(16), 0, 10, 1024,
                           C.c_void_p(16), 4096, null, 0, null),
        lib.spectra_encode(C.byref(_plan_struct(spx, basis=7)), C.c_void_p(16), 0, 10, 1024,
                           C.c_void_p(16), 4096, null, 0, null),
        lib.spectra_encode(C.byref(_plan_struct(spx)), C.c_void_p(16), 0, 10, 100,   # stride < H*d
                           C.c_void_p(16), 4096, null, 0, null),
        lib.spectra_encode(C.byref(_plan_struct(spx)), C.c_void_p(18), 0, 10, 1024,  # misaligned x
                           C.c_void_p(16), 4096, null, 0, null),
        lib.spectra_encode(C.byref(_plan_struct(spx)), C.c_void_p(16), 0, 10, 1024,
                           C.c_void_p(16), 16, null, 0, null),                         # stream too small
        lib.spectra_encode(C.byref(_plan_struct(spx)), C.c_void_p(16), 5, 10, 1024,   # bad dtype
                           C.c_void_p(16), 4096, null, 0, null),
        lib.spectra_encode(C.byref(_plan_struct(spx, derived=264)), C.c_void_p(16), 0, 10, 1024,
                           C.c_void_p(16), 4096, null, 0, null),                       # derived unaligned
        lib.spectra_alloc_bits(C.byref(_plan_struct(spx)), -1.0, 0, null),
        lib.spectra_alloc_bits(C.byref(_plan_struct(spx)), 2.0, 9, null),
        lib.spectra_alloc_bits(C.byref(_plan_struct(spx)), float("nan"), 0, null),
        lib.spectra_calibrate(C.byref(_plan_struct(spx)), C.c_void_p(16), 0, 2048, 1024, 0,
                              C.c_void_p(256), 1 << 30, null, null),                   # max_sweeps 0
        lib.spectra_calibrate(C.byref(_plan_struct(spx)), C.c_void_p(16), 0, 2048, 1024, 30,
                              C.c_void_p(256), 16, null, null),                        # workspace small
        lib.spectra_attn_decode(C.byref(_plan_struct(spx)), C.byref(_plan_struct(spx)), C.c_void_p(16),
                                0, 2, 12, C.c_void_p(16), C.c_void_p(16), 1 << 20, null, null, 0,
                                100, 1.0, C.c_void_p(16), C.c_void_p(256), 1 << 30, null),  # Hq % Hkv
        lib.spectra_decode(C.byref(_plan_struct(spx, quant=1, basis=1, signs=16)), C.c_void_p(16),
                           4096, null, 0, 10, C.c_void_p(16), 0, 1024, null),           # RWHT w/o norms
    ]
    assert all(b != 0 for b in bad), bad
    assert lib.spectra_encode(C.byref(_plan_struct(spx, head_dim=96)), C.c_void_p(16), 0, 10, 1024,
                              C.c_void_p(16), 4096, null, 0, null) == 2   # UNSUPPORTED


def test_no_cpu_fallback_in_binding():
    """The binding has no compute path of its own: it never imports the
    oracle and every public function goes through the CUDA library."""
    src = open(os.path.join(ROOT, "kv_cache_transform_encode_b300", "__init__.py")).read()
    assert "oracle" not in src.replace("no CPU fallback", "")
    assert "numpy" not in src


def test_kernel_family_setting(spx):
    """The process-wide kernel family: settable, read back, unknown values
    refused (host logic only, no launch)."""
    prev = spx.spectra_get_kernel_family()
    try:
        for f in (spx.SPECTRA_KERNELS_CUDA_CORE, spx.SPECTRA_KERNELS_TENSOR_CORE, spx.SPECTRA_KERNELS_AUTO):
            spx.spectra_set_kernel_family(f)
            assert spx.spectra_get_kernel_family() == f
        assert spx.lib().spectra_set_kernel_family(3) == 1
        assert spx.lib().spectra_set_kernel_family(-1) == 1
        assert spx.spectra_get_kernel_family() == spx.SPECTRA_KERNELS_AUTO
    finally:
        spx.spectra_set_kernel_family(prev)

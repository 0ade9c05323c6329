"""CPU checks of the C ABI: the library builds for sm_103a, loads, and exports
every function declared in include/*.h; the binding's signature table covers
the same set.  No compute call is made (there may be no GPU)."""
from __future__ import annotations

import ctypes
import glob
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b(vt_\w+)\s*\(", text, re.M):
            names.add(m.group(1))
    return names


@pytest.fixture(scope="module")
def lib_path():
    from device_token_sampling_gb300 import _build
    return _build.build()


def test_header_declares_the_entry_points():
    names = declared_functions()
    for want in ("vt_sampler_create", "vt_sampler_destroy", "vt_reset_params",
                 "vt_reset_token_counts", "vt_sample", "vt_get_row_status",
                 "vt_debug_filter_boundary", "vt_debug_get_counts", "vt_last_error"):
        assert want in names, want


def test_library_exports_every_declared_symbol(lib_path):
    out = subprocess.run(["nm", "-D", "--defined-only", lib_path], capture_output=True,
                         text=True, check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if " T " in line}
    missing = declared_functions() - exported
    assert not missing, missing


def test_library_loads_and_binding_matches_header(lib_path):
    lib = ctypes.CDLL(lib_path)
    for name in declared_functions():
        assert hasattr(lib, name), name
    from device_token_sampling_gb300 import sampler
    assert set(sampler.SIGNATURES) == declared_functions()
    sampler.load_library()


def test_status_strings_without_gpu(lib_path):
    from device_token_sampling_gb300 import sampler
    lib = sampler.load_library()
    assert lib.vt_status_string(0) == b"VT_OK"
    assert lib.vt_status_string(-5) == b"VT_ERR_TIMEOUT"
    assert lib.vt_last_error(None) == b"null handle"


def test_create_rejects_bad_config_without_gpu(lib_path):
    from device_token_sampling_gb300 import sampler
    lib = sampler.load_library()
    h = ctypes.c_void_p()
    bad = sampler.Config(0, 1000, 0, 0, 0, 0)
    assert lib.vt_sampler_create(ctypes.byref(bad), ctypes.byref(h)) == sampler.VT_ERR_INVALID_ARG
    bad = sampler.Config(4, 1000, 33, 0, 0, 0)
    assert lib.vt_sampler_create(ctypes.byref(bad), ctypes.byref(h)) == sampler.VT_ERR_INVALID_ARG
    assert lib.vt_sampler_create(None, ctypes.byref(h)) == sampler.VT_ERR_INVALID_ARG


def test_product_package_does_not_import_the_oracle():
    pkg = os.path.join(ROOT, "device_token_sampling_gb300")
    for path in glob.glob(os.path.join(pkg, "**", "*.*"), recursive=True):
        if path.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
            text = open(path, errors="ignore").read()
            assert "import oracle" not in text and "from oracle" not in text, path
            assert "oracle.h" not in text, path


def test_probs_plan_without_gpu(lib_path):
    """The filtered distribution's grid: every split holds 1 to 64 K elements (a
    multiple of 64 wide), the splits cover the row exactly, and B x splits stays
    within the partials a handle allocates at create: max_batch x (ceil(max_vocab
    / 64 K) + 1) + 6 per SM."""
    from device_token_sampling_gb300 import sampler
    lib = sampler.load_library()
    sp, rg = ctypes.c_int32(), ctypes.c_int32()

    def plan(B, V, sms):
        assert lib.vt_debug_probs_plan(B, V, sms, ctypes.byref(sp), ctypes.byref(rg)) == 0
        return sp.value, rg.value

    def cap(max_b, max_v, sms):
        return max_b * ((max_v + 65535) // 65536 + 1) + 6 * sms

    sizes_b = [1, 2, 7, 64, 255, 256, 1000, 4096, 1 << 20]
    sizes_v = [1, 63, 64, 65, 1000, 65536, 65537, 151_936, 248_320, 1 << 20]
    for sms in (1, 152):
        for B in sizes_b:
            for V in sizes_v:
                s, r = plan(B, V, sms)
                assert r % 64 == 0 and 64 <= r <= 65536, (B, V, r)
                assert (s - 1) * r < V <= s * r, (B, V, s, r)
                assert B * s <= cap(B, V, sms), (B, V, s)
        for mb in sizes_b:
            for mv in sizes_v:
                for B in [b for b in sizes_b if b <= mb][-3:]:
                    for V in [v for v in sizes_v if v <= mv][-3:]:
                        assert B * plan(B, V, sms)[0] <= cap(mb, mv, sms), (mb, mv, B, V)
    assert lib.vt_debug_probs_plan(0, 10, 152, ctypes.byref(sp), ctypes.byref(rg)) == \
        sampler.VT_ERR_INVALID_ARG

"""The C-ABI library builds for sm_103a, loads, and exports every entry point include/vfy.h
declares (no compute calls: this runs without a GPU)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_symbols():
    text = open(os.path.join(ROOT, "include", "vfy.h")).read()
    return sorted(set(re.findall(r"VFY_API[^;{]*?\b(vfy_[a-z_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    __graft_entry__.build()
    from speculative_decode_verify_attn_gb300 import vfy
    return vfy.lib()


def test_header_declares_the_boundary():
    names = declared_symbols()
    for required in ("vfy_create", "vfy_attend_full", "vfy_attend_swa", "vfy_select_resident", "vfy_accept",
                     "vfy_page_in", "vfy_destroy", "vfy_get_status", "vfy_strerror"):
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_symbols():
        assert hasattr(lib, name), name
    from speculative_decode_verify_attn_gb300 import vfy
    assert set(vfy.EXPORTS) == set(declared_symbols())


def test_only_the_abi_is_exported(lib):
    import subprocess
    from speculative_decode_verify_attn_gb300 import vfy
    out = subprocess.run(["nm", "-D", "--defined-only", vfy.lib_path()], capture_output=True, text=True).stdout
    text_syms = {l.split()[-1] for l in out.splitlines() if " T " in l}
    assert {s for s in text_syms if s.startswith("vfy_")} == set(declared_symbols())


def test_launch_count_of_no_context_is_zero(lib):
    assert lib.vfy_launch_count(None) == 0


def test_strerror_needs_no_device(lib):
    from speculative_decode_verify_attn_gb300 import vfy
    assert vfy.strerror(vfy.VFY_OK) == "ok"
    assert "invalid" in vfy.strerror(vfy.VFY_EINVAL)


def test_create_validates_on_the_host(lib):
    """A bad configuration is rejected before any device is touched."""
    from speculative_decode_verify_attn_gb300 import vfy
    cfg = vfy.Config(16, 4, 96, 64, 512, 2048, 1, 17, 64, 0.0)        # head_dim 96 unsupported
    h = ctypes.c_void_p()
    assert lib.vfy_create(ctypes.byref(cfg), 0, ctypes.byref(h)) == vfy.VFY_EINVAL
    cfg = vfy.Config(16, 4, 128, 64, 512, 8192, 1, 1025, 64, 0.0)     # 1025 queries x 4 > 4096 rows
    assert lib.vfy_create(ctypes.byref(cfg), 0, ctypes.byref(h)) == vfy.VFY_EINVAL
    cfg = vfy.Config(16, 4, 128, 32, 512, 2048, 1, 17, 64, 0.0)       # chunk must be 64
    assert lib.vfy_create(ctypes.byref(cfg), 0, ctypes.byref(h)) == vfy.VFY_EINVAL
    cfg = vfy.Config(16, 4, 128, 64, 2000, 2048, 1, 17, 64, 0.0)      # ring too small for window
    assert lib.vfy_create(ctypes.byref(cfg), 0, ctypes.byref(h)) == vfy.VFY_EINVAL
    assert lib.vfy_attend_full(None, None, None, None, None, 0, None, None, None, 0, None, None, None, 1,
                               None) == vfy.VFY_EINVAL

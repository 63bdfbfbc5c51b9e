"""The C-ABI library builds for sm_103a, loads, and exports every function that
include/dflash.h declares (CPU only: no compute call is made)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    names = set()
    for h in os.listdir(os.path.join(ROOT, "include")):
        if h.endswith(".h"):
            src = open(os.path.join(ROOT, "include", h)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names |= set(re.findall(r"^\s*(?:const\s+)?[\w\s\*]+?\b(\w+)\s*\(", src, flags=re.M))
    return {n for n in names if n not in ("if", "return", "sizeof")}


def test_library_exports_every_declared_symbol():
    from block_diffusion_draft_dflash_gb300 import build
    lib_path = build.build()
    lib = ctypes.CDLL(lib_path)
    declared = _declared()
    assert {"dflash_draft_block", "ddtree_build", "tree_verify_attention", "accept_and_compact",
            "dflash_target_tree_forward"} <= declared
    missing = [n for n in declared if not hasattr(lib, n)]
    assert not missing, missing


def test_binding_covers_header():
    from block_diffusion_draft_dflash_gb300 import _lib
    assert _declared() == set(_lib.exported_symbols())


def test_status_strings_without_gpu():
    from block_diffusion_draft_dflash_gb300 import _lib
    assert _lib.status_string(0) == "ok"
    assert "NaN" in _lib.status_string(-6)


def test_host_argument_checks_without_gpu():
    # invalid arguments are rejected on the host before anything touches the device
    from block_diffusion_draft_dflash_gb300 import _lib
    lib = _lib.load()
    assert lib.ddtree_build(None, 1, 0, 10, 4, *([None] * 6), None, 0, None) == -1      # D < 1
    assert lib.ddtree_build(None, 1, 2, 3, 13, *([None] * 6), None, 0, None) == -1      # B > 3 + 9
    assert lib.tree_verify_attention(1, 5, 8, 2, 64, None, None, None, 64, None, None, 1.0, None,
                                     None, 0, None) == -2                               # hd != 128
    assert lib.dflash_linear(None, None, 4, 4, 100, None, 0, None, 0, None) == -2      # K % 64


def test_checked_build_is_separate_and_compiles():
    # DFLASH_CHECKED=1 selects the checked build: its own output directory, and the index
    # checks compile (one translation unit compiled here; the GPU tests run the whole library)
    import subprocess
    import sys
    import tempfile
    code = "import block_diffusion_draft_dflash_gb300.build as b; print(b.CHECKED, b.LIB)"
    out = subprocess.run([sys.executable, "-c", code], cwd=ROOT, capture_output=True, text=True,
                         env=dict(os.environ, DFLASH_CHECKED="1")).stdout.split()
    assert out[0] == "True" and out[1].endswith(os.path.join("_build_checked", "libdflash.so"))
    from block_diffusion_draft_dflash_gb300 import build
    assert not build.CHECKED and build.LIB.endswith(os.path.join("_build", "libdflash.so"))
    with tempfile.TemporaryDirectory() as d:
        r = subprocess.run([build._nvcc(), *build.ARCH, *build.FLAGS, "-DDFLASH_CHECKED=1", "-I", build.INCLUDE, "-c",
                            os.path.join(build.CSRC, "accept.cu"), "-o", os.path.join(d, "accept.o")],
                           capture_output=True, text=True)
        assert r.returncode == 0, r.stderr


def test_status_string_of_every_code():
    from block_diffusion_draft_dflash_gb300 import _lib
    for code in range(-11, 0):
        assert _lib.status_string(code) != "unknown status", code

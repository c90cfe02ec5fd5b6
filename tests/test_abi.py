"""The C-ABI library builds, loads and exports every entry point include/*.h declares
(no compute calls: this runs without a GPU)."""
import glob
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_symbols():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        src = open(h).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        for m in re.finditer(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\**\s+\**\s*(spec_[a-z0-9_]+)\s*\(",
                             src, flags=re.M):
            names.add(m.group(1))
    return names


@pytest.fixture(scope="module")
def lib_path():
    from speculative_decoding_verify_step_gb300 import build
    return build.build()


def test_header_declares_the_boundary():
    names = declared_symbols()
    for must in ["spec_model_create", "spec_decode_step", "spec_verify_step", "spec_verify_tree_step",
                 "spec_accept_probs", "spec_sync_status"]:
        assert must in names


def test_library_exports_every_declared_symbol(lib_path):
    out = subprocess.run(["nm", "-D", "--defined-only", lib_path], capture_output=True, text=True, check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if " T " in line}
    missing = declared_symbols() - exported
    assert not missing, f"declared but not exported: {sorted(missing)}"


def test_library_loads_and_binds(lib_path):
    from speculative_decoding_verify_step_gb300 import spec
    lib = spec.load_library(lib_path)
    for name in declared_symbols():
        assert hasattr(lib, name)
    assert set(spec.EXPORTS) == declared_symbols()
    assert lib.spec_last_error() == b""


def test_binding_refuses_missing_library(tmp_path):
    from speculative_decoding_verify_step_gb300 import spec
    saved = spec._lib
    spec._lib = None
    try:
        with pytest.raises(ImportError):
            spec.load_library(str(tmp_path / "nope.so"))
    finally:
        spec._lib = saved


def test_no_oracle_import_in_product():
    pkg = os.path.join(ROOT, "speculative_decoding_verify_step_gb300")
    for f in glob.glob(os.path.join(pkg, "**", "*.*"), recursive=True):
        if f.endswith((".py", ".cu", ".cuh", ".h")):
            txt = open(f).read()
            assert "import oracle" not in txt and "from oracle" not in txt, f

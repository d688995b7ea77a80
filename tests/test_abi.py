"""The C-ABI library loads, exports every declared symbol, and rejects bad
arguments on the host before touching the GPU (CPU only: no compute call).

The refusal checks themselves (tests/abi_host_checks.py) hand the entry points
invented device addresses and expect every call to fail on the host.  They run
in a child process that sees no GPU, so that a host check that ever stopped
refusing could not launch a kernel on an unmapped address of a real GPU.
"""

import ctypes
import os
import re
import subprocess
import sys

import pytest

from conftest import ROOT

HEADER_DIR = os.path.join(ROOT, "include")


def _declared_functions():
    names = []
    for f in sorted(os.listdir(HEADER_DIR)):
        if not f.endswith(".h"):
            continue
        text = open(os.path.join(HEADER_DIR, f)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        text = re.sub(r"//[^\n]*", "", text)
        text = re.sub(r"#[^\n]*", "", text)
        for m in re.finditer(r"\b([A-Za-z_]\w*)\s*\(((?:[^()]|\([^()]*\))*)\)\s*;", text):
            if m.group(1) not in ("sizeof",):
                names.append(m.group(1))
    return names


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    __graft_entry__.build()
    from tree_speculative_decoding_spec_gb300 import _binding
    return _binding


def test_header_declares_the_four_entry_points():
    names = _declared_functions()
    for n in ["spec_tree_build", "hydra_draft", "tree_attention", "tree_accept"]:
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    raw = ctypes.CDLL(lib.LIB_PATH)
    for name in _declared_functions():
        assert hasattr(raw, name), f"{name} declared in include/ but not exported"


def test_library_has_no_fallback_dependency_on_torch(lib):
    # the shared object must not link against torch or python
    with open(lib.LIB_PATH, "rb") as f:
        blob = f.read()
    assert b"libtorch" not in blob and b"libpython" not in blob


def test_host_checks_refuse_before_any_device_access():
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "abi_host_checks.py")],
                       env=env, cwd=ROOT, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, (r.stdout[-4000:] + r.stderr[-2000:])
    assert " passed" in r.stdout and "failed" not in r.stdout


def test_binding_refuses_to_run_without_library(tmp_path, monkeypatch):
    # the product path fails loudly when the compiled library is absent
    import importlib
    import tree_speculative_decoding_spec_gb300._binding as b
    monkeypatch.setattr(os.path, "exists", lambda p: False if p == b.LIB_PATH else os.path.isfile(p) or os.path.isdir(p))
    with pytest.raises(ImportError):
        b._load()

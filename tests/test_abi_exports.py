"""The C-ABI library builds for sm_103a, loads, and exports every symbol that
include/mla.h declares (no compute calls: CPU only)."""
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "mla.h")


def _declared():
    with open(HEADER) as f:
        src = f.read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"\b(mla_[a-z_0-9]+)\s*\(", src)
    return sorted(set(names))


@pytest.fixture(scope="module")
def lib_path():
    from mla_absorbed_latent_02_gb300 import _build
    return _build.build()


def test_header_declares_the_decode_path():
    names = _declared()
    for n in ["mla_append_latent", "mla_absorb_q", "mla_decode_attn", "mla_expand_v",
              "mla_create", "mla_destroy", "mla_decode_workspace_size"]:
        assert n in names


def test_library_exports_every_declared_symbol(lib_path):
    out = subprocess.run(["nm", "-D", "--defined-only", lib_path], capture_output=True, text=True, check=True).stdout
    exported = set(re.findall(r"\s[TW]\s+(\S+)$", out, flags=re.M))
    missing = [n for n in _declared() if n not in exported]
    assert not missing, missing


def test_binding_covers_every_declared_symbol(lib_path):
    import mla_absorbed_latent_02_gb300 as m
    lib = m.load_library(lib_path)
    for n in _declared():
        assert n in m.SIGNATURES, n
        assert getattr(lib, n) is not None


def test_create_fails_cleanly_without_gpu(lib_path):
    import torch
    if torch.cuda.is_available():
        pytest.skip("GPU present")
    import ctypes
    import mla_absorbed_latent_02_gb300 as m
    lib = m.load_library(lib_path)
    h = ctypes.c_void_p()
    rc = lib.mla_create(ctypes.byref(h), 0, 1024, 10000.0)
    assert rc != 0 and not h.value

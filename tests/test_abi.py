"""The C-ABI library builds, loads and exports every declared entry point (CPU)."""

import ctypes
import os
import re

import pytest

import radixattention_prefix_shared_radix_gb300 as sgl
from radixattention_prefix_shared_radix_gb300 import build as sglbuild

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "sglattn.h")


@pytest.fixture(scope="module")
def lib():
    sglbuild.build()
    return ctypes.CDLL(sglbuild.LIB)


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(sgl_[a-z0-9_]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert len(names) >= 25
    for n in names:
        assert hasattr(lib, n), n


def test_binding_covers_every_declared_symbol():
    assert set(declared_functions()) <= set(sgl.exported_symbols())


def test_status_strings_and_version(lib):
    sglbuild.build()
    assert sgl.sgl_status_string(0) == "SGL_OK"
    assert sgl.sgl_status_string(-2) == "SGL_ERR_NO_SLOTS"
    assert "sm_103a" in sgl.sgl_version()


def test_host_errors_do_not_need_a_gpu():
    sglbuild.build()
    with pytest.raises(sgl.SglError) as e:
        sgl.sgl_tree_create(10, 3)
    assert e.value.status == -1
    p = sgl.make_params(sgl.SGL_DTYPE_BF16, 1, 6, 4, 128, 1024)     # G not an integer
    with pytest.raises(sgl.SglError) as e:
        sgl.sgl_extend_workspace_bytes(p)
    assert e.value.status == -3
    p = sgl.make_params(sgl.SGL_DTYPE_BF16, 1, 8, 8, 96, 1024)      # head_dim 96
    with pytest.raises(sgl.SglError) as e:
        sgl.sgl_extend_workspace_bytes(p)
    assert e.value.status == -3

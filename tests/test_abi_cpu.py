"""The C-ABI library: it builds for sm_103a, loads without a GPU, exports every entry
point that include/lwm_attn.h declares, and rejects bad arguments on the host."""

import ctypes
import os
import re

import pytest

import blockwise_ringattention_causal_b300 as lwm
from blockwise_ringattention_causal_b300 import build as lwm_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    lwm_build.build()
    return lwm.load_library()


def declared_functions():
    text = open(os.path.join(ROOT, "include", "lwm_attn.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(lwm_\w+)\s*\(", text)))


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert "lwm_attn_fwd" in names and "lwm_attn_bwd" in names
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(lwm._SIGNATURES), "binding and header disagree"


def test_status_strings(lib):
    for code, name in lwm.STATUS_NAMES.items():
        assert lwm.lwm_status_string(code).startswith(name)


def test_workspace_size(lib):
    a = lwm.lwm_attn_workspace_size(1, 1024, 4, 128)
    b = lwm.lwm_attn_workspace_size(2, 65536, 32, 128)
    assert a > 0 and b > a and b % 256 == 0
    assert lwm.lwm_attn_workspace_size(1, 1024, 4, 64) == 0
    assert lwm.lwm_attn_workspace_size(0, 1024, 4, 128) == 0
    # padded fp32 row terms dominate: 2 x B x H x S_pad x 4 bytes
    assert b >= 2 * 2 * 32 * 65536 * 4


def _fwd(lib, q=8192, k=8192, v=8192, out=8192, lse=8192, B=1, S=128, H=1, D=128, ws=1 << 20, nbytes=1 << 30):
    P = ctypes.c_void_p
    return lib.lwm_attn_fwd(P(q), P(k), P(v), None, None, P(out), P(lse), B, S, H, D, P(ws), nbytes, None)


def test_host_argument_errors(lib):
    assert _fwd(lib, D=64) == 2                       # unsupported head dim
    assert _fwd(lib, B=0) == 1 and _fwd(lib, S=-1) == 1
    assert _fwd(lib, q=0) == 1                        # null pointer
    assert _fwd(lib, k=8200) == 3                     # not 16-byte aligned
    assert _fwd(lib, ws=(1 << 20) + 16) == 5          # workspace not 256-byte aligned
    assert _fwd(lib, nbytes=16) == 1                  # workspace too small
    P = ctypes.c_void_p
    assert lib.lwm_attn_prepare(None, None, 1, 128, 1, 128, 0, P(1 << 20), 1 << 30, None) == 1
    assert lib.lwm_attn_prepare(P(8194), None, 1, 128, 1, 128, 1, P(1 << 20), 1 << 30, None) == 3
    assert lib.lwm_attn_check(None, None) == 1


def test_product_path_never_touches_the_oracle():
    pkg = os.path.join(ROOT, "blockwise_ringattention_causal_b300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                src = open(os.path.join(dirpath, f)).read()
                assert not re.search(r"^\s*(import|from)\s+oracle", src, re.M), f
                assert "oracle/" not in src, f

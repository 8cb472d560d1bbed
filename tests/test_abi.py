"""C ABI checks that need no GPU: the library loads, exports every function the
header declares, sizes workspaces, and rejects invalid arguments before it
launches anything (explicit rejection of unsupported configurations: Megatron-LM
PR #6808 "Add state-passing context parallelism for Mamba2", "Not supported yet")."""
from __future__ import annotations

import ctypes
import os
import re

import pytest

import mamba2_ssd_selective_gb300 as ssd
from mamba2_ssd_selective_gb300.build import build
from mamba2_ssd_selective_gb300.inputs import SsdShape

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build()
    return ssd.load()


def declared_functions() -> list[str]:
    names = []
    for h in os.listdir(os.path.join(ROOT, "include")):
        if h.endswith(".h"):
            text = open(os.path.join(ROOT, "include", h)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names += re.findall(r"^[A-Za-z_][\w\s\*]*?\b(ssd_\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert {"ssd_forward", "ssd_backward", "ssd_workspace_size", "ssd_cu_seqlens_to_seq_idx",
            "ssd_status_string", "ssd_device_status"} <= set(names)
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings(lib):
    for code in range(0, -10, -1):
        s = ssd.ssd_status_string(code)
        assert s and s != "unknown status"


SHAPE = SsdShape(2, 1024, 8, 64, 128, 2, 256, 2)


def test_workspace_size_host_only(lib):
    d = ssd.make_dims(SHAPE, "bf16")
    f, b = ssd.ssd_workspace_size(d, False), ssd.ssd_workspace_size(d, True)
    assert 0 < f < b
    # the post-conv activations alone need b*L*Cd bf16
    assert f > SHAPE.tokens * SHAPE.conv_dim * 2


@pytest.mark.parametrize("field,value,status", [
    ("seqlen", 1000, -2),      # not a multiple of n_segments * chunk
    ("n_segments", 8, -2),     # 8 * 256 > 1024
    ("d_conv", 3, -1),
    ("ngroups", 3, -1),        # 8 heads not divisible by 3 groups
    ("headdim", 0, -1),
    ("dtype", 7, -5),
    ("chunk", 16, -7),         # not a multiple of 32
    ("dstate", 12, -7),        # not a multiple of 8
])
def test_invalid_dims_rejected(lib, field, value, status):
    d = ssd.make_dims(SHAPE, "bf16")
    setattr(d, field, value)
    assert ssd.ssd_workspace_size(d, False) == 0
    inp = ssd.SsdInputs()
    rc = lib.ssd_forward(ctypes.byref(d), ctypes.byref(inp), None, None, None, None, 0, None)
    assert rc == status


def _fake_inputs(eb=2, misalign=0):
    # host addresses that are never dereferenced: validation rejects before launch
    base = 1 << 20
    s = SHAPE
    HP, GN, Cd = s.nheads * s.headdim, s.ngroups * s.dstate, s.conv_dim
    return ssd.SsdInputs(base + misalign, Cd, base + HP * eb, Cd, base + (HP + GN) * eb, Cd, base, s.nheads,
                         base, base, base, base, base, None)


def test_null_and_alignment_and_workspace_rejected(lib):
    d = ssd.make_dims(SHAPE, "bf16")
    ws = ssd.ssd_workspace_size(d, False)
    inp = _fake_inputs()
    inp.D = None
    assert lib.ssd_forward(ctypes.byref(d), ctypes.byref(inp), 1 << 20, None, None, 1 << 24, ws, None) == -3
    inp = _fake_inputs(misalign=2)
    assert lib.ssd_forward(ctypes.byref(d), ctypes.byref(inp), 1 << 20, None, None, 1 << 24, ws, None) == -4
    inp = _fake_inputs()
    inp.seq_idx = (1 << 20) + 4  # seq_idx must be 16-byte aligned
    assert lib.ssd_forward(ctypes.byref(d), ctypes.byref(inp), 1 << 20, None, None, 1 << 24, ws, None) == -4
    inp = _fake_inputs()
    inp.B_tok_stride = SHAPE.conv_dim + 1  # not a multiple of 8 bf16 elements
    assert lib.ssd_forward(ctypes.byref(d), ctypes.byref(inp), 1 << 20, None, None, 1 << 24, ws, None) == -4
    inp = _fake_inputs()
    assert lib.ssd_forward(ctypes.byref(d), ctypes.byref(inp), None, None, None, 1 << 24, ws, None) == -3
    assert lib.ssd_forward(ctypes.byref(d), ctypes.byref(inp), 1 << 20, None, None, 1 << 24, ws - 1, None) == -6
    assert lib.ssd_forward(ctypes.byref(d), ctypes.byref(inp), 1 << 20, None, None, None, ws, None) == -6
    g = ssd.SsdGrads()
    wsb = ssd.ssd_workspace_size(d, True)
    assert lib.ssd_backward(ctypes.byref(d), ctypes.byref(inp), 1 << 20, None, None, ctypes.byref(g), 1 << 24,
                            wsb, None) == -3


def test_cu_seqlens_rejects_bad_args(lib):
    assert lib.ssd_cu_seqlens_to_seq_idx(None, 3, 1 << 20, 10, None) == -3
    assert lib.ssd_cu_seqlens_to_seq_idx(1 << 20, 0, 1 << 20, 10, None) == -1

"""fp64 CPU oracle for the Mamba2 SSD mixer core -- TEST INFRASTRUCTURE ONLY.

Only the test suite, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg (and its ``--impl reference`` arm) may import this package.  The product
path (``mamba2_ssd_selective_gb300``) never imports it and shares no code with it.

The arithmetic lives in ``ssd_oracle.c`` (plain C, fp64, pthreads over heads):
token-by-token conv + SiLU, the selective state-space recurrence, the segmented
variant (per-segment affine summary, exclusive scan, correction) and the adjoint
recurrence for the backward.  This module only marshals arrays into it, one batch
row at a time, and sums per-row parameter gradients over rows in row order.

Parity of every function here is pinned by tests/test_oracle_pins.py.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ssd_oracle.c")
_LIB = os.path.join(_HERE, "libssd_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the C oracle in-tree (plain gcc, no target-specific flags)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", "-o", tmp, _SRC, "-lm"],
                       check=True)
        os.replace(tmp, _LIB)
    return _LIB


class _Row(ctypes.Structure):
    _fields_ = [
        ("L", ctypes.c_int), ("H", ctypes.c_int), ("P", ctypes.c_int), ("N", ctypes.c_int), ("G", ctypes.c_int),
        ("xBC", ctypes.c_void_p), ("dt_raw", ctypes.c_void_p), ("dt_bias", ctypes.c_void_p),
        ("A_log", ctypes.c_void_p), ("D", ctypes.c_void_p), ("conv_w", ctypes.c_void_p),
        ("conv_b", ctypes.c_void_p), ("seq_idx", ctypes.c_void_p), ("init", ctypes.c_void_p),
    ]


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            P = ctypes.c_void_p
            I = ctypes.c_int
            lib.orc_forward.argtypes = [ctypes.POINTER(_Row), I, I, I, P, P, P, P, P, I]
            lib.orc_forward.restype = I
            lib.orc_backward.argtypes = [ctypes.POINTER(_Row), I, I, P, P, P, P, P, P, P, P, P, P, I]
            lib.orc_backward.restype = I
            lib.orc_conv.argtypes = [ctypes.POINTER(_Row), I, I, P, P, I]
            lib.orc_conv.restype = I
            lib.orc_subset_size.argtypes = [ctypes.POINTER(_Row), I, I]
            lib.orc_subset_size.restype = I
            lib.orc_subset_channel.argtypes = [ctypes.POINTER(_Row), I, I, I]
            lib.orc_subset_channel.restype = I
            lib.orc_default_threads.restype = I
            lib.orc_seq_finals.argtypes = [ctypes.POINTER(_Row), I, I, P, I]
            lib.orc_seq_finals.restype = I
            lib.orc_num_seqs.argtypes = [ctypes.POINTER(_Row)]
            lib.orc_num_seqs.restype = I
            D = ctypes.c_double
            lib.orc_gated_norm_fwd.argtypes = [I, I, I, P, P, P, D, P]
            lib.orc_gated_norm_fwd.restype = I
            lib.orc_gated_norm_bwd.argtypes = [I, I, I, P, P, P, D, P, P, P, P]
            lib.orc_gated_norm_bwd.restype = I
            _lib = lib
    return _lib


def default_threads() -> int:
    return int(_load().orc_default_threads())


def _f64(a) -> np.ndarray:
    if a is None:
        return None
    if hasattr(a, "detach"):
        a = a.detach().cpu().double().numpy()
    return np.ascontiguousarray(a, dtype=np.float64)


def _ptr(a) -> int | None:
    return None if a is None else a.ctypes.data


class _RowArgs:
    """Keeps the fp64 copies of one batch row alive while C reads them."""

    def __init__(self, inp: dict, dims: tuple, b: int):
        L, H, P, N, G = dims
        self.xBC = _f64(inp["xBC"][b])
        self.dt_raw = _f64(inp["dt_raw"][b])
        self.dt_bias = _f64(inp["dt_bias"])
        self.A_log = _f64(inp["A_log"])
        self.D = _f64(inp["D"])
        self.conv_w = _f64(inp["conv_w"])
        self.conv_b = _f64(inp["conv_b"])
        si = inp.get("seq_idx")
        self.seq_idx = None if si is None else np.ascontiguousarray(
            si[b].cpu().numpy() if hasattr(si, "cpu") else si[b], dtype=np.int32)
        h0 = inp.get("init")
        self.init = None if h0 is None else _f64(h0[b])
        self.row = _Row(L, H, P, N, G, _ptr(self.xBC), _ptr(self.dt_raw), _ptr(self.dt_bias), _ptr(self.A_log),
                        _ptr(self.D), _ptr(self.conv_w), _ptr(self.conv_b), _ptr(self.seq_idx), _ptr(self.init))


def _dims(shape) -> tuple:
    return (shape.seqlen, shape.nheads, shape.headdim, shape.dstate, shape.ngroups)


def conv(inp: dict, shape, b: int = 0, heads: tuple | None = None, nthreads: int = 0):
    """Post-conv u and pre-activation v for the channel subset of ``heads`` in row b.

    Returns (u, v, channels): u, v are (L, nsub) float64, channels the global
    channel index of each column (x of the heads, then B, C of their groups)."""
    lib = _load()
    h0, h1 = heads or (0, shape.nheads)
    ra = _RowArgs(inp, _dims(shape), b)
    nsub = lib.orc_subset_size(ctypes.byref(ra.row), h0, h1)
    u = np.empty((nsub, shape.seqlen))
    v = np.empty((nsub, shape.seqlen))
    lib.orc_conv(ctypes.byref(ra.row), h0, h1, _ptr(u), _ptr(v), nthreads)
    ch = np.array([lib.orc_subset_channel(ctypes.byref(ra.row), h0, h1, j) for j in range(nsub)])
    return u.T.copy(), v.T.copy(), ch


def gated_norm(y: np.ndarray, z: np.ndarray, w: np.ndarray, ngroups: int, eps: float) -> np.ndarray:
    """Gated RMSNorm of one or more rows: y, z (rows, L, C), w (C) -> out (rows, L, C)."""
    lib = _load()
    y, z, w = _f64(y), _f64(z), _f64(w)
    out = np.empty_like(y)
    for r in range(y.shape[0]):
        if lib.orc_gated_norm_fwd(y.shape[1], y.shape[2], ngroups, _ptr(y[r]), _ptr(z[r]), _ptr(w), eps,
                                  _ptr(out[r])) != 0:
            raise ValueError("oracle gated_norm rejected its arguments")
    return out


def gated_norm_backward(y, z, w, ngroups: int, eps: float, dout) -> tuple:
    """(dy, dz, dw) of the gated RMSNorm given dout; dw summed over rows in row order."""
    lib = _load()
    y, z, w, dout = _f64(y), _f64(z), _f64(w), _f64(dout)
    dy, dz = np.empty_like(y), np.empty_like(y)
    dw = np.zeros_like(w)
    for r in range(y.shape[0]):
        if lib.orc_gated_norm_bwd(y.shape[1], y.shape[2], ngroups, _ptr(y[r]), _ptr(z[r]), _ptr(w), eps,
                                  _ptr(dout[r]), _ptr(dy[r]), _ptr(dz[r]), _ptr(dw)) != 0:
            raise ValueError("oracle gated_norm_backward rejected its arguments")
    return dy, dz, dw


def _norm_slices(inp: dict, shape, h0: int, h1: int, rows: list):
    """z and the norm weight of heads [h0, h1) (whole groups) and the groups they cover."""
    hpg, P = shape.nheads // shape.ngroups, shape.headdim
    if h0 % hpg or h1 % hpg:
        raise ValueError("the gated norm needs whole groups of heads")
    z = _f64(inp["z"])[rows][..., h0 * P:h1 * P]
    w = _f64(inp["norm_weight"])[h0 * P:h1 * P]
    return z, w, (h1 - h0) // hpg


def forward(inp: dict, shape, n_segments: int | None = None, heads: tuple | None = None,
            rows: list | None = None, nthreads: int = 0) -> dict:
    """y (rows, L, nh, P), final_state (rows, nh, P, N) and, for S > 1, the
    segment summaries: seg_in / s_ext (rows, S, nh, P, N), a_block (rows, S, nh).
    inp["init"] (b, H, P, N), when present, is each row's initial state.  With
    inp["z"] present, y is the gated RMSNorm of the mixer output (norm_weight,
    norm_eps) and the output before the norm is returned as y_pre."""
    lib = _load()
    S = shape.n_segments if n_segments is None else n_segments
    h0, h1 = heads or (0, shape.nheads)
    nh = h1 - h0
    rows = list(range(shape.batch)) if rows is None else list(rows)
    L, P, N = shape.seqlen, shape.headdim, shape.dstate
    out = {k: [] for k in ("y", "final_state", "seg_in", "s_ext", "a_block")}
    for b in rows:
        ra = _RowArgs(inp, _dims(shape), b)
        y = np.empty((L, nh, P))
        fin = np.empty((nh, P, N))
        seg_in = np.empty((S, nh, P, N))
        s_ext = np.empty((S, nh, P, N))
        a_blk = np.empty((S, nh))
        rc = lib.orc_forward(ctypes.byref(ra.row), h0, h1, S, _ptr(y), _ptr(fin), _ptr(seg_in), _ptr(s_ext),
                             _ptr(a_blk), nthreads)
        if rc != 0:
            raise ValueError("oracle forward rejected its arguments")
        for k, v in zip(out, (y, fin, seg_in, s_ext, a_blk)):
            out[k].append(v)
    res = {k: np.stack(v) for k, v in out.items()}
    if inp.get("z") is not None:
        z, w, ng = _norm_slices(inp, shape, h0, h1, rows)
        res["y_pre"] = res["y"]
        nr = len(rows)
        res["y"] = gated_norm(res["y"].reshape(nr, L, nh * P), z, w, ng, float(inp["norm_eps"])).reshape(nr, L, nh, P)
    return res


def backward(inp: dict, shape, heads: tuple | None = None, rows: list | None = None,
             use_dfinal: bool = True, nthreads: int = 0) -> dict:
    """Gradients of L = <dy, y> + <dfinal, final_state> w.r.t. every input
    (with inp["init"] present, also w.r.t. each row's initial state: dinit;
    with inp["z"] present y is the gated norm's output, and dz (rows, L, nh*P)
    and dnorm_weight (nh*P) are returned too).

    For heads=(h0,h1) covering whole groups the results are exact for those heads'
    x channels / dt columns and their groups' B/C channels.  Returns float64:
      dxBC (rows, L, nsub) with ``channels`` (global channel of each column),
      ddt_raw (rows, L, nh), dconv_w (nsub, 4), dconv_b (nsub), ddt_bias, dA_log, dD (nh),
      dinit (rows, nh, P, N) or None
    with parameter gradients summed over the rows in row order."""
    lib = _load()
    h0, h1 = heads or (0, shape.nheads)
    nh = h1 - h0
    rows = list(range(shape.batch)) if rows is None else list(rows)
    L = shape.seqlen
    P = shape.headdim
    norm = None
    if inp.get("z") is not None:
        # the gated norm's backward turns dout into the mixer output's gradient
        # (every head of the row: the mixer's backward reads dy of all heads)
        y_pre = forward(inp, shape, n_segments=1, rows=rows, nthreads=nthreads)["y_pre"]
        nr = len(rows)
        z, w, ng = _norm_slices(inp, shape, 0, shape.nheads, rows)
        dout = _f64(inp["dy"])[rows]
        dyn, dzn, dwn = gated_norm_backward(y_pre.reshape(nr, L, -1), z, w, ng, float(inp["norm_eps"]), dout)
        norm = {"dy": dyn, "dz": dzn[..., h0 * P:h1 * P], "dnorm_weight": dwn[h0 * P:h1 * P]}
    dxs, ddts, dinits = [], [], []
    acc = None
    ch = None
    for b in rows:
        ra = _RowArgs(inp, _dims(shape), b)
        nsub = lib.orc_subset_size(ctypes.byref(ra.row), h0, h1)
        if ch is None:
            ch = np.array([lib.orc_subset_channel(ctypes.byref(ra.row), h0, h1, j) for j in range(nsub)])
        dy = _f64(inp["dy"][b]) if norm is None else np.ascontiguousarray(norm["dy"][rows.index(b)])
        dfin = _f64(inp["dfinal"][b]) if use_dfinal and inp.get("dfinal") is not None else None
        dxr = np.empty((L, nsub))
        dw = np.empty((nsub, 4))
        db = np.empty(nsub)
        ddt = np.empty((L, nh))
        dbias = np.empty(nh)
        dalog = np.empty(nh)
        dD = np.empty(nh)
        dinit = np.empty((nh, shape.headdim, shape.dstate)) if ra.init is not None else None
        rc = lib.orc_backward(ctypes.byref(ra.row), h0, h1, _ptr(dy), _ptr(dfin), _ptr(dxr), _ptr(dw), _ptr(db),
                              _ptr(ddt), _ptr(dbias), _ptr(dalog), _ptr(dD), _ptr(dinit), nthreads)
        if rc != 0:
            raise ValueError("oracle backward rejected its arguments")
        dxs.append(dxr)
        ddts.append(ddt)
        dinits.append(dinit)
        part = (dw, db, dbias, dalog, dD)
        acc = part if acc is None else tuple(a + p for a, p in zip(acc, part))
    return {
        "dxBC": np.stack(dxs), "channels": ch, "ddt_raw": np.stack(ddts),
        "dconv_w": acc[0], "dconv_b": acc[1], "ddt_bias": acc[2], "dA_log": acc[3], "dD": acc[4],
        "dinit": None if dinits[0] is None else np.stack(dinits),
        "dz": None if norm is None else norm["dz"],
        "dnorm_weight": None if norm is None else norm["dnorm_weight"],
    }


def seq_finals(inp: dict, shape, b: int = 0, heads: tuple | None = None, nthreads: int = 0) -> np.ndarray:
    """The state after the last token of every packed sequence of row b, in order:
    (nseq, nh, P, N) float64 (the plain token recurrence, from inp["init"][b] if given)."""
    lib = _load()
    h0, h1 = heads or (0, shape.nheads)
    ra = _RowArgs(inp, _dims(shape), b)
    nseq = lib.orc_num_seqs(ctypes.byref(ra.row))
    out = np.empty((nseq, h1 - h0, shape.headdim, shape.dstate))
    if lib.orc_seq_finals(ctypes.byref(ra.row), h0, h1, _ptr(out), nthreads) != nseq:
        raise ValueError("oracle seq_finals rejected its arguments")
    return out

"""Mamba2 SSD mixer core on GB300: Python binding of libssd's C ABI.

The functions below carry the C names (``ssd_forward``, ``ssd_backward``,
``ssd_workspace_size``, ``ssd_cu_seqlens_to_seq_idx``, ``ssd_device_status``,
``ssd_status_string``) and only marshal arguments: torch tensors become device
pointers, the current torch stream becomes the cudaStream_t.  Every step of the
computation runs in libssd's CUDA kernels; there is no Python or CPU fallback,
and loading fails loudly when the compiled library is missing.
"""
from __future__ import annotations

import ctypes
import os

import torch

__all__ = [
    "SsdError", "SsdDims", "SsdInputs", "SsdGrads", "load", "ssd_workspace_size", "ssd_forward", "ssd_backward",
    "ssd_forward_static", "STATIC_SCRATCH_BYTES", "ssd_forward_varlen",
    "ssd_cu_seqlens_to_seq_idx", "ssd_device_status", "ssd_set_wait_limit_ns", "DEFAULT_WAIT_LIMIT_NS",
    "ssd_status_string", "ssd_profile_begin",
    "ssd_profile_end", "SsdKernelTime", "SsdRunner",
    "SSD_BF16", "SSD_F32",
]

SSD_BF16, SSD_F32 = 0, 1
_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libssd.so")
_lib = None


class SsdError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {ssd_status_string(status)} (status {status})")
        self.status = status


class SsdDims(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "batch", "seqlen", "nheads", "headdim", "dstate", "ngroups", "d_conv", "chunk", "n_segments", "dtype",
        "gated_norm")]


class SsdInputs(ctypes.Structure):
    _fields_ = [
        ("x", ctypes.c_void_p), ("x_tok_stride", ctypes.c_int64),
        ("B", ctypes.c_void_p), ("B_tok_stride", ctypes.c_int64),
        ("C", ctypes.c_void_p), ("C_tok_stride", ctypes.c_int64),
        ("dt", ctypes.c_void_p), ("dt_tok_stride", ctypes.c_int64),
        ("dt_bias", ctypes.c_void_p), ("A_log", ctypes.c_void_p), ("D", ctypes.c_void_p),
        ("conv_w", ctypes.c_void_p), ("conv_b", ctypes.c_void_p), ("seq_idx", ctypes.c_void_p),
        ("initial_states", ctypes.c_void_p),
        ("z", ctypes.c_void_p), ("z_tok_stride", ctypes.c_int64), ("norm_weight", ctypes.c_void_p),
        ("norm_eps", ctypes.c_float),
    ]


class SsdGrads(ctypes.Structure):
    _fields_ = [
        ("dx", ctypes.c_void_p), ("dx_tok_stride", ctypes.c_int64),
        ("dB", ctypes.c_void_p), ("dB_tok_stride", ctypes.c_int64),
        ("dC", ctypes.c_void_p), ("dC_tok_stride", ctypes.c_int64),
        ("ddt", ctypes.c_void_p), ("ddt_tok_stride", ctypes.c_int64),
        ("ddt_bias", ctypes.c_void_p), ("dA_log", ctypes.c_void_p), ("dD", ctypes.c_void_p),
        ("dconv_w", ctypes.c_void_p), ("dconv_b", ctypes.c_void_p), ("dinitial_states", ctypes.c_void_p),
        ("dz", ctypes.c_void_p), ("dz_tok_stride", ctypes.c_int64), ("dnorm_weight", ctypes.c_void_p),
    ]


class SsdKernelTime(ctypes.Structure):
    _fields_ = [("name", ctypes.c_char_p), ("launches", ctypes.c_int32), ("total_ms", ctypes.c_float)]


def load():
    """Load libssd.so (built by ``python -m mamba2_ssd_selective_gb300.build``)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libssd.so is not built ({LIB_PATH}); run python -m mamba2_ssd_selective_gb300.build")
        lib = ctypes.CDLL(LIB_PATH)
        P, I, S = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
        lib.ssd_workspace_size.argtypes = [ctypes.POINTER(SsdDims), I]
        lib.ssd_workspace_size.restype = S
        lib.ssd_forward.argtypes = [ctypes.POINTER(SsdDims), ctypes.POINTER(SsdInputs), P, P, P, P, S, P]
        lib.ssd_forward.restype = I
        lib.ssd_forward_static.argtypes = [ctypes.POINTER(SsdDims), ctypes.POINTER(SsdInputs), P, P, P, P]
        lib.ssd_forward_static.restype = I
        lib.ssd_forward_varlen.argtypes = [ctypes.POINTER(SsdDims), ctypes.POINTER(SsdInputs), P, P, P, P,
                                           ctypes.c_int32, P, P, S, P]
        lib.ssd_forward_varlen.restype = I
        lib.ssd_backward.argtypes = [ctypes.POINTER(SsdDims), ctypes.POINTER(SsdInputs), P, P, P,
                                     ctypes.POINTER(SsdGrads), P, S, P]
        lib.ssd_backward.restype = I
        lib.ssd_cu_seqlens_to_seq_idx.argtypes = [P, ctypes.c_int32, P, ctypes.c_int32, P]
        lib.ssd_cu_seqlens_to_seq_idx.restype = I
        lib.ssd_device_status.argtypes = [P, P]
        lib.ssd_device_status.restype = I
        lib.ssd_set_wait_limit_ns.argtypes = [ctypes.c_uint64]
        lib.ssd_set_wait_limit_ns.restype = ctypes.c_uint64
        lib.ssd_profile_begin.argtypes = []
        lib.ssd_profile_begin.restype = I
        lib.ssd_profile_end.argtypes = [ctypes.POINTER(SsdKernelTime), ctypes.c_int32]
        lib.ssd_profile_end.restype = ctypes.c_int32
        lib.ssd_status_string.argtypes = [I]
        lib.ssd_status_string.restype = ctypes.c_char_p
        _lib = lib
    return _lib


def _ptr(t) -> int | None:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(status: int, what: str) -> None:
    if status != 0:
        raise SsdError(status, what)


def ssd_status_string(status: int) -> str:
    return load().ssd_status_string(int(status)).decode()


def ssd_workspace_size(dims: SsdDims, backward: bool) -> int:
    return int(load().ssd_workspace_size(ctypes.byref(dims), int(bool(backward))))


def ssd_forward(dims: SsdDims, inputs: SsdInputs, y, final_state, seg_init_states, workspace, ws_bytes=None,
                stream=None) -> None:
    ws_bytes = workspace.numel() * workspace.element_size() if ws_bytes is None else ws_bytes
    _check(load().ssd_forward(ctypes.byref(dims), ctypes.byref(inputs), _ptr(y), _ptr(final_state),
                              _ptr(seg_init_states), _ptr(workspace), ws_bytes, _stream(stream)), "ssd_forward")


def ssd_forward_varlen(dims: SsdDims, inputs: SsdInputs, y, final_state, seg_init_states, cu_seqlens,
                       seq_final_states, workspace, ws_bytes=None, stream=None) -> None:
    """ssd_forward of one packed row that also writes the state after every
    sequence's last token into seq_final_states (nseq, H, P, N)."""
    ws_bytes = workspace.numel() * workspace.element_size() if ws_bytes is None else ws_bytes
    _check(load().ssd_forward_varlen(ctypes.byref(dims), ctypes.byref(inputs), _ptr(y), _ptr(final_state),
                                     _ptr(seg_init_states), _ptr(cu_seqlens), cu_seqlens.numel() - 1,
                                     _ptr(seq_final_states), _ptr(workspace), ws_bytes, _stream(stream)),
           "ssd_forward_varlen")


def ssd_forward_static(dims: SsdDims, inputs: SsdInputs, y, final_state, seg_init_states, stream=None) -> None:
    """ssd_forward without a workspace: the library's fixed device scratch array is
    used instead (for callers that cannot allocate; see include/ssd.h)."""
    _check(load().ssd_forward_static(ctypes.byref(dims), ctypes.byref(inputs), _ptr(y), _ptr(final_state),
                                     _ptr(seg_init_states), _stream(stream)), "ssd_forward_static")


STATIC_SCRATCH_BYTES = 32 << 20


def ssd_backward(dims: SsdDims, inputs: SsdInputs, dy, dfinal_state, seg_init_states, grads: SsdGrads, workspace,
                 ws_bytes=None, stream=None) -> None:
    ws_bytes = workspace.numel() * workspace.element_size() if ws_bytes is None else ws_bytes
    _check(load().ssd_backward(ctypes.byref(dims), ctypes.byref(inputs), _ptr(dy), _ptr(dfinal_state),
                               _ptr(seg_init_states), ctypes.byref(grads), _ptr(workspace), ws_bytes,
                               _stream(stream)), "ssd_backward")


def ssd_cu_seqlens_to_seq_idx(cu_seqlens, seq_idx, stream=None) -> None:
    _check(load().ssd_cu_seqlens_to_seq_idx(_ptr(cu_seqlens), cu_seqlens.numel() - 1, _ptr(seq_idx),
                                            seq_idx.numel(), _stream(stream)), "ssd_cu_seqlens_to_seq_idx")


def ssd_device_status(workspace, stream=None) -> int:
    """Status word of the last call that used ``workspace`` (None: the static
    scratch of ssd_forward_static); 0 = ok, -9 = a device-side wait gave up."""
    return int(load().ssd_device_status(_ptr(workspace), _stream(stream)))


DEFAULT_WAIT_LIMIT_NS = 1_500_000_000


def ssd_set_wait_limit_ns(limit_ns: int) -> int:
    """Limit of the kernels' bounded device-side waits for later calls; returns the previous one."""
    return int(load().ssd_set_wait_limit_ns(int(limit_ns)))


def ssd_profile_begin() -> None:
    _check(load().ssd_profile_begin(), "ssd_profile_begin")


def ssd_profile_end(max_entries: int = 64) -> list[tuple[str, int, float]]:
    """[(kernel name, launches, total ms)] recorded since ssd_profile_begin()."""
    buf = (SsdKernelTime * max_entries)()
    n = load().ssd_profile_end(buf, max_entries)
    if n < 0:
        raise SsdError(n, "ssd_profile_end")
    return [(buf[i].name.decode(), int(buf[i].launches), float(buf[i].total_ms)) for i in range(n)]


# ---------------------------------------------------------------- marshalling helpers

def make_dims(shape, dtype: str, gated_norm: bool = False) -> SsdDims:
    return SsdDims(shape.batch, shape.seqlen, shape.nheads, shape.headdim, shape.dstate, shape.ngroups,
                   shape.d_conv, shape.chunk, shape.n_segments, SSD_BF16 if dtype == "bf16" else SSD_F32,
                   int(bool(gated_norm)))


class SsdRunner:
    """Holds device buffers for one shape and calls the C ABI on them.

    ``t`` is a dict of device tensors as produced by ``inputs.make_inputs`` (moved
    to the GPU): xBC (b, L, Cd) with x, B, C as token-strided views, dt_raw,
    parameters and optional seq_idx, init, z / norm_weight (gated_norm=True)."""

    def __init__(self, shape, dtype: str, device="cuda", gated_norm: bool = False):
        self.shape, self.dtype, self.device = shape, dtype, torch.device(device)
        self.gated_norm = gated_norm
        self.dims = make_dims(shape, dtype, gated_norm)
        self.tdtype = torch.bfloat16 if dtype == "bf16" else torch.float32
        self.ws_fwd = ssd_workspace_size(self.dims, False)
        self.ws_bwd = ssd_workspace_size(self.dims, True)
        if self.ws_fwd == 0:
            raise ValueError("invalid dims for libssd")
        self.workspace = torch.empty(max(self.ws_fwd, self.ws_bwd), dtype=torch.uint8, device=self.device)

    def inputs(self, t: dict) -> SsdInputs:
        s = self.shape
        HP, GN, Cd = s.nheads * s.headdim, s.ngroups * s.dstate, s.conv_dim
        xBC = t["xBC"]
        es = xBC.element_size()
        base = xBC.data_ptr()
        return SsdInputs(base, Cd, base + HP * es, Cd, base + (HP + GN) * es, Cd, t["dt_raw"].data_ptr(), s.nheads,
                         _ptr(t["dt_bias"]), _ptr(t["A_log"]), _ptr(t["D"]), _ptr(t["conv_w"]), _ptr(t["conv_b"]),
                         _ptr(t.get("seq_idx")), _ptr(t.get("init")),
                         _ptr(t.get("z")) if self.gated_norm else None, s.nheads * s.headdim,
                         _ptr(t.get("norm_weight")) if self.gated_norm else None,
                         float(t.get("norm_eps", 1e-5)))

    def alloc_outputs(self):
        s = self.shape
        y = torch.empty(s.batch, s.seqlen, s.nheads * s.headdim, dtype=self.tdtype, device=self.device)
        fin = torch.empty(s.batch, s.nheads, s.headdim, s.dstate, dtype=torch.float32, device=self.device)
        seg = torch.empty(s.batch, s.n_segments, s.nheads, s.headdim, s.dstate, dtype=torch.float32,
                          device=self.device)
        return y, fin, seg

    def alloc_grads(self, init: bool = False):
        s = self.shape
        g = {
            "dxBC": torch.empty(s.batch, s.seqlen, s.conv_dim, dtype=self.tdtype, device=self.device),
            "ddt_raw": torch.empty(s.batch, s.seqlen, s.nheads, dtype=self.tdtype, device=self.device),
            "ddt_bias": torch.empty(s.nheads, dtype=torch.float32, device=self.device),
            "dA_log": torch.empty(s.nheads, dtype=torch.float32, device=self.device),
            "dD": torch.empty(s.nheads, dtype=torch.float32, device=self.device),
            "dconv_w": torch.empty(s.conv_dim, 4, dtype=torch.float32, device=self.device),
            "dconv_b": torch.empty(s.conv_dim, dtype=torch.float32, device=self.device),
        }
        if init:
            g["dinit"] = torch.empty(s.batch, s.nheads, s.headdim, s.dstate, dtype=torch.float32, device=self.device)
        if self.gated_norm:
            g["dz"] = torch.empty(s.batch, s.seqlen, s.nheads * s.headdim, dtype=self.tdtype, device=self.device)
            g["dnorm_weight"] = torch.empty(s.nheads * s.headdim, dtype=torch.float32, device=self.device)
        return g

    def grads_struct(self, g: dict) -> SsdGrads:
        s = self.shape
        HP, GN, Cd = s.nheads * s.headdim, s.ngroups * s.dstate, s.conv_dim
        d = g["dxBC"]
        es = d.element_size()
        base = d.data_ptr()
        return SsdGrads(base, Cd, base + HP * es, Cd, base + (HP + GN) * es, Cd, g["ddt_raw"].data_ptr(), s.nheads,
                        _ptr(g["ddt_bias"]), _ptr(g["dA_log"]), _ptr(g["dD"]), _ptr(g["dconv_w"]),
                        _ptr(g["dconv_b"]), _ptr(g.get("dinit")), _ptr(g.get("dz")), s.nheads * s.headdim,
                        _ptr(g.get("dnorm_weight")))

    def forward_varlen(self, t: dict, out=None, stream=None):
        """Forward of a packed row (t["cu_seqlens"], t["seq_idx"]); returns y,
        final_state, seg_init_states and the per-sequence final states."""
        y, fin, seg = out if out is not None else self.alloc_outputs()
        cu = t["cu_seqlens"]
        s = self.shape
        sf = torch.empty(cu.numel() - 1, s.nheads, s.headdim, s.dstate, dtype=torch.float32, device=self.device)
        ssd_forward_varlen(self.dims, self.inputs(t), y, fin, seg, cu, sf, self.workspace, stream=stream)
        return y, fin, seg, sf

    def forward(self, t: dict, out=None, stream=None):
        y, fin, seg = out if out is not None else self.alloc_outputs()
        ssd_forward(self.dims, self.inputs(t), y, fin, seg, self.workspace, stream=stream)
        return y, fin, seg

    def backward(self, t: dict, dy, dfinal=None, seg=None, grads=None, stream=None):
        g = grads if grads is not None else self.alloc_grads(init=t.get("init") is not None)
        ssd_backward(self.dims, self.inputs(t), dy, dfinal, seg, self.grads_struct(g), self.workspace,
                     stream=stream)
        return g

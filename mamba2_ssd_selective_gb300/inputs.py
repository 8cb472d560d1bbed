"""Seeded synthetic inputs for the Mamba2 SSD mixer core.

This module only draws random numbers and lays them out; it holds none of the
method's arithmetic.  Both the CUDA path (tests, bench) and the fp64 oracle read
the arrays it returns, so the two sides always see bit-identical inputs.

Distributions (the Mamba2 initialisation conventions used by the pages'
benchmarks, which time the mixer core on random post-projection activations):

* raw x, B, C (pre-conv), dt_raw, D and the upstream gradient dy ~ N(0, 1);
* dt_bias = softplus^-1(dt0) with dt0 log-uniform on [1e-3, 1e-1];
* A_log = log(U[1, 16]);
* conv_w ~ U(-0.5, 0.5) with shape (conv_dim, 4); conv_b = 0;
* packed batches: sequence lengths ~ U{512..8192} drawn until they cover the
  token count, the last one truncated.

Draw order from ``numpy.random.default_rng(seed)`` (PCG64), all in float32:
x, B, C, dt_raw, dt_bias, A_log, D, conv_w, [sequence lengths], dy, [dfinal],
[initial states ~ N(0, 1), (batch, H, P, N)], [the gate z ~ N(0, 1), (batch, L, H*P),
then the norm weight ~ U(0.5, 1.5), (H*P)]; the norm's eps is 1e-5.
Activations are then rounded to the activation dtype (round to nearest even);
parameters stay float32.
"""
from __future__ import annotations

from dataclasses import dataclass, replace

import numpy as np
import torch


@dataclass(frozen=True)
class SsdShape:
    batch: int
    seqlen: int
    nheads: int
    headdim: int
    dstate: int
    ngroups: int
    chunk: int
    n_segments: int
    d_conv: int = 4
    packed: bool = False  # seq_idx from random sequence lengths (batch must be 1)

    @property
    def conv_dim(self) -> int:
        return self.nheads * self.headdim + 2 * self.ngroups * self.dstate

    @property
    def tokens(self) -> int:
        return self.batch * self.seqlen

    def with_(self, **kw) -> "SsdShape":
        return replace(self, **kw)


# The five named workloads.  Seeds: 0 for the tiny fp32 case, 1-4 for the others.
WORKLOADS = {
    "tiny-fp32": (SsdShape(1, 512, 4, 32, 16, 1, 64, 4), "f32", 0),
    "mamba2-1b-fwd": (SsdShape(4, 8192, 64, 64, 128, 1, 256, 8), "bf16", 1),
    "mamba2-1b-fwdbwd": (SsdShape(4, 8192, 64, 64, 128, 1, 256, 8), "bf16", 2),
    "long-131k": (SsdShape(1, 131072, 64, 64, 128, 8, 256, 8), "bf16", 3),
    "packed-32k": (SsdShape(1, 32768, 48, 64, 128, 1, 256, 8, packed=True), "bf16", 4),
}

TORCH_DTYPES = {"bf16": torch.bfloat16, "f32": torch.float32}


def packed_lengths(rng: np.random.Generator, total: int, lo: int = 512, hi: int = 8192) -> list[int]:
    """Sequence lengths ~ U{lo..hi} drawn until they cover ``total``; last one truncated."""
    lens: list[int] = []
    acc = 0
    while acc < total:
        n = int(rng.integers(lo, hi + 1))
        n = min(n, total - acc)
        lens.append(n)
        acc += n
    return lens


def seq_idx_from_lengths(lengths: list[int]) -> np.ndarray:
    return np.repeat(np.arange(len(lengths), dtype=np.int32), lengths)


def make_inputs(shape: SsdShape, seed: int, dtype: str = "bf16", *, dfinal: bool = False,
                seq_lengths: list[int] | None = None, init_states: bool = False, gated_norm: bool = False) -> dict:
    """Return a dict of CPU tensors.

    ``xBC`` is one (batch, seqlen, conv_dim) activation buffer with channels
    [x (H*P) | B (G*N) | C (G*N)], the layout the in-projection produces; x, B and C
    are token-strided views into it.  ``seq_idx`` is None unless the shape is packed or
    ``seq_lengths`` (per batch row, summing to seqlen) is given.  ``init`` (each
    row's initial state, fp32) is None unless ``init_states``; ``z`` (the gate,
    activation dtype) and ``norm_weight`` are None unless ``gated_norm``.
    """
    rng = np.random.default_rng(seed)
    b, L, H, P, N, G = shape.batch, shape.seqlen, shape.nheads, shape.headdim, shape.dstate, shape.ngroups
    Cd = shape.conv_dim
    f32 = np.float32
    x = rng.standard_normal((b, L, H * P), dtype=f32)
    Bm = rng.standard_normal((b, L, G * N), dtype=f32)
    Cm = rng.standard_normal((b, L, G * N), dtype=f32)
    dt_raw = rng.standard_normal((b, L, H), dtype=f32)
    dt0 = np.exp(rng.uniform(np.log(1e-3), np.log(1e-1), size=H))
    dt_bias = np.log(np.expm1(dt0)).astype(f32)
    A_log = np.log(rng.uniform(1.0, 16.0, size=H)).astype(f32)
    D = rng.standard_normal(H, dtype=f32)
    conv_w = rng.uniform(-0.5, 0.5, size=(Cd, shape.d_conv)).astype(f32)
    conv_b = np.zeros(Cd, dtype=f32)
    seq_idx = None
    cu_seqlens = None
    if shape.packed:
        if b != 1:
            raise ValueError("packed workloads use batch=1 (THD layout)")
        lens = packed_lengths(rng, L)
        seq_idx = seq_idx_from_lengths(lens)[None, :]
        cu_seqlens = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    elif seq_lengths is not None:
        rows = seq_lengths if isinstance(seq_lengths[0], (list, tuple)) else [seq_lengths] * b
        seq_idx = np.stack([seq_idx_from_lengths(list(r)) for r in rows]).astype(np.int32)
        if seq_idx.shape != (b, L):
            raise ValueError("seq_lengths must sum to seqlen in every row")
    dy = rng.standard_normal((b, L, H * P), dtype=f32)
    df = rng.standard_normal((b, H, P, N), dtype=f32) if dfinal else np.zeros((b, H, P, N), f32)
    h0 = rng.standard_normal((b, H, P, N), dtype=f32) if init_states else None
    z = rng.standard_normal((b, L, H * P), dtype=f32) if gated_norm else None
    nw = rng.uniform(0.5, 1.5, size=H * P).astype(f32) if gated_norm else None

    tdt = TORCH_DTYPES[dtype]
    xBC = torch.from_numpy(np.concatenate([x, Bm, Cm], axis=-1)).to(tdt).contiguous()
    out = {
        "xBC": xBC,
        "dt_raw": torch.from_numpy(dt_raw).to(tdt).contiguous(),
        "dt_bias": torch.from_numpy(dt_bias),
        "A_log": torch.from_numpy(A_log),
        "D": torch.from_numpy(D),
        "conv_w": torch.from_numpy(conv_w),
        "conv_b": torch.from_numpy(conv_b),
        "seq_idx": None if seq_idx is None else torch.from_numpy(np.ascontiguousarray(seq_idx)),
        "cu_seqlens": None if cu_seqlens is None else torch.from_numpy(cu_seqlens),
        "dy": torch.from_numpy(dy).to(tdt).contiguous(),
        "dfinal": torch.from_numpy(df),
        "init": None if h0 is None else torch.from_numpy(h0),
        "z": None if z is None else torch.from_numpy(z).to(tdt).contiguous(),
        "norm_weight": None if nw is None else torch.from_numpy(nw),
        "norm_eps": 1e-5,
    }
    return out

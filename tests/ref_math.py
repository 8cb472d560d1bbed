"""Independent fp64 formulations used to pin the oracle (tests only).

None of this is the oracle's code: the conv is PyTorch's own conv1d, the SSD is
its quadratic (masked-attention) form -- the dual of the token recurrence in the
Mamba2 chunked algorithm that state-spaces/mamba issue #482 ("Sequence
parallelism in the mixer") refers to -- evaluated with dense matrices.
"""
from __future__ import annotations

import numpy as np
import torch


def conv_silu_torch(inp: dict, shape) -> tuple[np.ndarray, np.ndarray]:
    """(v, u) of shape (b, L, Cd) via torch conv1d(groups=Cd, padding=3), run per
    packed sequence so that no tap crosses a sequence boundary."""
    xBC = inp["xBC"].double()
    w = inp["conv_w"].double()[:, None, :]
    bias = inp["conv_b"].double()
    b, L, Cd = xBC.shape
    v = torch.empty_like(xBC)
    for r in range(b):
        if inp.get("seq_idx") is None:
            bounds = [(0, L)]
        else:
            si = inp["seq_idx"][r].numpy()
            cuts = [0] + [t for t in range(1, L) if si[t] != si[t - 1]] + [L]
            bounds = list(zip(cuts[:-1], cuts[1:]))
        for s0, s1 in bounds:
            seg = xBC[r, s0:s1].T[None]  # (1, Cd, len)
            out = torch.nn.functional.conv1d(seg, w, bias, padding=w.shape[-1] - 1, groups=Cd)
            v[r, s0:s1] = out[0, :, : s1 - s0].T
    u = v * torch.sigmoid(v)
    return v.numpy(), u.numpy()


def quadratic_ssd(inp: dict, shape) -> tuple[np.ndarray, np.ndarray]:
    """y (b, L, H, P) and final state (b, H, P, N) from the masked-attention form

        Y = (Lmask o (C B^T)) (dt o X) + D X,   Lmask[t,s] = exp(sum_{r=s+1..t} dt_r A)
                                                 for s <= t in the same sequence, else 0.
    """
    b, L, H, P, N, G = shape.batch, shape.seqlen, shape.nheads, shape.headdim, shape.dstate, shape.ngroups
    _, u = conv_silu_torch(inp, shape)
    ux = u[..., : H * P].reshape(b, L, H, P)
    uB = u[..., H * P: H * P + G * N].reshape(b, L, G, N)
    uC = u[..., H * P + G * N:].reshape(b, L, G, N)
    z = inp["dt_raw"].double().numpy() + inp["dt_bias"].double().numpy()
    dt = np.logaddexp(0.0, z)  # softplus
    A = -np.exp(inp["A_log"].double().numpy())
    D = inp["D"].double().numpy()
    y = np.zeros((b, L, H, P))
    fin = np.zeros((b, H, P, N))
    t_idx = np.arange(L)
    causal = t_idx[:, None] >= t_idx[None, :]
    for r in range(b):
        if inp.get("seq_idx") is None:
            same = np.ones((L, L), bool)
        else:
            si = inp["seq_idx"][r].numpy()
            same = si[:, None] == si[None, :]
        for h in range(H):
            g = h // (H // G)
            cs = np.cumsum(dt[r, :, h] * A[h])
            seg = cs[:, None] - cs[None, :]
            Lm = np.where(causal & same, np.exp(np.where(causal, seg, 0.0)), 0.0)
            Xs = dt[r, :, h, None] * ux[r, :, h]
            y[r, :, h] = (Lm * (uC[r, :, g] @ uB[r, :, g].T)) @ Xs + D[h] * ux[r, :, h]
            w_last = Lm[L - 1]  # weights of every token in the final state
            fin[r, h] = (w_last[:, None] * Xs).T @ uB[r, :, g]
    return y, fin

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
                                                 for s <= t in the same sequence, else 0,

    plus, with an initial state h0 (inp["init"]), the term exp(sum_{r=0..t} dt_r A) C_t h0
    for every token t of the row's first sequence (h0 is the state before token 0).
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
            if inp.get("init") is not None:
                h0 = inp["init"][r, h].double().numpy()  # P x N
                first = same[0]  # tokens of the row's first sequence
                e = np.where(first, np.exp(cs), 0.0)
                y[r, :, h] += e[:, None] * (uC[r, :, g] @ h0.T)
                fin[r, h] += e[L - 1] * h0
    return y, fin


def ssd_dt_bias_grad_f64(inp: dict, shape, round_u: bool) -> tuple[np.ndarray, np.ndarray]:
    """(ddt_bias, ddt_raw) of L = <dy, y> + <dfinal, final_state> by float64
    autograd through the quadratic form of the whole row, conv + SiLU per packed
    sequence.  With round_u the
    post-conv activations u are rounded to bf16 in the forward (the gradient
    passes straight through the rounding): everything else stays exact, so the
    difference to round_u=False is the error that storing u in bf16 alone puts
    into the dt gradients of any implementation that does so."""
    b, L, H, P, N, G = shape.batch, shape.seqlen, shape.nheads, shape.headdim, shape.dstate, shape.ngroups
    Cd, HP, GN = shape.conv_dim, H * P, G * N
    f64 = torch.float64
    xBC = inp["xBC"].to(f64)
    w = inp["conv_w"].to(f64)[:, None, :]
    dt_raw = inp["dt_raw"].to(f64).clone().requires_grad_(True)
    bias = inp["dt_bias"].to(f64).clone().requires_grad_(True)
    A = -torch.exp(inp["A_log"].to(f64))
    D = inp["D"].to(f64)
    dy = inp["dy"].to(f64)
    dfin = inp["dfinal"].to(f64)
    loss = torch.zeros((), dtype=f64)
    for r in range(b):
        si = None if inp.get("seq_idx") is None else inp["seq_idx"][r].numpy()
        cuts = [0] + ([t for t in range(1, L) if si[t] != si[t - 1]] if si is not None else []) + [L]
        v = torch.empty(L, Cd, dtype=f64)
        for s0, s1 in zip(cuts[:-1], cuts[1:]):
            seg = xBC[r, s0:s1].T[None]
            v[s0:s1] = torch.nn.functional.conv1d(seg, w, inp["conv_b"].to(f64), padding=3, groups=Cd)[0, :, :s1 - s0].T
        u = v * torch.sigmoid(v)
        if round_u:
            u = u + (u.to(torch.bfloat16).to(f64) - u).detach()
        same = torch.ones(L, L, dtype=torch.bool) if si is None else torch.from_numpy(si[:, None] == si[None, :])
        mask = torch.tril(torch.ones(L, L, dtype=torch.bool)) & same
        dt = torch.nn.functional.softplus(dt_raw[r] + bias)
        for h in range(H):
            g = h // (H // G)
            x, Bm, Cm = u[:, h * P:(h + 1) * P], u[:, HP + g * N:HP + (g + 1) * N], u[:, HP + GN + g * N:HP + GN + (g + 1) * N]
            cs = torch.cumsum(dt[:, h] * A[h], 0)
            Lm = torch.exp(torch.where(mask, cs[:, None] - cs[None, :], torch.full((L, L), -1e300, dtype=f64)))
            y = ((Cm @ Bm.T) * Lm * dt[None, :, h]) @ x + D[h] * x
            loss = loss + (y * dy[r, :, h * P:(h + 1) * P]).sum()
            wl = Lm[L - 1] * dt[:, h]  # the last token's weights (its own sequence only)
            fin = (x * wl[:, None]).T @ Bm  # state after the row's last token, P x N
            loss = loss + (fin * dfin[r, h]).sum()
    loss.backward()
    return bias.grad.numpy().copy(), dt_raw.grad.numpy().copy()

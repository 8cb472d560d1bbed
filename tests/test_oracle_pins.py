"""Pins for the fp64 oracle against facts fixed by the mathematics (CPU only).

The pages print no worked numeric example, so every pin is a closed form, an
independent formulation, a special case or an invariant the pages state:

* conv + SiLU equals PyTorch's grouped conv1d (a library routine) per sequence;
* the token recurrence equals the quadratic (masked-attention) SSD form;
* constant inputs with N = P = 1 give the geometric-series closed form;
* a -> 0 gives a memoryless output; B = 0 or C = 0 gives y = D x exactly;
* any segment count gives the unsegmented result, and the segment transform is
  affine in its initial state, S_out = a_block * S_in + S_ext (Megatron-LM PR
  #6808 "Add state-passing context parallelism for Mamba2", description);
* seq_idx resets make a packed row equal separate per-sequence runs (NeMo
  Automodel PR #1441, Key changes: seq_idx from cu_seqlens), and the state after
  each packed sequence equals that run's final state;
* an initial state (listed as not supported yet by the Megatron-LM PR, read as
  the state before a row's first token): the quadratic form with its decayed
  term, segment-count invariance with it, and continuation -- a row cut in two,
  the second part started from the first part's final state, gives the uncut
  row's outputs and final state;
* the backward equals central finite differences of the forward in every input,
  the initial state included;
* the gated RMSNorm after the mixer (kept outside the fused function by the
  Megatron-LM PR; Mamba2's gated norm, one norm group per B/C group): equal to
  torch's rms_norm of y * silu(z) per group (library routines), unit RMS per
  group with eps = 0 and unit weight, and its backward -- alone and through the
  whole path -- equal to central finite differences.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

from mamba2_ssd_selective_gb300.inputs import SsdShape, make_inputs
from tests.ref_math import conv_silu_torch, quadratic_ssd

SMALL = SsdShape(batch=2, seqlen=96, nheads=4, headdim=8, dstate=6, ngroups=2, chunk=16, n_segments=4)
TINY = SsdShape(1, 512, 4, 32, 16, 1, 64, 4)


def rel(a, b):
    return float(np.linalg.norm(np.asarray(a) - np.asarray(b)) / max(np.linalg.norm(np.asarray(b)), 1e-300))


def f64(inp):
    return {k: (v.double() if torch.is_tensor(v) and v.is_floating_point() else v) for k, v in inp.items()}


@pytest.mark.parametrize("seq", [None, [30, 2, 41, 23]])
def test_conv_matches_torch_conv1d(oracle_lib, seq):
    inp = make_inputs(SMALL, 11, "f32", seq_lengths=seq)
    v_ref, u_ref = conv_silu_torch(inp, SMALL)
    for b in range(SMALL.batch):
        u, v, ch = oracle_lib.conv(inp, SMALL, b=b)
        assert sorted(ch.tolist()) == list(range(SMALL.conv_dim))
        assert rel(v, v_ref[b][:, ch]) < 1e-14
        assert rel(u, u_ref[b][:, ch]) < 1e-14


@pytest.mark.parametrize("shape,seq", [
    (SMALL, None),
    (SMALL, [30, 2, 41, 23]),
    (SsdShape(1, 200, 3, 5, 7, 1, 8, 1), [1, 1, 3, 195]),
    (TINY, None),
])
def test_recurrence_equals_quadratic_form(oracle_lib, shape, seq):
    inp = make_inputs(shape, 5, "f32", seq_lengths=seq)
    y_ref, fin_ref = quadratic_ssd(inp, shape)
    out = oracle_lib.forward(inp, shape, n_segments=1)
    assert rel(out["y"], y_ref) < 1e-12
    assert rel(out["final_state"], fin_ref) < 1e-12


def test_geometric_series_closed_form(oracle_lib):
    L = 300
    shape = SsdShape(1, L, 1, 1, 1, 1, 4, 1)
    cx, cb, cc, zr = 0.7, -0.4, 1.3, 0.25
    xBC = torch.tensor([[[cx, cb, cc]] * L], dtype=torch.float64)
    inp = {
        "xBC": xBC, "dt_raw": torch.full((1, L, 1), zr, dtype=torch.float64),
        "dt_bias": torch.tensor([-1.0], dtype=torch.float64), "A_log": torch.tensor([np.log(0.8)]),
        "D": torch.tensor([0.3], dtype=torch.float64),
        "conv_w": torch.tensor([[0.0, 0.0, 0.0, 1.0]] * 3, dtype=torch.float64),
        "conv_b": torch.zeros(3, dtype=torch.float64), "seq_idx": None,
    }
    silu = lambda v: v / (1 + np.exp(-v))  # noqa: E731
    ux, uB, uC = silu(cx), silu(cb), silu(cc)
    dt = np.log1p(np.exp(zr - 1.0))
    a = np.exp(-0.8 * dt)
    t = np.arange(L)
    y_cf = uC * uB * dt * ux * (1 - a ** (t + 1)) / (1 - a) + 0.3 * ux
    fin_cf = uB * dt * ux * (1 - a ** L) / (1 - a)
    out = oracle_lib.forward(inp, shape, n_segments=1)
    assert rel(out["y"][0, :, 0, 0], y_cf) < 1e-13
    assert abs(out["final_state"][0, 0, 0, 0] - fin_cf) < 1e-13 * abs(fin_cf)
    out4 = oracle_lib.forward(inp, shape.with_(n_segments=4), n_segments=4)
    assert rel(out4["y"][0, :, 0, 0], y_cf) < 1e-13


def test_memoryless_limit(oracle_lib):
    inp = make_inputs(SMALL, 3, "f32")
    inp["A_log"] = torch.full_like(inp["A_log"], 40.0)  # A = -e^40: a_t underflows to 0
    _, u = conv_silu_torch(inp, SMALL)
    H, P, N, G = SMALL.nheads, SMALL.headdim, SMALL.dstate, SMALL.ngroups
    ux = u[..., : H * P].reshape(2, -1, H, P)
    uB = u[..., H * P: H * P + G * N].reshape(2, -1, G, N)
    uC = u[..., H * P + G * N:].reshape(2, -1, G, N)
    dt = np.logaddexp(0, inp["dt_raw"].double().numpy() + inp["dt_bias"].double().numpy())
    g = np.arange(H) // (H // G)
    bc = np.einsum("blgn,blgn->blg", uB, uC)[:, :, g]
    y_ref = dt[..., None] * ux * bc[..., None] + inp["D"].double().numpy()[None, None, :, None] * ux
    out = oracle_lib.forward(inp, SMALL, n_segments=2)
    assert rel(out["y"], y_ref) < 1e-13


@pytest.mark.parametrize("which", ["B", "C"])
def test_zero_B_or_C_gives_Dx(oracle_lib, which):
    inp = make_inputs(SMALL, 4, "f32")
    H, P, N, G = SMALL.nheads, SMALL.headdim, SMALL.dstate, SMALL.ngroups
    lo = H * P + (0 if which == "B" else G * N)
    inp["xBC"][..., lo: lo + G * N] = 0.0  # conv_b = 0 as well, so silu(0) = 0
    _, u = conv_silu_torch(inp, SMALL)
    ux = u[..., : H * P].reshape(2, -1, H, P)
    out = oracle_lib.forward(inp, SMALL, n_segments=4)
    # exact up to the last-bit difference between two SiLU evaluations
    np.testing.assert_allclose(out["y"], inp["D"].double().numpy()[None, None, :, None] * ux, rtol=1e-14, atol=0)


@pytest.mark.parametrize("seq", [None, [100, 156, 7, 249]])
def test_segment_count_invariance(oracle_lib, seq):
    shape = SsdShape(1, 512, 4, 8, 8, 2, 16, 1)
    inp = make_inputs(shape, 9, "f32", seq_lengths=seq)
    base = oracle_lib.forward(inp, shape, n_segments=1)
    for S in (2, 4, 8, 16):
        out = oracle_lib.forward(inp, shape, n_segments=S)
        assert rel(out["y"], base["y"]) < 1e-12, S
        assert rel(out["final_state"], base["final_state"]) < 1e-12, S


def test_affine_segment_identity(oracle_lib):
    """Two rows share the second half (and the 3-token conv halo before it) but
    differ earlier, so the second segment sees two different initial states."""
    shape = SsdShape(2, 128, 2, 4, 5, 1, 8, 2)
    inp = make_inputs(shape, 21, "f32")
    inp["xBC"][1, 61:] = inp["xBC"][0, 61:]
    inp["dt_raw"][1, 64:] = inp["dt_raw"][0, 64:]
    inp["A_log"][:] = float(np.log(0.05))  # slow decay: a_block = O(1), no cancellation in d_out
    out = oracle_lib.forward(inp, shape, n_segments=2)
    s_ext, a_blk, s_in = out["s_ext"][:, 1], out["a_block"][:, 1], out["seg_in"][:, 1]
    assert rel(s_ext[0], s_ext[1]) < 1e-15 and rel(a_blk[0], a_blk[1]) < 1e-15
    assert rel(s_in[0], s_in[1]) > 1e-2  # genuinely different initial states
    assert a_blk.min() > 0.1
    d_out = out["final_state"][0] - out["final_state"][1]
    d_in = s_in[0] - s_in[1]
    assert rel(d_out, a_blk[0][:, None, None] * d_in) < 1e-13
    # and S_out(0) = S_ext: the unsegmented run of the second half alone
    fin = out["final_state"][0]
    assert rel(fin, a_blk[0][:, None, None] * s_in[0] + s_ext[0]) < 1e-13


def test_packed_equals_separate_runs(oracle_lib):
    lens = [37, 3, 90, 1, 125]
    L = sum(lens)
    shape = SsdShape(1, L, 2, 6, 4, 1, 8, 1)
    inp = make_inputs(shape, 13, "f32", seq_lengths=lens)
    out = oracle_lib.forward(inp, shape, n_segments=1)
    s0 = 0
    for n in lens:
        sub = {k: (v[:, s0:s0 + n] if k in ("xBC", "dt_raw") else v) for k, v in inp.items()}
        sub["seq_idx"] = None
        o = oracle_lib.forward(sub, shape.with_(seqlen=n), n_segments=1)
        assert rel(out["y"][:, s0:s0 + n], o["y"]) < 1e-14
        s0 += n
    assert rel(out["final_state"], o["final_state"]) < 1e-14


def test_packed_sequence_finals_equal_separate_runs(oracle_lib):
    lens = [37, 3, 90, 1, 125]
    L = sum(lens)
    shape = SsdShape(1, L, 2, 6, 4, 1, 8, 1)
    inp = make_inputs(shape, 14, "f32", seq_lengths=lens, init_states=True)
    fins = oracle_lib.seq_finals(inp, shape)
    assert fins.shape == (len(lens), 2, 6, 4)
    s0 = 0
    for q, n in enumerate(lens):
        sub = {k: (v[:, s0:s0 + n] if k in ("xBC", "dt_raw") else v) for k, v in inp.items()}
        sub["seq_idx"] = None
        if q > 0:
            sub["init"] = None  # only the row's first sequence starts from the initial state
        o = oracle_lib.forward(sub, shape.with_(seqlen=n), n_segments=1)
        assert rel(fins[q], o["final_state"][0]) < 1e-14
        s0 += n
    assert rel(fins[-1], oracle_lib.forward(inp, shape, n_segments=1)["final_state"][0]) < 1e-14


@pytest.mark.parametrize("shape,seq", [
    (SMALL, None),
    (SMALL, [30, 2, 41, 23]),
    (SsdShape(1, 200, 3, 5, 7, 1, 8, 1), [1, 1, 3, 195]),
])
def test_initial_state_equals_quadratic_form(oracle_lib, shape, seq):
    inp = make_inputs(shape, 6, "f32", seq_lengths=seq, init_states=True)
    y_ref, fin_ref = quadratic_ssd(inp, shape)
    out = oracle_lib.forward(inp, shape, n_segments=1)
    assert rel(out["y"], y_ref) < 1e-12
    assert rel(out["final_state"], fin_ref) < 1e-12
    for S in (2, 4, 8):
        o = oracle_lib.forward(inp, shape, n_segments=S)
        assert rel(o["y"], y_ref) < 1e-12 and rel(o["final_state"], fin_ref) < 1e-12, S
        assert rel(o["seg_in"][:, 0], inp["init"].double().numpy()) == 0.0  # the scan starts from it


@pytest.mark.parametrize("cut", [1, 57, 128])
def test_continuation_from_a_final_state(oracle_lib, cut):
    """A row cut at token `cut`: the second part, started from the first part's
    final state, reproduces the uncut row.  Conv taps before the current token
    are zeroed so that the conv carries nothing across the cut."""
    shape = SsdShape(2, 256, 4, 8, 6, 2, 16, 1)
    inp = make_inputs(shape, 15, "f32", init_states=True)
    inp["conv_w"][:, :3] = 0.0
    full = oracle_lib.forward(inp, shape, n_segments=1)
    a = {k: (v[:, :cut] if k in ("xBC", "dt_raw") else v) for k, v in inp.items()}
    pa = oracle_lib.forward(a, shape.with_(seqlen=cut), n_segments=1)
    b = {k: (v[:, cut:] if k in ("xBC", "dt_raw") else v) for k, v in inp.items()}
    b["init"] = torch.from_numpy(pa["final_state"])
    pb = oracle_lib.forward(b, shape.with_(seqlen=256 - cut), n_segments=1)
    assert rel(pa["y"], full["y"][:, :cut]) < 1e-13
    assert rel(pb["y"], full["y"][:, cut:]) < 1e-12
    assert rel(pb["final_state"], full["final_state"]) < 1e-12


def test_head_subsets_match_full(oracle_lib):
    shape = SsdShape(1, 64, 6, 4, 3, 3, 8, 2)
    inp = make_inputs(shape, 17, "f32", dfinal=True)
    full = oracle_lib.forward(inp, shape)
    part = oracle_lib.forward(inp, shape, heads=(2, 4))
    np.testing.assert_array_equal(part["y"], full["y"][:, :, 2:4])
    gf = oracle_lib.backward(inp, shape)
    gp = oracle_lib.backward(inp, shape, heads=(2, 4))
    idx = [list(gf["channels"]).index(c) for c in gp["channels"]]
    np.testing.assert_allclose(gp["dxBC"], gf["dxBC"][..., idx], rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(gp["ddt_raw"], gf["ddt_raw"][..., 2:4], rtol=1e-13, atol=1e-14)


# ---------------------------------------------------------------- backward

def _loss(oracle_lib, inp, shape):
    out = oracle_lib.forward(inp, shape, n_segments=1, nthreads=1)
    y = out["y"].reshape(shape.batch, shape.seqlen, -1)
    return float(np.sum(inp["dy"].double().numpy() * y) + np.sum(inp["dfinal"].double().numpy() * out["final_state"]))


@pytest.mark.parametrize("shape,seq,init", [
    (SsdShape(2, 40, 4, 3, 5, 2, 8, 1), None, False),
    (SsdShape(1, 60, 2, 4, 3, 1, 8, 1), [17, 1, 2, 40], False),
    # longer than the oracle's 256-token checkpoint interval
    (SsdShape(1, 600, 2, 3, 2, 1, 8, 1), [255, 1, 344], False),
    # with initial states: every input and the initial state itself
    (SsdShape(2, 40, 4, 3, 5, 2, 8, 1), None, True),
    (SsdShape(1, 300, 2, 4, 3, 1, 8, 1), [260, 1, 39], True),
    # the whole path through the gated norm: also z and the norm weight
    (SsdShape(2, 40, 4, 3, 5, 2, 8, 1), [15, 25], "norm"),
])
def test_backward_matches_finite_differences(oracle_lib, shape, seq, init):
    norm = init == "norm"
    inp = f64(make_inputs(shape, 23, "f32", dfinal=True, seq_lengths=seq, init_states=init is True, gated_norm=norm))
    g = oracle_lib.backward(inp, shape, nthreads=1)
    dxBC = np.zeros((shape.batch, shape.seqlen, shape.conv_dim))
    dxBC[..., g["channels"]] = g["dxBC"]
    dconv_w = np.zeros((shape.conv_dim, 4))
    dconv_w[g["channels"]] = g["dconv_w"]
    dconv_b = np.zeros(shape.conv_dim)
    dconv_b[g["channels"]] = g["dconv_b"]
    grads = {"xBC": dxBC, "dt_raw": g["ddt_raw"], "dt_bias": g["ddt_bias"], "A_log": g["dA_log"], "D": g["dD"],
             "conv_w": dconv_w, "conv_b": dconv_b}
    if init is True:
        grads["init"] = g["dinit"]
    if norm:
        grads["z"] = g["dz"]
        grads["norm_weight"] = g["dnorm_weight"]
    rng = np.random.default_rng(0)
    HP, GN = shape.nheads * shape.headdim, shape.ngroups * shape.dstate
    parts = {"x": slice(0, HP), "B": slice(HP, HP + GN), "C": slice(HP + GN, HP + 2 * GN)}
    cases = [("xBC", k) for k in parts] + [(k, None) for k in grads if k != "xBC"]
    for name, part in cases:
        v = rng.standard_normal(grads[name].shape)
        if part is not None:
            mask = np.zeros_like(v)
            mask[..., parts[part]] = 1.0
            v *= mask
        eps = 1e-5
        plus, minus = dict(inp), dict(inp)
        plus[name] = inp[name] + eps * torch.from_numpy(v)
        minus[name] = inp[name] - eps * torch.from_numpy(v)
        fd = (_loss(oracle_lib, plus, shape) - _loss(oracle_lib, minus, shape)) / (2 * eps)
        an = float(np.sum(grads[name] * v))
        assert abs(fd - an) <= 1e-7 * max(1.0, abs(an)), (name, part, fd, an)


# ---------------------------------------------------------------- gated RMSNorm

@pytest.mark.parametrize("G", [1, 2, 4])
def test_gated_norm_equals_torch_rms_norm(oracle_lib, G):
    rng = np.random.default_rng(31)
    L, C = 50, 96
    y, z = rng.standard_normal((2, L, C)), rng.standard_normal((2, L, C))
    w = rng.uniform(0.5, 1.5, C)
    out = oracle_lib.gated_norm(y, z, w, G, 1e-5)
    g = torch.from_numpy(y) * torch.nn.functional.silu(torch.from_numpy(z))
    ref = torch.nn.functional.rms_norm(g.reshape(2, L, G, C // G), (C // G,), eps=1e-5).reshape(2, L, C)
    ref = ref * torch.from_numpy(w)
    assert rel(out, ref.numpy()) < 1e-14


def test_gated_norm_unit_rms_per_group(oracle_lib):
    rng = np.random.default_rng(32)
    L, C, G = 20, 64, 4
    y, z = rng.standard_normal((1, L, C)) * 7.0, rng.standard_normal((1, L, C))
    out = oracle_lib.gated_norm(y, z, np.ones(C), G, 0.0)
    ms = np.mean(out.reshape(1, L, G, C // G) ** 2, axis=-1)
    np.testing.assert_allclose(ms, 1.0, rtol=1e-13)
    # and a scaled input gives the same output (the norm removes the scale)
    assert rel(oracle_lib.gated_norm(3.5 * y, z, np.ones(C), G, 0.0), out) < 1e-14


def test_gated_norm_backward_matches_finite_differences(oracle_lib):
    rng = np.random.default_rng(33)
    L, C, G, eps = 7, 24, 2, 1e-5
    y, z = rng.standard_normal((2, L, C)), rng.standard_normal((2, L, C))
    w, dout = rng.uniform(0.5, 1.5, C), rng.standard_normal((2, L, C))
    dy, dz, dw = oracle_lib.gated_norm_backward(y, z, w, G, eps, dout)
    loss = lambda yy, zz, ww: float(np.sum(dout * oracle_lib.gated_norm(yy, zz, ww, G, eps)))  # noqa: E731
    h = 1e-6
    for name, grad in (("y", dy), ("z", dz), ("w", dw)):
        v = rng.standard_normal(grad.shape)
        args_p = {"y": y, "z": z, "w": w}
        args_m = dict(args_p)
        args_p[name] = args_p[name] + h * v
        args_m[name] = args_m[name] - h * v
        fd = (loss(args_p["y"], args_p["z"], args_p["w"]) - loss(args_m["y"], args_m["z"], args_m["w"])) / (2 * h)
        an = float(np.sum(grad * v))
        assert abs(fd - an) <= 1e-7 * max(1.0, abs(an)), (name, fd, an)

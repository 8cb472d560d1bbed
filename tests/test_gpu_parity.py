"""GPU parity: libssd through its C ABI against the fp64 oracle (relative L2).

Tolerances: 1e-4 for the fp32 path, 1e-2 for bf16 activations with fp32
accumulation (ddt_bias in three named small cases: see tests/gpu_util.py).  Shapes span several chunk tiles, partial tiles (chunk 96,
headdim 32, dstate 40), group mapping (G > 1), packed sequences with edge
cases (a boundary at a chunk start, at a segment start, sequences of 1-3
tokens and sequences shorter than a chunk), every segment count 1..16, initial
states with their gradient, per-sequence final states of packed rows, the
gated RMSNorm after the mixer with its backward, and the bitwise replay the
pages require of summaries, scans and outputs.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import mamba2_ssd_selective_gb300 as ssd
from mamba2_ssd_selective_gb300.inputs import WORKLOADS, SsdShape, make_inputs
from tests.gpu_util import TOL, compare_backward, compare_forward, gpu_backward, gpu_forward, np_, rel, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mamba2_ssd_selective_gb300.build import build

    build()
    ssd.load()


def test_tiny_fp32_forward_backward(oracle_lib):
    shape, dtype, seed = WORKLOADS["tiny-fp32"]
    inp = make_inputs(shape, seed, dtype, dfinal=True)
    got, _ = gpu_forward(shape, dtype, inp)
    compare_forward(got, oracle_lib.forward(inp, shape), TOL[dtype])
    g = gpu_backward(shape, dtype, inp)
    compare_backward(g, oracle_lib.backward(inp, shape), shape, TOL[dtype])


SHAPES = [
    (SsdShape(2, 1024, 8, 64, 128, 2, 256, 2), None, None),
    (SsdShape(1, 768, 4, 64, 64, 1, 96, 4), None, None),
    (SsdShape(1, 512, 6, 32, 40, 3, 64, 8), None, None),
    # boundaries at token 256 (a chunk start), 512 (a segment start), 1-3 token
    # sequences, and sequences shorter than a chunk
    (SsdShape(1, 2048, 4, 64, 128, 1, 256, 4), [256, 256, 1, 2, 3, 90, 160, 700, 580], "packed-2048-q256"),
    # the tensor-core path with 128-token chunks (one row tile per chunk), packed
    (SsdShape(2, 1024, 4, 64, 128, 1, 128, 2), [128, 5, 300, 77, 514], "packed-2x1024-q128"),
    # two heads per group (the tensor-core kernels' smallest head blocks) and sixteen
    # (their largest at this size), with more units than SMs in neither case
    (SsdShape(1, 1024, 8, 64, 128, 4, 256, 2), None, None),
    (SsdShape(2, 1024, 16, 64, 128, 1, 256, 4), None, None),
]


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("shape,seq,floor_case", SHAPES)
def test_forward_backward_parity(oracle_lib, shape, seq, floor_case, dtype):
    inp = make_inputs(shape, 7, dtype, dfinal=True, seq_lengths=seq)
    got, _ = gpu_forward(shape, dtype, inp)
    compare_forward(got, oracle_lib.forward(inp, shape), TOL[dtype])
    g = gpu_backward(shape, dtype, inp)
    compare_backward(g, oracle_lib.backward(inp, shape), shape, TOL[dtype],
                     floor_case=floor_case if dtype == "bf16" else None)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_heads_that_forget_within_a_token(oracle_lib, dtype):
    """Heads 0-1 with dt near 2 (per-token decay e^-2|A|): the diagonal of V
    enters the Acs adjoint twice with opposite signs, so it must cancel exactly
    for dA_log to keep its accuracy; heads 2-3 keep the workload's decays."""
    shape = SsdShape(1, 1024, 4, 64, 128, 1, 256, 2)
    inp = make_inputs(shape, 11, dtype, dfinal=True, seq_lengths=[300, 1, 211, 512])
    inp["dt_bias"][:2] = 2.0
    got, _ = gpu_forward(shape, dtype, inp)
    compare_forward(got, oracle_lib.forward(inp, shape), TOL[dtype])
    g = gpu_backward(shape, dtype, inp)
    compare_backward(g, oracle_lib.backward(inp, shape), shape, TOL[dtype],
                     floor_case="forget-1024" if dtype == "bf16" else None)


@pytest.mark.parametrize("dtype,seq", [("f32", None), ("bf16", None), ("bf16", [1000, 3, 2093, 1000])])
@pytest.mark.parametrize("S", [1, 2, 4, 8, 16])
def test_segment_count_sweep(oracle_lib, S, dtype, seq):
    shape = SsdShape(1, 4096, 4, 64, 128, 1, 256, S)
    inp = make_inputs(shape, 8, dtype, seq_lengths=seq)
    ref = oracle_lib.forward(inp, shape, n_segments=1)
    got, _ = gpu_forward(shape, dtype, inp)
    assert rel(got["y"], ref["y"]) <= TOL[dtype]
    assert rel(got["final_state"], ref["final_state"]) <= TOL[dtype]
    g = gpu_backward(shape, dtype, inp, use_dfinal=False)
    compare_backward(g, oracle_lib.backward(inp, shape, use_dfinal=False), shape, TOL[dtype])


def test_reads_the_in_projection_output_in_place(oracle_lib):
    """x, B, C and dt read straight out of one (b, L, z | x | B | C | dt) buffer, the
    layout the in-projection GEMM writes, through token strides; the gradients
    written into the matching slots of one such buffer.  Nothing is copied."""
    shape = SsdShape(1, 1024, 8, 64, 128, 1, 256, 2)
    inp = make_inputs(shape, 13, "bf16", dfinal=True, seq_lengths=[700, 324])
    s = shape
    HP, GN, H, Cd = s.nheads * s.headdim, s.ngroups * s.dstate, s.nheads, s.conv_dim
    D_in = 2 * HP + 2 * GN + H  # z | x | B | C | dt, a multiple of 8 elements here
    t = to_dev(inp)
    zxbcdt = torch.randn(s.batch, s.seqlen, D_in, device="cuda").to(torch.bfloat16)
    zxbcdt[..., HP:HP + Cd] = t["xBC"]
    zxbcdt[..., HP + Cd:] = t["dt_raw"]
    es, base = zxbcdt.element_size(), zxbcdt.data_ptr()
    ins = ssd.SsdInputs(base + HP * es, D_in, base + 2 * HP * es, D_in, base + (2 * HP + GN) * es, D_in,
                        base + (HP + Cd) * es, D_in, t["dt_bias"].data_ptr(), t["A_log"].data_ptr(),
                        t["D"].data_ptr(), t["conv_w"].data_ptr(), t["conv_b"].data_ptr(), t["seq_idx"].data_ptr())
    r = ssd.SsdRunner(shape, "bf16")
    y, fin, seg = r.alloc_outputs()
    ssd.ssd_forward(r.dims, ins, y, fin, seg, r.workspace)
    torch.cuda.synchronize()
    got = {"y": y.float().cpu().numpy().reshape(s.batch, s.seqlen, H, s.headdim),
           "final_state": fin.cpu().numpy(), "seg_in": seg.cpu().numpy()}
    compare_forward(got, oracle_lib.forward(inp, shape), TOL["bf16"])
    dbuf = torch.full_like(zxbcdt, float("nan"))  # the z slot must stay untouched
    g = r.alloc_grads()
    gb, dbase = dbuf.element_size(), dbuf.data_ptr()
    gs = ssd.SsdGrads(dbase + HP * gb, D_in, dbase + 2 * HP * gb, D_in, dbase + (2 * HP + GN) * gb, D_in,
                      dbase + (HP + Cd) * gb, D_in, g["ddt_bias"].data_ptr(), g["dA_log"].data_ptr(),
                      g["dD"].data_ptr(), g["dconv_w"].data_ptr(), g["dconv_b"].data_ptr())
    ssd.ssd_backward(r.dims, ins, t["dy"], t["dfinal"], seg, gs, r.workspace)
    torch.cuda.synchronize()
    assert torch.isnan(dbuf[..., :HP].float()).all()
    out = {"dxBC": dbuf[..., HP:HP + Cd].float().cpu().numpy(), "ddt_raw": dbuf[..., HP + Cd:].float().cpu().numpy()}
    out.update({k: g[k].float().cpu().numpy() for k in ("ddt_bias", "dA_log", "dD", "dconv_w", "dconv_b")})
    compare_backward(out, oracle_lib.backward(inp, shape), shape, TOL["bf16"])


INIT_SHAPES = [
    (SsdShape(2, 1024, 8, 64, 128, 2, 256, 2), None),
    (SsdShape(1, 768, 4, 64, 64, 1, 96, 4), [70, 3, 695]),
    # the tensor-core path with 128-token chunks: the first sequence ends inside chunk 0
    (SsdShape(1, 1024, 4, 64, 128, 1, 128, 4), [100, 5, 919]),
    (SsdShape(1, 2048, 4, 64, 128, 1, 256, 8), [1300, 748]),
]


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("shape,seq", INIT_SHAPES)
def test_initial_states_forward_backward(oracle_lib, shape, seq, dtype):
    """Each row starts from its own initial state; with packed rows only the
    first sequence does.  The gradient of the initial states comes from the
    reverse segment scan carried one step past the first segment."""
    inp = make_inputs(shape, 19, dtype, dfinal=True, seq_lengths=seq, init_states=True)
    got, _ = gpu_forward(shape, dtype, inp)
    ref = oracle_lib.forward(inp, shape)
    compare_forward(got, ref, TOL[dtype])
    assert np.array_equal(got["seg_in"][:, 0], inp["init"].numpy())  # the scan starts from it
    g = gpu_backward(shape, dtype, inp)
    errs = compare_backward(g, oracle_lib.backward(inp, shape), shape, TOL[dtype])
    assert "dinit" in errs


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("init", [False, True])
def test_varlen_sequence_final_states(oracle_lib, dtype, init):
    """ssd_forward_varlen: the state after every packed sequence's last token,
    including sequences of 1-3 tokens, one ending on a chunk's last token and one
    inside the row's first chunk."""
    lens = [200, 56, 1, 2, 3, 250, 512, 1000, 24]
    shape = SsdShape(1, sum(lens), 4, 64, 128, 1, 256, 4)
    inp = make_inputs(shape, 20, dtype, seq_lengths=lens, init_states=init)
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int32)
    r = ssd.SsdRunner(shape, dtype)
    t = to_dev(inp)
    t["cu_seqlens"] = cu.cuda()
    y, fin, seg, sf = r.forward_varlen(t)
    torch.cuda.synchronize()
    ref = oracle_lib.forward(inp, shape)
    got = {"y": np_(y).reshape(1, shape.seqlen, shape.nheads, shape.headdim), "final_state": np_(fin),
           "seg_in": np_(seg)}
    compare_forward(got, ref, TOL[dtype])
    fins = oracle_lib.seq_finals(inp, shape)
    assert rel(np_(sf), fins) <= TOL[dtype]
    for q in range(len(lens)):
        assert rel(np_(sf[q]), fins[q]) <= 2 * TOL[dtype], q
    # the row's last sequence ends at the row's last token: its state is the final state
    assert rel(np_(sf[-1]), np_(fin)[0]) <= TOL[dtype]


NORM_SHAPES = [
    # norm groups of 8 and 4 heads (512 and 256 channels: a warp per token and group)
    (SsdShape(2, 1024, 8, 64, 128, 1, 256, 2), None),
    (SsdShape(1, 1024, 8, 64, 128, 2, 256, 4), [300, 3, 721]),
    # a group of 32 heads (2048 channels: a block per token and group)
    (SsdShape(1, 512, 32, 64, 128, 1, 256, 2), [200, 312]),
    (SsdShape(1, 512, 8, 32, 40, 4, 64, 2), None),  # CUDA-core path (headdim 32) in bf16 as well
]


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("shape,seq", NORM_SHAPES)
def test_gated_norm_forward_backward(oracle_lib, shape, seq, dtype):
    """y = gated RMSNorm of the mixer output (one norm group per B/C group);
    the backward recomputes the mixer output and returns dz and the norm
    weight's gradient besides every other gradient."""
    inp = make_inputs(shape, 29, dtype, dfinal=True, seq_lengths=seq, gated_norm=True)
    got, _ = gpu_forward(shape, dtype, inp)
    compare_forward(got, oracle_lib.forward(inp, shape), TOL[dtype])
    g = gpu_backward(shape, dtype, inp)
    errs = compare_backward(g, oracle_lib.backward(inp, shape), shape, TOL[dtype])
    assert "dz" in errs and "dnorm_weight" in errs


def test_gated_norm_reads_z_from_the_in_projection_output(oracle_lib):
    """z, x, B, C and dt all read in place from one (z | x | B | C | dt) buffer, and
    dz, dx, dB, dC, ddt written into the slots of one such gradient buffer."""
    shape = SsdShape(1, 1024, 8, 64, 128, 1, 256, 2)
    inp = make_inputs(shape, 30, "bf16", dfinal=True, seq_lengths=[600, 424], gated_norm=True)
    s = shape
    HP, GN, H, Cd = s.nheads * s.headdim, s.ngroups * s.dstate, s.nheads, s.conv_dim
    D_in = 2 * HP + 2 * GN + H
    t = to_dev(inp)
    buf = torch.empty(s.batch, s.seqlen, D_in, device="cuda", dtype=torch.bfloat16)
    buf[..., :HP] = t["z"]
    buf[..., HP:HP + Cd] = t["xBC"]
    buf[..., HP + Cd:] = t["dt_raw"]
    es, base = buf.element_size(), buf.data_ptr()
    ins = ssd.SsdInputs(base + HP * es, D_in, base + 2 * HP * es, D_in, base + (2 * HP + GN) * es, D_in,
                        base + (HP + Cd) * es, D_in, t["dt_bias"].data_ptr(), t["A_log"].data_ptr(),
                        t["D"].data_ptr(), t["conv_w"].data_ptr(), t["conv_b"].data_ptr(), t["seq_idx"].data_ptr(),
                        None, base, D_in, t["norm_weight"].data_ptr(), inp["norm_eps"])
    r = ssd.SsdRunner(shape, "bf16", gated_norm=True)
    y, fin, seg = r.alloc_outputs()
    ssd.ssd_forward(r.dims, ins, y, fin, seg, r.workspace)
    dbuf = torch.full_like(buf, float("nan"))
    g = r.alloc_grads()
    gb, dbase = dbuf.element_size(), dbuf.data_ptr()
    gs = ssd.SsdGrads(dbase + HP * gb, D_in, dbase + 2 * HP * gb, D_in, dbase + (2 * HP + GN) * gb, D_in,
                      dbase + (HP + Cd) * gb, D_in, g["ddt_bias"].data_ptr(), g["dA_log"].data_ptr(),
                      g["dD"].data_ptr(), g["dconv_w"].data_ptr(), g["dconv_b"].data_ptr(), None, dbase, D_in,
                      g["dnorm_weight"].data_ptr())
    ssd.ssd_backward(r.dims, ins, t["dy"], t["dfinal"], seg, gs, r.workspace)
    torch.cuda.synchronize()
    got = {"y": np_(y).reshape(1, s.seqlen, H, s.headdim), "final_state": np_(fin), "seg_in": np_(seg)}
    compare_forward(got, oracle_lib.forward(inp, shape), TOL["bf16"])
    out = {"dxBC": np_(dbuf[..., HP:HP + Cd]), "ddt_raw": np_(dbuf[..., HP + Cd:]), "dz": np_(dbuf[..., :HP])}
    out.update({k: np_(g[k]) for k in ("ddt_bias", "dA_log", "dD", "dconv_w", "dconv_b", "dnorm_weight")})
    compare_backward(out, oracle_lib.backward(inp, shape), shape, TOL["bf16"])


def test_backward_recomputes_segment_states(oracle_lib):
    shape = SsdShape(1, 1024, 4, 64, 128, 1, 128, 4)
    inp = make_inputs(shape, 12, "bf16", dfinal=True)
    a = gpu_backward(shape, "bf16", inp, pass_seg=True)
    b = gpu_backward(shape, "bf16", inp, pass_seg=False)
    for k in a:
        assert np.array_equal(a[k], b[k]), k


def test_replay_is_bitwise_identical():
    shape = SsdShape(2, 2048, 8, 64, 128, 1, 256, 4)
    inp = make_inputs(shape, 3, "bf16", dfinal=True, seq_lengths=[700, 3, 1345])
    r = ssd.SsdRunner(shape, "bf16")
    t = to_dev(inp)
    y1, f1, s1 = [x.clone() for x in r.forward(t)]
    g1 = {k: v.clone() for k, v in r.backward(t, t["dy"], t["dfinal"], s1).items()}
    y2, f2, s2 = r.forward(t)
    g2 = r.backward(t, t["dy"], t["dfinal"], s2)
    torch.cuda.synchronize()
    assert torch.equal(y1, y2) and torch.equal(f1, f2) and torch.equal(s1, s2)
    for k in g1:
        assert torch.equal(g1[k], g2[k]), k
    assert ssd.ssd_device_status(r.workspace) == 0


def test_cu_seqlens_to_seq_idx():
    lens = [5, 1, 300, 2, 700]
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int32, device="cuda")
    out = torch.empty(int(cu[-1]), dtype=torch.int32, device="cuda")
    ssd.ssd_cu_seqlens_to_seq_idx(cu, out)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(out.cpu().numpy(), np.repeat(np.arange(len(lens)), lens))

"""Full-size parity: every named workload at its real size, run exactly as the
benchmark runs it (same entry points, same workspace), compared with the fp64
oracle on samples it can compute: whole batch rows, or whole groups of heads
(so the B/C channel and parameter gradients of the sample are exact).

  mamba2-1b-fwd     b4 L8192 H64 P64 N128 G1 Q256 S8   forward, rows 0 and 3 all heads
  mamba2-1b-fwdbwd  same shape, forward + backward, all rows, all heads
  long-131k         b1 L131072 H64 G8, segment count swept over 1..16: heads 0-7
                    (group 0) against one unsegmented oracle run (invariance)
  packed-32k        b1 T32768 H48 G1, packed sequences, forward + backward, all heads;
                    and again from a random initial state, with every sequence's
                    final state (ssd_forward_varlen) and the initial state's gradient
  with the gated RMSNorm: mamba2-1b-fwdbwd (one 64-head norm group: a separate
                    norm pass) forward + backward, and long-131k S8 forward, heads
                    0-7 (8-head groups: the norm inside the output kernel)
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import mamba2_ssd_selective_gb300 as ssd
from mamba2_ssd_selective_gb300.inputs import WORKLOADS, make_inputs
from tests.gpu_util import TOL, compare_backward, compare_forward, np_, to_dev

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mamba2_ssd_selective_gb300.build import build

    build()
    ssd.load()


def _run(shape, dtype, inp, backward: bool, use_dfinal: bool = False):
    r = ssd.SsdRunner(shape, dtype)
    t = to_dev(inp)
    y, fin, seg = r.forward(t)
    out = {"y": np_(y).reshape(shape.batch, shape.seqlen, shape.nheads, shape.headdim),
           "final_state": np_(fin), "seg_in": np_(seg)}
    g = None
    if backward:
        gr = r.backward(t, t["dy"], t["dfinal"] if use_dfinal else None, seg)
        torch.cuda.synchronize()
        g = {k: np_(v) for k, v in gr.items()}
    del r, t
    torch.cuda.empty_cache()
    return out, g


def test_mamba2_1b_forward(oracle_lib):
    shape, dtype, seed = WORKLOADS["mamba2-1b-fwd"]
    inp = make_inputs(shape, seed, dtype)
    got, _ = _run(shape, dtype, inp, backward=False)
    rows = [0, 3]
    ref = oracle_lib.forward(inp, shape, rows=rows)
    errs = compare_forward(got, ref, TOL[dtype], rows=rows)
    print("mamba2-1b-fwd", errs)


def test_mamba2_1b_forward_backward(oracle_lib):
    shape, dtype, seed = WORKLOADS["mamba2-1b-fwdbwd"]
    inp = make_inputs(shape, seed, dtype)
    got, g = _run(shape, dtype, inp, backward=True)
    compare_forward(got, oracle_lib.forward(inp, shape, rows=[1]), TOL[dtype], rows=[1])
    gref = oracle_lib.backward(inp, shape, use_dfinal=False)
    errs = compare_backward(g, gref, shape, TOL[dtype])
    print("mamba2-1b-fwdbwd", errs)


def test_long_131k_segment_sweep(oracle_lib):
    base, dtype, seed = WORKLOADS["long-131k"]
    inp = make_inputs(base, seed, dtype, dfinal=True)
    heads = (0, base.nheads // base.ngroups)  # group 0
    ref = oracle_lib.forward(inp, base.with_(n_segments=1), n_segments=1, heads=heads)
    gref = oracle_lib.backward(inp, base, heads=heads)
    finals = []
    for S in (1, 2, 4, 8, 16):
        shape = base.with_(n_segments=S)
        got, g = _run(shape, dtype, inp, backward=True, use_dfinal=True)
        ref_s = dict(ref, seg_in=np.zeros((1, 1)))  # the segment states differ per S; y and final do not
        errs = compare_forward(got, ref_s, TOL[dtype], heads=heads)
        gerrs = compare_backward(g, gref, shape, TOL[dtype], heads=heads)
        finals.append(got["final_state"][:, heads[0]:heads[1]])
        print("long-131k S", S, errs, gerrs)
    for f in finals[1:]:  # invariant to the segment count up to bf16-path rounding
        assert np.linalg.norm(f - finals[0]) <= TOL[dtype] * np.linalg.norm(finals[0])


def test_packed_32k(oracle_lib):
    shape, dtype, seed = WORKLOADS["packed-32k"]
    inp = make_inputs(shape, seed, dtype)
    got, g = _run(shape, dtype, inp, backward=True)
    errs = compare_forward(got, oracle_lib.forward(inp, shape), TOL[dtype])
    gerrs = compare_backward(g, oracle_lib.backward(inp, shape, use_dfinal=False), shape, TOL[dtype])
    print("packed-32k", errs, gerrs)


def test_packed_32k_initial_state_and_sequence_finals(oracle_lib):
    shape, dtype, seed = WORKLOADS["packed-32k"]
    inp = make_inputs(shape, seed, dtype, init_states=True)
    r = ssd.SsdRunner(shape, dtype)
    t = to_dev(inp)
    y, fin, seg, sf = r.forward_varlen(t)
    g = r.backward(t, t["dy"], None, seg)
    torch.cuda.synchronize()
    got = {"y": np_(y).reshape(1, shape.seqlen, shape.nheads, shape.headdim), "final_state": np_(fin),
           "seg_in": np_(seg)}
    errs = compare_forward(got, oracle_lib.forward(inp, shape), TOL[dtype])
    fins = oracle_lib.seq_finals(inp, shape)
    errs["seq_finals"] = float(np.linalg.norm(np_(sf) - fins) / np.linalg.norm(fins))
    assert errs["seq_finals"] <= TOL[dtype]
    gerrs = compare_backward({k: np_(v) for k, v in g.items()}, oracle_lib.backward(inp, shape, use_dfinal=False),
                             shape, TOL[dtype])
    assert "dinit" in gerrs
    print("packed-32k init", errs, gerrs)


def test_mamba2_1b_gated_norm_forward_backward(oracle_lib):
    shape, dtype, seed = WORKLOADS["mamba2-1b-fwdbwd"]
    inp = make_inputs(shape, seed, dtype, gated_norm=True)
    r = ssd.SsdRunner(shape, dtype, gated_norm=True)
    t = to_dev(inp)
    y, fin, seg = r.forward(t)
    g = r.backward(t, t["dy"], None, seg)
    torch.cuda.synchronize()
    got = {"y": np_(y).reshape(shape.batch, shape.seqlen, shape.nheads, shape.headdim), "final_state": np_(fin),
           "seg_in": np_(seg)}
    errs = compare_forward(got, oracle_lib.forward(inp, shape, rows=[2]), TOL[dtype], rows=[2])
    gerrs = compare_backward({k: np_(v) for k, v in g.items()}, oracle_lib.backward(inp, shape, use_dfinal=False),
                             shape, TOL[dtype])
    print("mamba2-1b gated norm", errs, gerrs)


def test_long_131k_gated_norm_forward(oracle_lib):
    shape, dtype, seed = WORKLOADS["long-131k"]
    inp = make_inputs(shape, seed, dtype, gated_norm=True)
    heads = (0, shape.nheads // shape.ngroups)
    got, _ = _run_norm(shape, dtype, inp)
    errs = compare_forward(got, oracle_lib.forward(inp, shape, heads=heads), TOL[dtype], heads=heads)
    print("long-131k gated norm", errs)


def _run_norm(shape, dtype, inp):
    r = ssd.SsdRunner(shape, dtype, gated_norm=True)
    t = to_dev(inp)
    y, fin, seg = r.forward(t)
    torch.cuda.synchronize()
    out = {"y": np_(y).reshape(shape.batch, shape.seqlen, shape.nheads, shape.headdim), "final_state": np_(fin),
           "seg_in": np_(seg)}
    del r, t
    torch.cuda.empty_cache()
    return out, None

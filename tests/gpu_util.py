"""Helpers for the GPU parity tests: run libssd through its C ABI and compare
with the fp64 oracle by relative L2 error (= relative RMS, the criterion of
Megatron-LM PR #6808 "Add state-passing context parallelism for Mamba2",
Testing section)."""
from __future__ import annotations

import numpy as np
import torch

import mamba2_ssd_selective_gb300 as ssd

TOL = {"f32": 1e-4, "bf16": 1e-2}

# ddt_bias = sum over every token of ddt_raw.  In these bf16 parity cases (few
# tokens per head) the sum is only 0.26-0.40 times the root-sum-square of its
# terms, and rounding the post-conv activations to bf16, with every other step
# exact, already moves it by the relative error listed (the floor, pinned by
# tests/test_bf16_rounding_floor.py).  There the plain relative-L2 bound is
# max(1e-2, 1.5 x floor); everywhere else it is 1e-2 like every other gradient.
DDT_BIAS_FLOOR = {"packed-2048-q256": 1.42e-2, "packed-2x1024-q128": 1.45e-2, "forget-1024": 7.69e-3}


def ddt_bias_tol(case: str | None, tol: float) -> float:
    return max(tol, 1.5 * DDT_BIAS_FLOOR[case]) if case in DDT_BIAS_FLOOR else tol


def rel(a, b) -> float:
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


def to_dev(inp: dict) -> dict:
    return {k: (v.cuda() if torch.is_tensor(v) else v) for k, v in inp.items()}


def np_(t) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def gpu_forward(shape, dtype, inp, runner=None):
    r = runner or ssd.SsdRunner(shape, dtype, gated_norm=inp.get("z") is not None)
    t = to_dev(inp)
    y, fin, seg = r.forward(t)
    torch.cuda.synchronize()
    s = shape
    return {
        "y": np_(y).reshape(s.batch, s.seqlen, s.nheads, s.headdim),
        "final_state": np_(fin),
        "seg_in": np_(seg),
    }, (r, t, y, fin, seg)


def gpu_backward(shape, dtype, inp, use_dfinal=True, pass_seg=True):
    r = ssd.SsdRunner(shape, dtype, gated_norm=inp.get("z") is not None)
    t = to_dev(inp)
    y, fin, seg = r.forward(t)
    g = r.backward(t, t["dy"], t["dfinal"] if use_dfinal else None, seg if pass_seg else None)
    torch.cuda.synchronize()
    return {k: np_(v) for k, v in g.items()}


def compare_forward(got: dict, ref: dict, tol: float, heads=None, rows=None):
    h0, h1 = heads if heads else (0, got["y"].shape[2])
    rows = list(range(got["y"].shape[0])) if rows is None else rows
    errs = {
        "y": rel(got["y"][rows][:, :, h0:h1], ref["y"]),
        "final_state": rel(got["final_state"][rows][:, h0:h1], ref["final_state"]),
    }
    if ref["seg_in"].shape[1] > 1:
        errs["seg_in"] = rel(got["seg_in"][rows][:, :, h0:h1], ref["seg_in"])
    for k, e in errs.items():
        assert e <= tol, (k, e, errs)
    return errs


# reported, not asserted: ddt_bias's error against the root-sum-square of its
# per-token terms (the scale that per-term rounding produces), beside the plain
# relative L2 that is asserted like every other gradient's
REPORT_ONLY = {"ddt_bias_rss"}


def compare_backward(got: dict, ref: dict, shape, tol: float, rows=None, heads=None, floor_case=None):
    rows = list(range(shape.batch)) if rows is None else rows
    h0, h1 = heads if heads else (0, shape.nheads)
    ch = ref["channels"]
    errs = {
        "dxBC": rel(got["dxBC"][rows][..., ch], ref["dxBC"]),
        "ddt_raw": rel(got["ddt_raw"][rows][..., h0:h1], ref["ddt_raw"]),
    }
    if len(rows) == shape.batch:  # parameter grads sum over every row
        errs.update({
            "dconv_w": rel(got["dconv_w"][ch], ref["dconv_w"]),
            "dconv_b": rel(got["dconv_b"][ch], ref["dconv_b"]) if np.any(ref["dconv_b"]) else 0.0,
            "ddt_bias": rel(got["ddt_bias"][h0:h1], ref["ddt_bias"]),
            "ddt_bias_rss": float(np.linalg.norm(got["ddt_bias"][h0:h1] - ref["ddt_bias"])
                                  / np.linalg.norm(np.sqrt(np.sum(ref["ddt_raw"] ** 2, axis=(0, 1))))),
            "dA_log": rel(got["dA_log"][h0:h1], ref["dA_log"]),
            "dD": rel(got["dD"][h0:h1], ref["dD"]),
        })
    if ref.get("dinit") is not None:
        errs["dinit"] = rel(got["dinit"][rows][:, h0:h1], ref["dinit"])
    if ref.get("dz") is not None:
        P = shape.headdim
        errs["dz"] = rel(got["dz"][rows][..., h0 * P:h1 * P], ref["dz"])
        if len(rows) == shape.batch:
            errs["dnorm_weight"] = rel(got["dnorm_weight"][h0 * P:h1 * P], ref["dnorm_weight"])
    for k, e in errs.items():
        bound = ddt_bias_tol(floor_case, tol) if k == "ddt_bias" else tol
        assert k in REPORT_ONLY or e <= bound, (k, e, bound, errs)
    return errs

"""The rounding floor of ddt_bias in the bf16 parity cases (CPU only).

ddt_bias is a sum of ddt_raw over every token of a head.  In three of the bf16
parity cases (few tokens per head, packed sequences or heads that forget
within a token) the sum is small against the root-sum-square of its terms.
This pins what rounding the post-conv activations u to bf16 -- the storage of
every bf16 implementation of the mixer, with everything else exact in float64
-- does to ddt_bias there: the floors that tests/gpu_util.py scales its bound
for those cases from.  The per-token gradient ddt_raw itself stays within
3e-3, far inside the 1e-2 bound."""
from __future__ import annotations

import numpy as np
import pytest

from mamba2_ssd_selective_gb300.inputs import SsdShape, make_inputs
from tests.gpu_util import DDT_BIAS_FLOOR
from tests.ref_math import ssd_dt_bias_grad_f64

CASES = {
    "packed-2048-q256": (SsdShape(1, 2048, 4, 64, 128, 1, 256, 4), [256, 256, 1, 2, 3, 90, 160, 700, 580], 7, None),
    "packed-2x1024-q128": (SsdShape(2, 1024, 4, 64, 128, 1, 128, 2), [128, 5, 300, 77, 514], 7, None),
    "forget-1024": (SsdShape(1, 1024, 4, 64, 128, 1, 256, 2), [300, 1, 211, 512], 11, 2.0),
}


@pytest.mark.parametrize("case", sorted(CASES))
def test_bf16_storage_of_u_sets_the_ddt_bias_floor(case):
    shape, seq, seed, forget_bias = CASES[case]
    inp = make_inputs(shape, seed, "bf16", dfinal=True, seq_lengths=seq)
    if forget_bias is not None:
        inp["dt_bias"][:2] = forget_bias
    exact_b, exact_r = ssd_dt_bias_grad_f64(inp, shape, round_u=False)
    round_b, round_r = ssd_dt_bias_grad_f64(inp, shape, round_u=True)
    floor = np.linalg.norm(round_b - exact_b) / np.linalg.norm(exact_b)
    assert abs(floor - DDT_BIAS_FLOOR[case]) <= 0.05 * DDT_BIAS_FLOOR[case], floor
    assert np.linalg.norm(round_r - exact_r) / np.linalg.norm(exact_r) < 3e-3

"""ssd_forward_static: the forward for callers that cannot allocate device
memory (host frameworks that own every allocation, latency-bound loops where a
cudaMalloc would synchronise the device).  Its scratch is the library's fixed
device array, so the test checks, through the C ABI, that two calls in a row
(on different inputs, so stale scratch contents would show) give exactly what
the workspace-taking ssd_forward gives (the same kernels on the same inputs),
that the first call agrees with the fp64 oracle, that the array's status word
reads ok afterwards, and that a problem too large for the array is rejected
before launch.  Collected last on purpose."""
from __future__ import annotations

import pytest
import torch

import mamba2_ssd_selective_gb300 as ssd
from mamba2_ssd_selective_gb300.inputs import SsdShape, make_inputs
from tests.gpu_util import TOL, compare_forward, np_, to_dev

pytestmark = pytest.mark.gpu

SHAPE = SsdShape(1, 1024, 8, 64, 128, 1, 256, 4)


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mamba2_ssd_selective_gb300.build import build

    build()
    ssd.load()


def test_static_scratch_forward_matches_workspace_forward(oracle_lib):
    dims = ssd.make_dims(SHAPE, "bf16")
    assert ssd.ssd_workspace_size(dims, False) <= ssd.STATIC_SCRATCH_BYTES
    runner = ssd.SsdRunner(SHAPE, "bf16")
    for n, seed in enumerate((31, 32)):  # two calls in a row on different inputs
        inp = make_inputs(SHAPE, seed, "bf16", seq_lengths=[300, 2, 722])
        t = to_dev(inp)
        y_ref, fin_ref, seg_ref = runner.forward(t)
        y, fin, seg = runner.alloc_outputs()
        ssd.ssd_forward_static(dims, runner.inputs(t), y, fin, seg)
        torch.cuda.synchronize()
        assert torch.equal(y, y_ref) and torch.equal(fin, fin_ref) and torch.equal(seg, seg_ref)
        assert ssd.ssd_device_status(None) == 0
        if n == 0:
            got = {"y": np_(y).reshape(1, SHAPE.seqlen, SHAPE.nheads, SHAPE.headdim), "final_state": np_(fin),
                   "seg_in": np_(seg)}
            compare_forward(got, oracle_lib.forward(inp, SHAPE), TOL["bf16"])


def test_static_scratch_rejects_oversized_problem():
    big = SsdShape(4, 8192, 64, 64, 128, 1, 256, 8)
    dims = ssd.make_dims(big, "bf16")
    assert ssd.ssd_workspace_size(dims, False) > ssd.STATIC_SCRATCH_BYTES
    # aligned device pointers with the large shape's strides; the call is
    # rejected on its scratch size before anything reads them
    buf = torch.zeros(1 << 16, dtype=torch.bfloat16, device="cuda")
    p, Cd, HP, GN = buf.data_ptr(), big.conv_dim, big.nheads * big.headdim, big.ngroups * big.dstate
    inputs = ssd.SsdInputs(p, Cd, p + 2 * HP, Cd, p + 2 * (HP + GN), Cd, p, big.nheads, p, p, p, p, p, None)
    y, fin, seg = buf, None, None
    with pytest.raises(ssd.SsdError) as e:
        ssd.ssd_forward_static(dims, inputs, y, fin, seg)
    assert e.value.status == -6  # SSD_ERR_WORKSPACE

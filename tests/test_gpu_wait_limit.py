"""Failure detection on the GPU without a fault: the tensor-core kernels' waits
of one role on another are bounded.  With the wait limit set to 0, every wait
that is not already satisfied gives up; the kernels then drain the copies and
tensor-core work they started, free their tensor memory and return, and the
status word reports SSD_ERR_DEVICE_TIMEOUT.  Nothing is broken on purpose: the
pipelines are the real ones, only impatient.  Afterwards, with the default
limit restored, the same calls run clean and give bit-identical results to a
run made before (failure detection as in the Testing section of Megatron-LM PR
#6808 "Add state-passing context parallelism for Mamba2": the verdict is read
before anything is asserted, so no state is left half-done)."""
from __future__ import annotations

import pytest
import torch

import mamba2_ssd_selective_gb300 as ssd
from mamba2_ssd_selective_gb300.inputs import SsdShape, make_inputs
from tests.gpu_util import to_dev

pytestmark = pytest.mark.gpu

TIMEOUT = -9  # SSD_ERR_DEVICE_TIMEOUT


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mamba2_ssd_selective_gb300.build import build

    build()
    ssd.load()


def _fwd_bwd(r, t):
    y, fin, seg = r.forward(t)
    st_f = ssd.ssd_device_status(r.workspace)
    g = r.backward(t, t["dy"], t["dfinal"], seg)
    st_b = ssd.ssd_device_status(r.workspace)
    torch.cuda.synchronize()
    return (y.clone(), fin.clone(), seg.clone(), {k: v.clone() for k, v in g.items()}), st_f, st_b


def test_waits_that_give_up_are_reported_and_the_next_call_is_clean():
    shape = SsdShape(1, 2048, 16, 64, 128, 1, 256, 2)
    inp = make_inputs(shape, 21, "bf16", dfinal=True, seq_lengths=[900, 3, 1145])
    r = ssd.SsdRunner(shape, "bf16")
    t = to_dev(inp)
    ref, st_f, st_b = _fwd_bwd(r, t)
    assert (st_f, st_b) == (0, 0)
    prev = ssd.ssd_set_wait_limit_ns(0)
    try:
        _, st_f, st_b = _fwd_bwd(r, t)
    finally:
        ssd.ssd_set_wait_limit_ns(prev)
    assert prev == ssd.DEFAULT_WAIT_LIMIT_NS
    assert (st_f, st_b) == (TIMEOUT, TIMEOUT)
    again, st_f, st_b = _fwd_bwd(r, t)
    assert (st_f, st_b) == (0, 0)
    for a, b in zip(ref[:3], again[:3]):
        assert torch.equal(a, b)
    for k in ref[3]:
        assert torch.equal(ref[3][k], again[3][k]), k

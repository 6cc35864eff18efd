"""Failure detection on the GPU without a fault: a bounded device wait that is made to run out
(a barrier that nothing arrives on, a 1 ms budget) must give up, set the device status word,
be reported by qsa_check_device_status as QSA_ERR_TIMEOUT, and leave the context usable: the
status reads clean afterwards and the next call of the layer is correct."""
import numpy as np
import pytest
import torch

import oracle
from int8_kv_top_gb300 import qsa, synth
from tests.qsa_testutil import assert_close, to_dev

pytestmark = pytest.mark.gpu


def test_a_wait_that_runs_out_is_reported_and_the_context_survives():
    qsa.qsa_check_device_status()                       # clean to begin with
    qsa.qsa_debug_wait_probe(1_000_000)
    with pytest.raises(qsa.QSAError) as e:
        qsa.qsa_check_device_status()
    assert e.value.code == qsa.QSA_ERR_TIMEOUT
    qsa.qsa_check_device_status()                       # read and cleared
    # the next call of the layer runs and is right
    T, pos0 = 40, 0
    inp = synth.layer_inputs(T, T, seed=17)
    d = to_dev(inp)
    out = torch.empty((T, 24, 256), dtype=torch.float16, device="cuda")
    ws = torch.empty(qsa.qsa_flash_prefill_workspace_bytes(T, pos0, T), dtype=torch.uint8, device="cuda")
    qsa.qsa_flash_prefill(d["q"], d["kq"], d["vq"], d["ksc"], d["vsc"], T, T, pos0, None, out, ws)
    qsa.qsa_check_device_status()
    ref, *_ = oracle.prefill(inp, T, pos0)
    assert_close(out.float().cpu().numpy(), ref, "prefill after a timed-out wait")


def test_the_wait_gives_up_after_its_budget_not_before():
    # a 20 ms budget: the probe's stream is busy for at least that long
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record()
    qsa.qsa_debug_wait_probe(20_000_000)
    stop.record()
    with pytest.raises(qsa.QSAError):
        qsa.qsa_check_device_status()
    assert start.elapsed_time(stop) >= 19.0

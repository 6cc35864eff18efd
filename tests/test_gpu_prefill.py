"""GPU parity: qsa_flash_prefill (identity tokens) against the CPU oracle."""
import numpy as np
import pytest
import torch

import oracle
from int8_kv_top_gb300 import qsa, synth
from tests.qsa_testutil import assert_close, to_dev

pytestmark = pytest.mark.gpu


def run_prefill(inp, T, pos0, ids=None, params=None):
    d = to_dev(inp)
    n_cells = inp["kq"].shape[0]
    out = torch.full((T, 24, 256), float("nan"), dtype=torch.float16, device="cuda")
    ws = torch.empty(qsa.qsa_flash_prefill_workspace_bytes(T, pos0, n_cells, params), dtype=torch.uint8, device="cuda")
    qsa.qsa_flash_prefill(d["q"], d["kq"], d["vq"], d["ksc"], d["vsc"], n_cells, T, pos0, ids, out, ws, params)
    qsa.qsa_check_device_status()
    return out.float().cpu().numpy()


@pytest.mark.parametrize("T,pos0", [(96, 0), (1, 0), (2, 0), (31, 0), (32, 0), (33, 0), (64, 0), (65, 0),
                                    (60, 1984), (67, 1984), (5, 2046), (200, 0)])
def test_identity_prefill_matches_oracle(T, pos0):
    inp = synth.layer_inputs(T, pos0 + T, seed=5 + T + pos0)
    got = run_prefill(inp, T, pos0)
    ref, *_ = oracle.prefill(inp, T, pos0)
    assert_close(got, ref, f"T={T} pos0={pos0}")


def test_config1_t512_full_output():
    inp = synth.layer_inputs(512, 512, seed=5)
    got = run_prefill(inp, 512, 0)
    ref, *_ = oracle.prefill(inp, 512, 0)
    assert_close(got, ref, "T=512")


def test_config2_t1984_full_output():
    # the identity prefill at the benchmark's size (T=1984 at pos0=0, seed 5), every token
    inp = synth.layer_inputs(1984, 1984, seed=5)
    got = run_prefill(inp, 1984, 0)
    ref, *_ = oracle.prefill(inp, 1984, 0)
    assert_close(got, ref, "T=1984 all tokens")
    # and per token, so that one bad tile cannot hide in the global norm
    for t in (0, 1, 63, 64, 127, 128, 1000, 1983):
        assert_close(got[t], ref[t], f"T=1984 token {t}")


def test_identity_path_never_reads_ids():
    T, pos0 = 40, 1990                       # every n_kv <= 2030 <= 2051
    inp = synth.layer_inputs(T, pos0 + T, seed=9)
    poison = torch.full((T, 2, 2048), -1, dtype=torch.int32, device="cuda")
    a = run_prefill(inp, T, pos0, ids=poison)
    b = run_prefill(inp, T, pos0, ids=None)
    np.testing.assert_array_equal(a, b)


def test_edge_inputs():
    T, n = 70, 70
    inp = synth.layer_inputs(T, n, seed=12)
    inp["vq"][:] = 0                          # all-zero V -> zero output
    np.testing.assert_array_equal(run_prefill(inp, T, 0), 0.0)
    inp = synth.layer_inputs(T, n, seed=13)
    inp["q"][:] = 0                           # uniform softmax -> mean of V over the causal prefix
    ref, *_ = oracle.prefill(inp, T, 0)
    assert_close(run_prefill(inp, T, 0), ref, "q=0")
    inp = synth.layer_inputs(T, n, seed=14)
    inp["ksc"][::3] = -0.0                    # signed-zero scales are valid inputs
    inp["vsc"][1::5] = 0.0
    ref, *_ = oracle.prefill(inp, T, 0)
    assert_close(run_prefill(inp, T, 0), ref, "zero scales")


def test_dominant_logit_and_rescale():
    # a cell far into the sequence whose logit beats the rest by ~40 e-folds forces the
    # running-max rescale of the accumulated output
    T, n = 300, 300
    inp = synth.layer_inputs(T, n, seed=15)
    inp["q"][:, :, :] = np.abs(inp["q"]).astype(np.float16)
    inp["kq"][200] = 127
    inp["ksc"][200] = 0.02
    ref, *_ = oracle.prefill(inp, T, 0)
    assert_close(run_prefill(inp, T, 0), ref, "dominant")

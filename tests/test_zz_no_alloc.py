"""qsa_select_noalloc: the selection entry point for callers that cannot allocate device
memory (for example a runtime whose device memory is reserved up front by its own pool, or
a plugin interface that passes only inputs and outputs).  It must give exactly the ids that
qsa_select gives with a caller workspace, on consecutive calls that share its built-in
scratch, and refuse calls too large for that scratch.

This file is collected last on purpose, so a run that stops at the first failure has run
every other test before it."""
import numpy as np
import pytest
import torch

from int8_kv_top_gb300 import qsa, synth

pytestmark = pytest.mark.gpu


def select_both(N, P, seed):
    inp = synth.layer_inputs(N, P + N, seed=seed)
    d = {k: torch.from_numpy(v).cuda() for k, v in inp.items()}
    n_cells = P + N
    ids_ws = torch.full((N, 2, 2048), -7, dtype=torch.int32, device="cuda")
    ids_na = torch.full((N, 2, 2048), -9, dtype=torch.int32, device="cuda")
    ws = torch.empty(qsa.qsa_select_workspace_bytes(N, P, n_cells), dtype=torch.uint8, device="cuda")
    qsa.qsa_select(d["q"], d["kq"], d["ksc"], n_cells, N, P, ids_ws, ws)
    qsa.qsa_select_noalloc(d["q"], d["kq"], d["ksc"], n_cells, N, P, ids_na)
    qsa.qsa_check_device_status()
    return ids_ws.cpu().numpy(), ids_na.cpu().numpy(), P + np.arange(N) + 1 > 2051


def test_noalloc_select_matches_workspace_select_on_consecutive_calls():
    # a larger call first, then smaller ones: later calls must not see earlier leftovers.  The
    # 16-token call has more than 8 selected rows, so it takes the tensor-core score path, whose
    # tensor maps then point into the built-in scratch; the others take the few-row path.
    for N, P, seed in [(4, 8192, 31), (16, 3000, 33), (2, 3000, 32)]:
        ids_ws, ids_na, sel = select_both(N, P, seed)
        np.testing.assert_array_equal(ids_na[sel], ids_ws[sel])
        assert (np.diff(ids_na[sel], axis=-1) > 0).all()


def test_noalloc_select_rejects_calls_beyond_its_scratch():
    T, pos0 = 64, 30000
    q = torch.zeros((T, 24, 256), dtype=torch.float16, device="cuda")
    kq = torch.zeros((pos0 + T, 2, 256), dtype=torch.int8, device="cuda")
    ksc = torch.zeros((pos0 + T, 2, 4), dtype=torch.float16, device="cuda")
    ids = torch.zeros((T, 2, 2048), dtype=torch.int32, device="cuda")
    with pytest.raises(qsa.QSAError) as e:
        qsa.qsa_select_noalloc(q, kq, ksc, pos0 + T, T, pos0, ids)
    assert e.value.code == qsa.QSA_ERR_UNSUPPORTED and "scratch" in str(e.value)

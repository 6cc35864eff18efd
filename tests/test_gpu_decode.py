"""GPU parity: qsa_decode_partial + qsa_merge against the CPU oracle (identity cells and
oracle-selected ids; the end-to-end path with qsa_select is in test_gpu_select)."""
import numpy as np
import pytest
import torch

import oracle
from int8_kv_top_gb300 import qsa, synth
from tests.qsa_testutil import assert_close, to_dev

pytestmark = pytest.mark.gpu
CAP = qsa.chunk_cap_for()


def run_decode(inp, N, P, ids=None):
    d = to_dev(inp)
    n_cells = inp["kq"].shape[0]
    part = torch.full((N, CAP, 24, 258), float("nan"), device="cuda")
    nch = torch.zeros(N, dtype=torch.int32, device="cuda")
    xp = torch.full((N, 24, 256), float("nan"), device="cuda")
    qsa.qsa_decode_partial(d["q"], d["kq"], d["vq"], d["ksc"], d["vsc"], n_cells, N, P, ids, part, nch, CAP)
    qsa.qsa_merge(part, nch, N, CAP, xp)
    qsa.qsa_check_device_status()
    return part.cpu().numpy(), nch.cpu().numpy(), xp.cpu().numpy()


@pytest.mark.parametrize("N,P", [(1, 0), (3, 3), (1, 63), (2, 64), (1, 512), (4, 512), (4, 2047), (4, 2048),
                                 (8, 2050), (1, 8192), (4, 8192), (8, 3000)])
def test_decode_matches_oracle(N, P):
    inp = synth.layer_inputs(N, P + N, seed=100 + N + P)
    ref_part, ref_nc, ref_out, ref_direct, ref_ids = oracle.decode(inp, N, P)
    ids = torch.from_numpy(ref_ids).cuda() if P + N > 2051 else None
    part, nch, xp = run_decode(inp, N, P, ids)
    np.testing.assert_array_equal(nch, ref_nc)
    assert_close(xp, ref_out, f"merged N={N} P={P}")
    for t in range(N):
        c = ref_nc[t]
        # partial diagnostics: m to 1e-4 absolute, o and l through the merged output above
        np.testing.assert_allclose(part[t, :c, :, 256], ref_part[t, :c, :, 256], atol=1e-4, rtol=0)
        np.testing.assert_allclose(part[t, :c, :, 257], ref_part[t, :c, :, 257], rtol=1e-3)
        assert_close(part[t, :c, :, :256], ref_part[t, :c, :, :256], f"partial o t={t}")


def test_decode_flags_out_of_range_ids():
    N, P = 1, 3000
    inp = synth.layer_inputs(N, P + N, seed=7)
    ids = torch.arange(2048, dtype=torch.int32, device="cuda").reshape(1, 1, 2048).repeat(1, 2, 1).contiguous()
    ids[0, 1, 5] = 99999
    d = to_dev(inp)
    part = torch.zeros((N, CAP, 24, 258), device="cuda")
    nch = torch.zeros(N, dtype=torch.int32, device="cuda")
    qsa.qsa_decode_partial(d["q"], d["kq"], d["vq"], d["ksc"], d["vsc"], P + N, N, P, ids, part, nch, CAP)
    with pytest.raises(qsa.QSAError) as e:
        qsa.qsa_check_device_status()
    assert e.value.code == qsa.QSA_ERR_DEVICE

"""GPU parity: qsa_merge and qsa_prep_quantize against the CPU oracle."""
import numpy as np
import pytest
import torch

import oracle
from int8_kv_top_gb300 import qsa, synth
from tests.qsa_testutil import assert_close

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("n_chunks,cap", [([33], 33), ([1, 2, 17, 33], 33), ([32, 32, 32, 33], 33), ([5], 7),
                                          ([64, 65, 100, 3, 70], 100)])
def test_merge_matches_oracle(n_chunks, cap):
    part = synth.merge_partials(n_chunks, cap, seed=sum(n_chunks))
    ref = oracle.merge_f32(part, n_chunks)
    d_part = torch.from_numpy(part).cuda()
    d_nc = torch.tensor(n_chunks, dtype=torch.int32, device="cuda")
    xp = torch.full((len(n_chunks), 24, 256), float("nan"), device="cuda")
    qsa.qsa_merge(d_part, d_nc, len(n_chunks), cap, xp)
    qsa.qsa_check_device_status()
    assert_close(xp.cpu().numpy(), ref, "merge")


def test_merge_flags_bad_chunk_count():
    part = synth.merge_partials([2], 4, seed=1)
    d_part = torch.from_numpy(part).cuda()
    xp = torch.zeros((1, 24, 256), device="cuda")
    qsa.qsa_merge(d_part, torch.tensor([9], dtype=torch.int32, device="cuda"), 1, 4, xp)
    with pytest.raises(qsa.QSAError) as e:
        qsa.qsa_check_device_status()
    assert e.value.code == qsa.QSA_ERR_DEVICE
    assert torch.isnan(xp).all()
    qsa.qsa_check_device_status()  # the word was cleared


@pytest.mark.parametrize("n_cells,seed", [(1, 1), (777, 2), (4096, 3)])
def test_quantize_bit_exact(n_cells, seed):
    x = synth.fp16_rows(n_cells, seed=seed)
    x[0, 0, :64] = 0.0                      # an all-zero block
    x[-1, 1, 64:128] = -0.0                 # negative zeros
    ref_q, ref_s = oracle.quantize(x)
    d_x = torch.from_numpy(x).cuda()
    xq = torch.empty((n_cells, 2, 256), dtype=torch.int8, device="cuda")
    xsc = torch.empty((n_cells, 2, 4), dtype=torch.float16, device="cuda")
    qsa.qsa_prep_quantize(d_x, xq, xsc)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(xq.cpu().numpy(), ref_q)
    np.testing.assert_array_equal(xsc.cpu().numpy().view(np.uint16), ref_s.view(np.uint16))

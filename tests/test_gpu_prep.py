"""GPU parity: qsa_prep (RMS norm + rotary embedding of q and k, quantisation of the new
tokens' K and V rows into the int8 cache) against the oracle.

qcur and kcur are compared in float with the library's tolerance; the cache codes and scales
are integers decided by the quantiser, so they are compared bit-exactly with the oracle's
quantiser applied to the same fp16 rows (kcur as the kernel wrote it, v as given)."""
import numpy as np
import pytest
import torch

import oracle
from int8_kv_top_gb300 import qsa, synth
from tests.qsa_testutil import assert_close

pytestmark = pytest.mark.gpu


def run_prep(inp, T, pos0, n_cells, pos3=None, rope=None, with_kcur=True, seed=0):
    dev = {k: torch.from_numpy(v).cuda() for k, v in inp.items()}
    rng = np.random.default_rng(seed)
    # a cache with other cells already filled: they must stay as they are
    kq0 = rng.integers(-127, 128, size=(n_cells, 2, 256), dtype=np.int8)
    vq0 = rng.integers(-127, 128, size=(n_cells, 2, 256), dtype=np.int8)
    ksc0 = rng.uniform(0.005, 0.02, size=(n_cells, 2, 4)).astype(np.float16)
    vsc0 = rng.uniform(0.005, 0.02, size=(n_cells, 2, 4)).astype(np.float16)
    kq, vq = torch.from_numpy(kq0).cuda(), torch.from_numpy(vq0).cuda()
    ksc, vsc = torch.from_numpy(ksc0).cuda(), torch.from_numpy(vsc0).cuda()
    qcur = torch.full((T, 24, 256), float("nan"), dtype=torch.float16, device="cuda")
    kcur = torch.full((T, 2, 256), float("nan"), dtype=torch.float16, device="cuda") if with_kcur else None
    p3 = torch.from_numpy(pos3).cuda() if pos3 is not None else None
    qsa.qsa_prep(dev["q_raw"], dev["k_raw"], dev["v_raw"], dev["q_gamma"], dev["k_gamma"], T, pos0, n_cells, qcur, kcur,
                 kq, ksc, vq, vsc, pos3=p3, rope=rope)
    qsa.qsa_check_device_status()
    out = {"qcur": qcur.float().cpu().numpy(), "kq": kq.cpu().numpy(), "ksc": ksc.cpu().numpy(),
           "vq": vq.cpu().numpy(), "vsc": vsc.cpu().numpy()}
    if with_kcur:
        out["kcur16"] = kcur.cpu().numpy()
    out["before"] = (kq0, ksc0, vq0, vsc0)
    return out


def check(inp, T, pos0, n_cells, pos3=None, rope=None):
    base, rd, eps, sec = rope if rope else (10000.0, 256, 1e-6, (32, 48, 48))
    got = run_prep(inp, T, pos0, n_cells, pos3, rope, seed=T + pos0)
    ref_q, ref_k = oracle.prep(inp["q_raw"], inp["k_raw"], inp["q_gamma"], inp["k_gamma"], T, pos0, pos3=pos3,
                               base=base, rotary_dim=rd, eps=eps, sections=sec)
    assert_close(got["qcur"], ref_q, f"qcur T={T} pos0={pos0}")
    assert_close(got["kcur16"].astype(np.float64), ref_k, f"kcur T={T} pos0={pos0}")
    cells = slice(pos0, pos0 + T)
    exp_kq, exp_ksc = oracle.quantize(got["kcur16"])
    exp_vq, exp_vsc = oracle.quantize(inp["v_raw"])
    np.testing.assert_array_equal(got["kq"][cells], exp_kq)
    np.testing.assert_array_equal(got["ksc"][cells].view(np.uint16), exp_ksc.view(np.uint16))
    np.testing.assert_array_equal(got["vq"][cells], exp_vq)
    np.testing.assert_array_equal(got["vsc"][cells].view(np.uint16), exp_vsc.view(np.uint16))
    kq0, ksc0, vq0, vsc0 = got["before"]
    other = np.ones(n_cells, bool)
    other[cells] = False
    np.testing.assert_array_equal(got["kq"][other], kq0[other])
    np.testing.assert_array_equal(got["vsc"][other].view(np.uint16), vsc0[other].view(np.uint16))


@pytest.mark.parametrize("T,pos0", [(1, 0), (5, 2040), (64, 0), (37, 30000), (3, 65533)])
def test_prep_matches_oracle(T, pos0):
    inp = synth.prep_inputs(T, seed=70 + T)
    check(inp, T, pos0, pos0 + T + 3)


@pytest.mark.parametrize("rd", [16, 64, 128])
def test_prep_partial_rotary(rd):
    T, pos0 = 6, 777
    inp = synth.prep_inputs(T, seed=80 + rd)
    check(inp, T, pos0, pos0 + T, rope=(500000.0, rd, 1e-5, (rd // 8, rd // 8 * 3 // 2, rd // 2 - rd // 8 - rd // 8 * 3 // 2)))


def test_prep_mrope_positions():
    # an image-like block: temporal index fixed, height and width positions over a 4 x 5 grid
    T, pos0 = 20, 100
    inp = synth.prep_inputs(T, seed=90)
    hw = np.array([(100, 100 + i // 5, 100 + i % 5) for i in range(T)], np.int32)
    check(inp, T, pos0, pos0 + T, pos3=hw)


def test_prep_without_kcur_writes_the_same_cache():
    T, pos0 = 9, 50
    inp = synth.prep_inputs(T, seed=91)
    a = run_prep(inp, T, pos0, pos0 + T, seed=1)
    b = run_prep(inp, T, pos0, pos0 + T, with_kcur=False, seed=1)
    for k in ("qcur", "kq", "ksc", "vq", "vsc"):
        np.testing.assert_array_equal(a[k], b[k])


def test_prep_then_prefill_attends_over_the_new_cache():
    # the new tokens' cache rows and queries from qsa_prep feed qsa_flash_prefill; the result must
    # be the oracle's attention over the same fp16 queries and int8 cache
    T, pos0 = 48, 100
    n = pos0 + T
    inp = synth.prep_inputs(T, seed=92)
    hist = synth.layer_inputs(T, n, seed=93)
    dev = {k: torch.from_numpy(v).cuda() for k, v in inp.items()}
    kq, vq = torch.from_numpy(hist["kq"]).cuda(), torch.from_numpy(hist["vq"]).cuda()
    ksc, vsc = torch.from_numpy(hist["ksc"]).cuda(), torch.from_numpy(hist["vsc"]).cuda()
    qcur = torch.empty((T, 24, 256), dtype=torch.float16, device="cuda")
    qsa.qsa_prep(dev["q_raw"], dev["k_raw"], dev["v_raw"], dev["q_gamma"], dev["k_gamma"], T, pos0, n, qcur, None, kq,
                 ksc, vq, vsc)
    out = torch.empty((T, 24, 256), dtype=torch.float16, device="cuda")
    ws = torch.empty(qsa.qsa_flash_prefill_workspace_bytes(T, pos0, n), dtype=torch.uint8, device="cuda")
    qsa.qsa_flash_prefill(qcur, kq, vq, ksc, vsc, n, T, pos0, None, out, ws)
    qsa.qsa_check_device_status()
    layer = {"q": qcur.cpu().numpy(), "kq": kq.cpu().numpy(), "vq": vq.cpu().numpy(), "ksc": ksc.cpu().numpy(),
             "vsc": vsc.cpu().numpy()}
    ref, *_ = oracle.prefill(layer, T, pos0)
    assert_close(out.float().cpu().numpy(), ref, "prep -> prefill")

"""GPU parity: the output gate (out * sigmoid(gate), elementwise) in the prefill epilogues
(identity and gathered paths), the decode merge and the fused decode layer, against the
oracle's float64 attention times the oracle's gate."""
import numpy as np
import pytest
import torch

import oracle
from int8_kv_top_gb300 import qsa, synth
from tests.qsa_testutil import assert_close, to_dev

pytestmark = pytest.mark.gpu


def prefill_gated(inp, gate, T, pos0, params=None, ids=None, gated=True):
    d = to_dev(inp)
    n = inp["kq"].shape[0]
    topk = params[0] if params else 2048
    if ids is None and pos0 + T > (params[1] if params else 2051):
        ids = torch.empty((T, 2, topk), dtype=torch.int32, device="cuda")
        sws = torch.empty(max(16, qsa.qsa_select_workspace_bytes(T, pos0, n, params)), dtype=torch.uint8, device="cuda")
        qsa.qsa_select(d["q"], d["kq"], d["ksc"], n, T, pos0, ids, sws, params)
    out = torch.full((T, 24, 256), float("nan"), dtype=torch.float16, device="cuda")
    ws = torch.empty(qsa.qsa_flash_prefill_workspace_bytes(T, pos0, n, params), dtype=torch.uint8, device="cuda")
    g = torch.from_numpy(gate).cuda() if gated else None
    qsa.qsa_flash_prefill_gated(d["q"], d["kq"], d["vq"], d["ksc"], d["vsc"], n, T, pos0, ids, g, out, ws, params)
    qsa.qsa_check_device_status()
    return out.float().cpu().numpy()


@pytest.mark.parametrize("T,pos0,params", [(200, 0, None), (33, 0, None), (96, 1984, None),
                                           (40, 160, (40, 71, 1 / 16))])
def test_gated_prefill_matches_oracle(T, pos0, params):
    inp = synth.layer_inputs(T, pos0 + T, seed=40 + T + pos0)
    gate = synth.gate_input(T, seed=41 + T)
    topk, idmax, scale = params if params else (2048, 2051, 1 / 16)
    got = prefill_gated(inp, gate, T, pos0, params)
    ref, *_ = oracle.prefill(inp, T, pos0, topk=topk, identity_max=idmax, sm_scale=scale)
    assert_close(got, oracle.apply_gate(ref, gate), f"gated prefill T={T} pos0={pos0}")


def test_zero_gate_halves_the_prefill_output_exactly():
    # sigmoid(0) = 1/2, and halving is exact for fp16 values whose half is still a normal fp16
    # number (>= 2^-14); below that the gated value is the fp16 rounding of the half, within half
    # a subnormal step (2^-25)
    T, pos0 = 70, 0
    inp = synth.layer_inputs(T, T, seed=44)
    zero = np.zeros((T, 24, 256), np.float16)
    half = prefill_gated(inp, zero, T, pos0)
    full = prefill_gated(inp, zero, T, pos0, gated=False)
    normal = np.abs(full) >= 2.0 ** -13
    assert normal.mean() > 0.9
    np.testing.assert_array_equal(half[normal], full[normal] / 2)
    assert np.abs(half[~normal] - full[~normal] / 2).max() <= 2.0 ** -25


def test_gated_merge_matches_oracle():
    N, P = 4, 3000
    inp = synth.layer_inputs(N, P + N, seed=45)
    gate = synth.gate_input(N, seed=46)
    d = to_dev(inp)
    cap = qsa.chunk_cap_for()
    _, _, ref_out, _, ref_ids = oracle.decode(inp, N, P)
    ids = torch.from_numpy(ref_ids).cuda()
    part = torch.empty((N, cap, 24, 258), device="cuda")
    nch = torch.empty(N, dtype=torch.int32, device="cuda")
    xp = torch.full((N, 24, 256), float("nan"), device="cuda")
    qsa.qsa_decode_partial(d["q"], d["kq"], d["vq"], d["ksc"], d["vsc"], P + N, N, P, ids, part, nch, cap)
    qsa.qsa_merge_gated(part, nch, N, cap, torch.from_numpy(gate).cuda(), xp)
    qsa.qsa_check_device_status()
    assert_close(xp.cpu().numpy(), oracle.apply_gate(ref_out, gate), "gated merge")


@pytest.mark.parametrize("N,P", [(1, 8192), (4, 2048), (2, 300)])
def test_gated_decode_layer_matches_oracle(N, P):
    inp = synth.layer_inputs(N, P + N, seed=47 + N + P)
    gate = synth.gate_input(N, seed=48 + P)
    d = to_dev(inp)
    xp = torch.full((N, 24, 256), float("nan"), device="cuda")
    qsa.qsa_decode_layer(d["q"], d["kq"], d["vq"], d["ksc"], d["vsc"], P + N, N, P, None, xp,
                         gate=torch.from_numpy(gate).cuda())
    qsa.qsa_check_device_status()
    _, _, ref_out, _, _ = oracle.decode(inp, N, P)
    assert_close(xp.cpu().numpy(), oracle.apply_gate(ref_out, gate), f"gated decode layer N={N} P={P}")


def test_gated_batched_decode_matches_oracle():
    specs = [(2052, 2048, 4), (8193, 8192, 1), (300, 290, 3)]
    pieces = [synth.layer_inputs(nt, n, seed=60 + i) for i, (n, p0, nt) in enumerate(specs)]
    pool = {k: np.concatenate([pc[k] for pc in pieces], axis=0) for k in ("q", "kq", "vq", "ksc", "vsc")}
    seqs, c0, t0 = [], 0, 0
    for n, p0, nt in specs:
        seqs.append((c0, n, p0, t0))
        c0 += n
        t0 += nt
    seqs = np.array(seqs, dtype=np.int32)
    n_tok = pool["q"].shape[0]
    gate = synth.gate_input(n_tok, seed=61)
    d = to_dev(pool)
    xp = torch.full((n_tok, 24, 256), float("nan"), device="cuda")
    qsa.qsa_decode_layer_batched(d["q"], d["kq"], d["vq"], d["ksc"], d["vsc"], c0, torch.from_numpy(seqs).cuda(),
                                 len(seqs), n_tok, 8193, None, xp, gate=torch.from_numpy(gate).cuda())
    qsa.qsa_check_device_status()
    ref_out, _ = oracle.decode_batch(pool, seqs)
    assert_close(xp.cpu().numpy(), oracle.apply_gate(ref_out, gate), "gated batched decode")

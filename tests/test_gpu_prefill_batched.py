"""GPU parity: qsa_flash_prefill_batched (many sequences per call: identity tokens on the tensor
cores over per-sequence mirrors, selected tokens through the cluster selection kernel) against
the oracle's per-sequence prefill: ids bit-exact, fp16 outputs within the float tolerance."""
import numpy as np
import pytest
import torch

import oracle
from int8_kv_top_gb300 import qsa, synth
from tests.qsa_testutil import assert_close, to_dev

pytestmark = pytest.mark.gpu


def make_pool(specs, seed0, gap=0):
    """specs: (n_cells, pos0, tokens) per sequence -> pool inputs and the seqs table.  `gap`
    unused cells with NaN scales sit before every sequence: nothing may read them."""
    pieces = [synth.layer_inputs(max(nt, 1), n, seed=seed0 + i) for i, (n, p0, nt) in enumerate(specs)]
    parts = {k: [] for k in ("kq", "vq", "ksc", "vsc")}
    seqs, c0, t0 = [], 0, 0
    for (n, p0, nt), pc in zip(specs, pieces):
        if gap:
            parts["kq"].append(np.full((gap, 2, 256), 127, np.int8))
            parts["vq"].append(np.full((gap, 2, 256), -127, np.int8))
            parts["ksc"].append(np.full((gap, 2, 4), np.nan, np.float16))
            parts["vsc"].append(np.full((gap, 2, 4), np.nan, np.float16))
            c0 += gap
        for k in parts:
            parts[k].append(pc[k])
        seqs.append((c0, n, p0, t0))
        c0 += n
        t0 += nt
    pool = {k: np.concatenate(v, axis=0) for k, v in parts.items()}
    pool["q"] = np.concatenate([pc["q"][:nt] for pc, (n, p0, nt) in zip(pieces, specs)], axis=0)
    return pool, np.array(seqs, dtype=np.int32)


def run(pool, seqs, max_n_kv, params=None, gate=None):
    d = to_dev(pool)
    n_tok = pool["q"].shape[0]
    topk = params[0] if params else 2048
    ids = torch.full((n_tok, 2, topk), -7, dtype=torch.int32, device="cuda")
    out = torch.full((n_tok, 24, 256), float("nan"), dtype=torch.float16, device="cuda")
    ws = torch.empty(qsa.qsa_flash_prefill_batched_workspace_bytes(len(seqs), n_tok, max_n_kv, params),
                     dtype=torch.uint8, device="cuda")
    g = torch.from_numpy(gate).cuda() if gate is not None else None
    qsa.qsa_flash_prefill_batched(d["q"], d["kq"], d["vq"], d["ksc"], d["vsc"], pool["kq"].shape[0],
                                  torch.from_numpy(seqs).cuda(), len(seqs), n_tok, max_n_kv, ids, out, ws, params,
                                  gate=g)
    return ids, out


def check(pool, seqs, max_n_kv, params=None, gate=None):
    topk, idmax, scale = params if params else (2048, 2051, 1 / 16)
    ids, out = run(pool, seqs, max_n_kv, params, gate)
    qsa.qsa_check_device_status()
    ids, out = ids.cpu().numpy(), out.float().cpu().numpy()
    ref_out, ref_ids = oracle.prefill_batch(pool, seqs, topk=topk, identity_max=idmax, sm_scale=scale)
    if gate is not None:
        ref_out = oracle.apply_gate(ref_out, gate)
    sel = ref_ids[:, :, 0] >= 0
    np.testing.assert_array_equal(ids[sel], ref_ids[sel])
    assert (ids[~sel] == -7).all(), "rows of identity tokens must not be written"
    assert_close(out, ref_out, "batched prefill")
    n_tok = out.shape[0]
    for s, (c0, n, p0, t0) in enumerate(seqs):
        t1 = seqs[s + 1][3] if s + 1 < len(seqs) else n_tok
        if t1 > t0:
            assert_close(out[t0:t1], ref_out[t0:t1], f"sequence {s} (n_cells {n}, pos0 {p0}, {t1 - t0} tokens)")
    return ids, out


def test_batched_prefill_identity_prompts():
    # short prompts only (every token at or under the threshold): one dense launch over the
    # work list; ragged tiles, a one-token prompt, a prompt up to exactly 2051 cells
    specs = [(100, 0, 100), (65, 0, 65), (1, 0, 1), (700, 600, 100), (300, 0, 300), (2051, 1900, 151), (33, 0, 33)]
    pool, seqs = make_pool(specs, seed0=2000, gap=5)
    check(pool, seqs, max_n_kv=2051)


def test_batched_prefill_mixed_with_selection():
    # identity, boundary (2051 / 2052 inside one sequence) and selected tokens in one call, with
    # unused NaN-scaled cells between the sequences and a sequence with no tokens
    specs = [(2100, 2000, 100), (5000, 4990, 10), (128, 0, 128), (40, 40, 0), (3000, 2990, 10), (70, 0, 70)]
    pool, seqs = make_pool(specs, seed0=2100, gap=3)
    check(pool, seqs, max_n_kv=5000)


def test_batched_prefill_small_budgets():
    specs = [(200, 60, 30), (90, 0, 90), (150, 140, 10), (72, 0, 72)]
    pool, seqs = make_pool(specs, seed0=2200)
    check(pool, seqs, max_n_kv=200, params=(40, 71, 1 / 16))


def test_batched_prefill_gated():
    specs = [(300, 0, 300), (2060, 2040, 20), (64, 0, 64)]
    pool, seqs = make_pool(specs, seed0=2300)
    gate = synth.gate_input(pool["q"].shape[0], seed=2301)
    check(pool, seqs, max_n_kv=2060, gate=gate)


def test_batched_identity_equals_the_single_sequence_call_bit_for_bit():
    # the same rows through the same dense kernel: the per-sequence mirror and the work list
    # change where the rows come from, not the arithmetic
    T, pos0 = 200, 500
    inp = synth.layer_inputs(T, pos0 + T, seed=2400)
    pool = dict(inp)
    seqs = np.array([(0, pos0 + T, pos0, 0)], dtype=np.int32)
    _, out_b = run(pool, seqs, max_n_kv=pos0 + T)
    d = to_dev(inp)
    out_s = torch.empty((T, 24, 256), dtype=torch.float16, device="cuda")
    ws = torch.empty(qsa.qsa_flash_prefill_workspace_bytes(T, pos0, pos0 + T), dtype=torch.uint8, device="cuda")
    qsa.qsa_flash_prefill(d["q"], d["kq"], d["vq"], d["ksc"], d["vsc"], pos0 + T, T, pos0, None, out_s, ws)
    qsa.qsa_check_device_status()
    np.testing.assert_array_equal(out_b.cpu().numpy().view(np.uint16), out_s.cpu().numpy().view(np.uint16))


def test_batched_prefill_many_short_prompts():
    # continuous batching: 40 prompts of 1 .. 300 tokens, some with a cached prefix
    rng = np.random.default_rng(9)
    specs = []
    for _ in range(40):
        T = int(rng.integers(1, 300))
        p0 = int(rng.integers(0, 400)) if rng.random() < 0.5 else 0
        specs.append((p0 + T, p0, T))
    pool, seqs = make_pool(specs, seed0=2500)
    check(pool, seqs, max_n_kv=max(p0 + T for _, p0, T in specs))


def test_batched_prefill_flags_a_bad_sequence_and_keeps_the_rest():
    specs = [(300, 0, 300), (200, 100, 50)]
    pool, seqs = make_pool(specs, seed0=2600)
    bad = seqs.copy()
    bad[1, 2] = 190                    # pos0 + 50 tokens > 200 cells: breaks the cache contract
    ids, out = run(pool, bad, max_n_kv=300)
    with pytest.raises(qsa.QSAError) as e:
        qsa.qsa_check_device_status()
    assert e.value.code == qsa.QSA_ERR_DEVICE
    out = out.float().cpu().numpy()
    assert np.isnan(out[300:]).all()   # the bad sequence's rows are not written
    good = dict(pool)
    good["q"] = pool["q"][:300]        # the good sequence's own tokens only
    ref_out, _ = oracle.prefill_batch(good, seqs[:1], topk=2048)
    assert_close(out[:300], ref_out, "the good sequence")


def test_batched_prefill_long_context_next_to_short_prompts():
    # a 100,004-cell sequence (selection in 16-CTA clusters) beside short prompts and a boundary one
    specs = [(100004, 100000, 4), (200, 0, 200), (2060, 2040, 20)]
    pool, seqs = make_pool(specs, seed0=2700, gap=2)
    check(pool, seqs, max_n_kv=100004)

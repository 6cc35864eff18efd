"""GPU parity: qsa_decode_layer (selection, attention and merge in one launch) and
qsa_decode_layer_batched (many sequences per launch) against the CPU oracle: ids bit-exact
against the exact ranking, merged outputs within the float tolerance."""
import numpy as np
import pytest
import torch

import oracle
from int8_kv_top_gb300 import qsa, synth
from tests.qsa_testutil import assert_close, to_dev

pytestmark = pytest.mark.gpu


def run_layer(inp, N, P, params=None, with_ids=True):
    d = to_dev(inp)
    n_cells = inp["kq"].shape[0]
    topk = params[0] if params else 2048
    ids = torch.full((N, 2, topk), -7, dtype=torch.int32, device="cuda") if with_ids else None
    xp = torch.full((N, 24, 256), float("nan"), device="cuda")
    qsa.qsa_decode_layer(d["q"], d["kq"], d["vq"], d["ksc"], d["vsc"], n_cells, N, P, ids, xp, params)
    qsa.qsa_check_device_status()
    return (ids.cpu().numpy() if with_ids else None), xp.cpu().numpy()


def check(inp, N, P, params=None):
    topk, idmax, scale = params if params else (2048, 2051, 1 / 16)
    ids, xp = run_layer(inp, N, P, params)
    _, ref_nc, ref_out, _, ref_ids = oracle.decode(inp, N, P, topk=topk, identity_max=idmax, sm_scale=scale)
    sel = (P + np.arange(N) + 1) > idmax
    np.testing.assert_array_equal(ids[sel], ref_ids[sel])
    assert (ids[~sel] == -7).all(), "rows of identity tokens must not be written"
    assert_close(xp, ref_out, f"decode layer N={N} P={P}")
    for t in range(N):
        assert_close(xp[t], ref_out[t], f"decode layer N={N} P={P} token {t}")


# single tokens and small batches at the pages' positions and the budget boundary; one or two
# tokens take clusters of 16 CTAs per (token, group), larger N clusters of 8 (as many as the GPU
# holds at once in one wave)
@pytest.mark.parametrize("N,P", [(1, 0), (3, 3), (1, 63), (2, 64), (1, 512), (4, 512), (1, 2048), (4, 2047),
                                 (4, 2048), (8, 2050), (1, 8192), (4, 8192), (8, 3000), (1, 30000)])
def test_decode_layer_matches_oracle(N, P):
    inp = synth.layer_inputs(N, P + N, seed=300 + N + P)
    check(inp, N, P)


@pytest.mark.parametrize("N,P,params", [(5, 160, (40, 71, 1 / 16)), (2, 700, (1000, 1500, 0.05)),
                                        (3, 100, (1, 50, 1 / 16))])
def test_decode_layer_small_budgets(N, P, params):
    inp = synth.layer_inputs(N, P + N, seed=7 * N + P)
    check(inp, N, P, params)


@pytest.mark.parametrize("N,P", [(2, 65534), (2, 100000), (1, 131071)])
def test_decode_layer_long_context(N, P):
    # long caches: up to 8,192 cells per CTA of a 16-CTA cluster, 131,072 cells in all
    inp = synth.layer_inputs(N, P + N, seed=77 + P)
    check(inp, N, P)


def test_decode_layer_exact_ties_go_to_the_lower_index():
    # identical K rows: every score ties exactly, every cell is a candidate, and the kept set
    # must be the lowest 2048 indices
    N, P = 2, 3000
    inp = synth.layer_inputs(N, P + N, seed=3)
    inp["kq"][:] = inp["kq"][0]
    inp["ksc"][:] = inp["ksc"][0]
    ids, xp = run_layer(inp, N, P)
    np.testing.assert_array_equal(ids, np.broadcast_to(np.arange(2048, dtype=np.int32), ids.shape))
    _, _, ref_out, _, _ = oracle.decode(inp, N, P)
    assert_close(xp, ref_out, "ties")


def test_decode_layer_near_ties_from_duplicates():
    N, P = 3, 5000
    inp = synth.layer_inputs(N, P + N, seed=21)
    src = np.arange(0, 5000, 5)
    inp["kq"][src + 2] = inp["kq"][src]
    inp["ksc"][src + 2] = inp["ksc"][src]
    check(inp, N, P)


def test_decode_layer_without_ids_and_against_the_three_call_path():
    N, P = 1, 8192
    inp = synth.layer_inputs(N, P + N, seed=205)
    _, xp_noids = run_layer(inp, N, P, with_ids=False)
    ids, xp = run_layer(inp, N, P)
    np.testing.assert_array_equal(xp_noids, xp)
    d = to_dev(inp)
    cap = qsa.chunk_cap_for()
    ids3 = torch.empty((N, 2, 2048), dtype=torch.int32, device="cuda")
    ws = torch.empty(qsa.qsa_select_workspace_bytes(N, P, P + N), dtype=torch.uint8, device="cuda")
    part = torch.empty((N, cap, 24, 258), device="cuda")
    nch = torch.empty(N, dtype=torch.int32, device="cuda")
    xp3 = torch.empty((N, 24, 256), device="cuda")
    qsa.qsa_select(d["q"], d["kq"], d["ksc"], P + N, N, P, ids3, ws)
    qsa.qsa_decode_partial(d["q"], d["kq"], d["vq"], d["ksc"], d["vsc"], P + N, N, P, ids3, part, nch, cap)
    qsa.qsa_merge(part, nch, N, cap, xp3)
    qsa.qsa_check_device_status()
    np.testing.assert_array_equal(ids, ids3.cpu().numpy())
    assert_close(xp, xp3.cpu().numpy(), "fused vs three calls")


def make_batch(specs, seed0=900):
    """specs: (n_cells, pos0, tokens) per sequence -> pool inputs and the seqs table."""
    pieces = [synth.layer_inputs(nt, n, seed=seed0 + i) for i, (n, p0, nt) in enumerate(specs)]
    pool = {k: np.concatenate([pc[k] for pc in pieces], axis=0) for k in ("q", "kq", "vq", "ksc", "vsc")}
    seqs, c0, t0 = [], 0, 0
    for n, p0, nt in specs:
        seqs.append((c0, n, p0, t0))
        c0 += n
        t0 += nt
    return pool, np.array(seqs, dtype=np.int32)


def run_batched(pool, seqs, max_n_kv, params=None):
    d = to_dev(pool)
    n_tok = pool["q"].shape[0]
    topk = params[0] if params else 2048
    ids = torch.full((n_tok, 2, topk), -7, dtype=torch.int32, device="cuda")
    xp = torch.full((n_tok, 24, 256), float("nan"), device="cuda")
    st = torch.from_numpy(seqs).cuda()
    qsa.qsa_decode_layer_batched(d["q"], d["kq"], d["vq"], d["ksc"], d["vsc"], pool["kq"].shape[0], st, len(seqs),
                                 n_tok, max_n_kv, ids, xp, params)
    return ids, xp


def test_decode_layer_batched_mixed_sequences():
    # identity-only, boundary and selected sequences of different lengths in one launch
    specs = [(513, 512, 1), (2052, 2048, 4), (8193, 8192, 1), (3008, 3000, 8), (65, 63, 2), (20000, 19990, 3)]
    pool, seqs = make_batch(specs)
    ids, xp = run_batched(pool, seqs, max_n_kv=20000)
    qsa.qsa_check_device_status()
    ref_out, ref_ids = oracle.decode_batch(pool, seqs)
    ids = ids.cpu().numpy()
    sel = ref_ids[:, :, 0] >= 0
    np.testing.assert_array_equal(ids[sel], ref_ids[sel])
    assert (ids[~sel] == -7).all()
    assert_close(xp.cpu().numpy(), ref_out, "batched decode")


def test_decode_layer_batched_many_single_token_sequences():
    # 48 sequences of one token each (continuous batching), 16-CTA clusters forced by max_n_kv
    rng = np.random.default_rng(5)
    specs = [(int(p) + 1, int(p), 1) for p in rng.integers(1, 12000, size=48)]
    pool, seqs = make_batch(specs, seed0=1500)
    ids, xp = run_batched(pool, seqs, max_n_kv=40000)
    qsa.qsa_check_device_status()
    ref_out, ref_ids = oracle.decode_batch(pool, seqs)
    ids = ids.cpu().numpy()
    sel = ref_ids[:, :, 0] >= 0
    np.testing.assert_array_equal(ids[sel], ref_ids[sel])
    assert_close(xp.cpu().numpy(), ref_out, "batched decode, 48 sequences")


def test_decode_layer_batched_flags_a_bad_sequence_and_keeps_the_rest():
    specs = [(600, 590, 2), (700, 650, 3)]
    pool, seqs = make_batch(specs, seed0=1700)
    bad = seqs.copy()
    bad[1, 2] = 699                    # pos0 + 3 tokens > 700 cells: breaks the cache contract
    ids, xp = run_batched(pool, bad, max_n_kv=800)
    with pytest.raises(qsa.QSAError) as e:
        qsa.qsa_check_device_status()
    assert e.value.code == qsa.QSA_ERR_DEVICE
    xp = xp.cpu().numpy()
    assert np.isnan(xp[2:]).all()      # the bad sequence's rows are not written
    first = {"q": pool["q"][:2]}
    first.update({k: pool[k][:600] for k in ("kq", "vq", "ksc", "vsc")})
    _, _, ref_out, _, _ = oracle.decode(first, 2, 590)
    assert_close(xp[:2], ref_out, "the good sequence")


def test_decode_layer_batched_four_cta_clusters():
    # 16 single-token sequences over caches of at most 32,768 cells: the launch takes clusters of 4
    # CTAs (8,192 cells each); one sequence sits exactly at that limit
    rng = np.random.default_rng(11)
    specs = [(32768, 32767, 1)] + [(int(p) + 1, int(p), 1) for p in rng.integers(2100, 20000, size=15)]
    pool, seqs = make_batch(specs, seed0=1900)
    ids, xp = run_batched(pool, seqs, max_n_kv=32768)
    qsa.qsa_check_device_status()
    ref_out, ref_ids = oracle.decode_batch(pool, seqs)
    ids = ids.cpu().numpy()
    sel = ref_ids[:, :, 0] >= 0
    np.testing.assert_array_equal(ids[sel], ref_ids[sel])
    assert_close(xp.cpu().numpy(), ref_out, "batched decode, clusters of 4")


def test_decode_layer_batched_two_cta_clusters():
    # 64 single-token sequences over caches of at most 16,384 cells: the launch takes clusters of 2
    # CTAs (8,192 cells each); one sequence sits exactly at that limit
    rng = np.random.default_rng(12)
    specs = [(16384, 16383, 1)] + [(int(p) + 1, int(p), 1) for p in rng.integers(2100, 16000, size=63)]
    pool, seqs = make_batch(specs, seed0=2100)
    ids, xp = run_batched(pool, seqs, max_n_kv=16384)
    qsa.qsa_check_device_status()
    ref_out, ref_ids = oracle.decode_batch(pool, seqs)
    ids = ids.cpu().numpy()
    sel = ref_ids[:, :, 0] >= 0
    np.testing.assert_array_equal(ids[sel], ref_ids[sel])
    assert_close(xp.cpu().numpy(), ref_out, "batched decode, clusters of 2")

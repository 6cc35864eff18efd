"""GPU parity: qsa_select (ids bit-exact against the oracle's exact ranking), the gathered
prefill path, and the end-to-end decode step (select -> partial -> merge)."""
import numpy as np
import pytest
import torch

import oracle
from int8_kv_top_gb300 import qsa, synth
from tests.qsa_testutil import assert_close, to_dev

pytestmark = pytest.mark.gpu


def gpu_select_prefill(inp, T, pos0, params=None, poison=True):
    d = to_dev(inp)
    n_cells = inp["kq"].shape[0]
    topk = params[0] if params else 2048
    ids = torch.full((T, 2, topk), -7 if poison else 0, dtype=torch.int32, device="cuda")
    nbytes = qsa.qsa_select_workspace_bytes(T, pos0, n_cells, params)
    ws = torch.empty(max(nbytes, 16), dtype=torch.uint8, device="cuda") if nbytes else None
    qsa.qsa_select(d["q"], d["kq"], d["ksc"], n_cells, T, pos0, ids, ws, params)
    out = torch.full((T, 24, 256), float("nan"), dtype=torch.float16, device="cuda")
    pb = qsa.qsa_flash_prefill_workspace_bytes(T, pos0, n_cells, params)
    pws = torch.empty(max(pb, 16), dtype=torch.uint8, device="cuda") if pb else None
    qsa.qsa_flash_prefill(d["q"], d["kq"], d["vq"], d["ksc"], d["vsc"], n_cells, T, pos0, ids, out, pws, params)
    qsa.qsa_check_device_status()
    return ids.cpu().numpy(), out.float().cpu().numpy()


def check_ids(ids_gpu, ids_ref, T, pos0, idmax):
    sel = (pos0 + np.arange(T) + 1) > idmax
    np.testing.assert_array_equal(ids_gpu[sel], ids_ref[sel])


@pytest.mark.parametrize("T,pos0,params", [
    (40, 160, (40, 71, 1 / 16)),       # every token selected, topk not a multiple of 128
    (30, 50, (40, 71, 1 / 16)),        # mixed window: tokens 0..20 identity, the rest selected
    (12, 400, (256, 300, 1 / 16)),     # two full gather tiles
    (8, 2050, None),                   # default budget boundary: n_kv 2051 identity, 2052 selected
    (96, 1984, None),                  # mixed-budget window at pos0 = 1984
    (32, 2050, None),
    (10, 2050, None),                  # 9 selected rows: the smallest call on the score GEMM path
    (5, 160, (40, 71, 1 / 16)),        # few-row path (histogram-seeded top-k) with a small budget
])
def test_select_and_prefill_small(T, pos0, params):
    inp = synth.layer_inputs(T, pos0 + T, seed=T * 7 + pos0)
    topk, idmax, scale = params if params else (2048, 2051, 1 / 16)
    ids, out = gpu_select_prefill(inp, T, pos0, params)
    ref_out, ref_ids, _, _ = oracle.prefill(inp, T, pos0, topk=topk, identity_max=idmax, sm_scale=scale)
    check_ids(ids, ref_ids, T, pos0, idmax)
    assert_close(out, ref_out, f"T={T} pos0={pos0}")


def test_config3_reduced_all_tokens():
    T, pos0 = 48, 30000
    inp = synth.layer_inputs(T, pos0 + T, seed=5)
    ids, out = gpu_select_prefill(inp, T, pos0)
    ref_out, ref_ids, _, differs = oracle.prefill(inp, T, pos0, f64_check=True)
    np.testing.assert_array_equal(ids, ref_ids)
    assert_close(out, ref_out, "T=48 pos0=30000")


def test_config3_full_size_every_row():
    # the selected prefill at the benchmark's size (T=1984 at pos0=30000 over 31,984 cells,
    # seed 5): all 3,968 (token, group) id rows bit-exact against the oracle's exact ranking,
    # and every token's output within tolerance
    T, pos0 = 1984, 30000
    inp = synth.layer_inputs(T, pos0 + T, seed=5)
    ids, out = gpu_select_prefill(inp, T, pos0)
    ref_out, ref_ids, n_set, _ = oracle.prefill(inp, T, pos0)
    assert (n_set == 2048).all()
    bad = np.nonzero((ids != ref_ids).any(axis=-1))
    assert len(bad[0]) == 0, f"{len(bad[0])} of {T * 2} id rows differ, first (token, group): {bad[0][0]}, {bad[1][0]}"
    assert_close(out, ref_out, "config 3 all tokens")
    for t in (0, 1, 127, 128, 1000, 1983):
        assert_close(out[t], ref_out[t], f"config 3 token {t}")
    # how often a float64 ranking of the same scores would pick a different set: those rows
    # are the ones only the exact re-ranking gets right (diagnostic, on a sample of tokens)
    toks = np.arange(0, T, 31, dtype=np.int32)
    _, ids64, _, differs = oracle.prefill(inp, T, pos0, toks=toks, f64_check=True)
    np.testing.assert_array_equal(ids[toks], ids64)
    print(f"config 3: {int(differs.sum())} of {differs.size} sampled rows rank differently in float64")


def test_exact_ties_resolve_to_lower_index():
    # every cell identical: all scores tie exactly; the band holds all cells (the large-band path)
    T, pos0 = 3, 2100
    inp = synth.layer_inputs(T, pos0 + T, seed=3)
    inp["kq"][:] = inp["kq"][0]
    inp["ksc"][:] = inp["ksc"][0]
    ids, out = gpu_select_prefill(inp, T, pos0)
    expect = np.broadcast_to(np.arange(2048, dtype=np.int32), ids.shape)
    np.testing.assert_array_equal(ids, expect)


def test_near_ties_from_duplicates():
    # a few duplicated rows scattered through the cache: equal exact scores straddle the cut
    T, pos0 = 4, 3000
    inp = synth.layer_inputs(T, pos0 + T, seed=21)
    src = np.arange(0, 3000, 7)
    inp["kq"][src + 3] = inp["kq"][src]
    inp["ksc"][src + 3] = inp["ksc"][src]
    ids, out = gpu_select_prefill(inp, T, pos0)
    ref_out, ref_ids, _, _ = oracle.prefill(inp, T, pos0)
    np.testing.assert_array_equal(ids, ref_ids)
    assert_close(out, ref_out, "duplicates")


@pytest.mark.parametrize("N,P", [(4, 2048), (1, 8192), (4, 8192), (8, 3000), (2, 2050)])
def test_decode_end_to_end_with_select(N, P):
    inp = synth.layer_inputs(N, P + N, seed=200 + N + P)
    d = to_dev(inp)
    n_cells = P + N
    cap = qsa.chunk_cap_for()
    ids = torch.full((N, 2, 2048), -7, dtype=torch.int32, device="cuda")
    nbytes = qsa.qsa_select_workspace_bytes(N, P, n_cells)
    ws = torch.empty(max(nbytes, 16), dtype=torch.uint8, device="cuda")
    part = torch.full((N, cap, 24, 258), float("nan"), device="cuda")
    nch = torch.zeros(N, dtype=torch.int32, device="cuda")
    xp = torch.full((N, 24, 256), float("nan"), device="cuda")
    qsa.qsa_select(d["q"], d["kq"], d["ksc"], n_cells, N, P, ids, ws)
    qsa.qsa_decode_partial(d["q"], d["kq"], d["vq"], d["ksc"], d["vsc"], n_cells, N, P, ids, part, nch, cap)
    qsa.qsa_merge(part, nch, N, cap, xp)
    qsa.qsa_check_device_status()
    _, ref_nc, ref_out, _, ref_ids = oracle.decode(inp, N, P)
    check_ids(ids.cpu().numpy(), ref_ids, N, P, 2051)
    np.testing.assert_array_equal(nch.cpu().numpy(), ref_nc)
    assert_close(xp.cpu().numpy(), ref_out, f"decode N={N} P={P}")


# ---- the score-GEMM path (more than 8 selected rows) on tied and structured caches

def test_gemm_path_exact_ties_resolve_to_lower_index():
    # every cell identical: all scores tie exactly, the band holds every cell (the top-k's
    # large-band exact radix select)
    T, pos0 = 16, 5000
    inp = synth.layer_inputs(T, pos0 + T, seed=4)
    inp["kq"][:] = inp["kq"][0]
    inp["ksc"][:] = inp["ksc"][0]
    ids, out = gpu_select_prefill(inp, T, pos0)
    np.testing.assert_array_equal(ids, np.broadcast_to(np.arange(2048, dtype=np.int32), ids.shape))


def test_gemm_path_near_ties_from_duplicates():
    T, pos0 = 24, 3000
    inp = synth.layer_inputs(T, pos0 + T, seed=22)
    src = np.arange(0, 3000, 7)
    inp["kq"][src + 3] = inp["kq"][src]
    inp["ksc"][src + 3] = inp["ksc"][src]
    ids, out = gpu_select_prefill(inp, T, pos0)
    ref_out, ref_ids, _, _ = oracle.prefill(inp, T, pos0)
    np.testing.assert_array_equal(ids, ref_ids)
    assert_close(out, ref_out, "duplicates, GEMM path")


def test_gemm_path_periodic_cache():
    # every 8th cell points along the first 8 tokens' query sum and outscores everything else
    # (a periodic structure that a sampled bracket sees in full); the other 8 tokens have their
    # own queries.  Both must give the exact ranking.
    T, pos0 = 16, 6000
    n = pos0 + T
    inp = synth.layer_inputs(T, n, seed=31)
    inp["q"][1:8] = inp["q"][0]
    qsum = inp["q"][0].astype(np.float64).reshape(2, 12, 256).sum(axis=1)  # [group][dim]
    hot = np.arange(0, n, 8)
    for g in range(2):
        inp["kq"][hot, g, :] = np.where(qsum[g] >= 0, 100, -100).astype(np.int8)
        inp["ksc"][hot, g, :] = np.float16(0.02)
    ids, out = gpu_select_prefill(inp, T, pos0)
    ref_out, ref_ids, _, _ = oracle.prefill(inp, T, pos0)
    np.testing.assert_array_equal(ids, ref_ids)
    assert_close(out, ref_out, "periodic cache")
    assert np.isin(hot[hot < pos0 + 1], ids[0, 0]).all()  # the hot cells are all kept


@pytest.mark.parametrize("T,pos0", [(2, 50000), (12, 65524)])
def test_select_at_the_largest_caches(T, pos0):
    # past 32,768 cells the top-k holds 128 cells per thread (its largest form); (12, 65524) ends
    # at the 65,536-cell limit on the score-GEMM path, (2, 50000) is a few-row call
    inp = synth.layer_inputs(T, pos0 + T, seed=T + pos0)
    ids, out = gpu_select_prefill(inp, T, pos0)
    ref_out, ref_ids, _, _ = oracle.prefill(inp, T, pos0)
    np.testing.assert_array_equal(ids, ref_ids)
    assert_close(out, ref_out, f"T={T} pos0={pos0}")


@pytest.mark.parametrize("T,pos0", [(3, 70000), (2, 100000)])
def test_select_beyond_the_score_path_limit(T, pos0):
    # n_kv above 65,536: qsa_select hands the call to the single-launch decode layer's cluster
    # kernel in its ids-only form (no workspace); ids bit-exact, and the gathered prefill over them
    inp = synth.layer_inputs(T, pos0 + T, seed=T + pos0)
    n = pos0 + T
    assert qsa.qsa_select_workspace_bytes(T, pos0, n) == 0
    d = to_dev(inp)
    ids = torch.full((T, 2, 2048), -7, dtype=torch.int32, device="cuda")
    qsa.qsa_select(d["q"], d["kq"], d["ksc"], n, T, pos0, ids, None)
    ids2 = torch.full((T, 2, 2048), -7, dtype=torch.int32, device="cuda")
    qsa.qsa_select_noalloc(d["q"], d["kq"], d["ksc"], n, T, pos0, ids2)
    qsa.qsa_check_device_status()
    ref_out, ref_ids, _, _ = oracle.prefill(inp, T, pos0)
    np.testing.assert_array_equal(ids.cpu().numpy(), ref_ids)
    np.testing.assert_array_equal(ids2.cpu().numpy(), ref_ids)
    out = torch.full((T, 24, 256), float("nan"), dtype=torch.float16, device="cuda")
    pws = torch.empty(qsa.qsa_flash_prefill_workspace_bytes(T, pos0, n), dtype=torch.uint8, device="cuda")
    qsa.qsa_flash_prefill(d["q"], d["kq"], d["vq"], d["ksc"], d["vsc"], n, T, pos0, ids, out, pws)
    qsa.qsa_check_device_status()
    assert_close(out.float().cpu().numpy(), ref_out, f"prefill over {n} cells")


@pytest.mark.parametrize("T,pos0,chunk", [(300, 30000, 64), (12, 3000, 1)])
def test_select_in_chunks_with_a_small_workspace(T, pos0, chunk):
    # a workspace sized for chunks of `chunk` tokens: the same ids as with the full workspace, and
    # the oracle's on a sample of tokens
    n = pos0 + T
    inp = synth.layer_inputs(T, n, seed=T + pos0 + chunk)
    full = qsa.qsa_select_workspace_bytes(T, pos0, n)
    small = qsa.qsa_select_workspace_bytes(chunk, pos0 + T - chunk, n)
    assert small < full
    d = to_dev(inp)
    ids_full = torch.full((T, 2, 2048), -7, dtype=torch.int32, device="cuda")
    ids_small = torch.full((T, 2, 2048), -7, dtype=torch.int32, device="cuda")
    qsa.qsa_select(d["q"], d["kq"], d["ksc"], n, T, pos0, ids_full, torch.empty(full, dtype=torch.uint8, device="cuda"))
    qsa.qsa_select(d["q"], d["kq"], d["ksc"], n, T, pos0, ids_small,
                   torch.empty(small, dtype=torch.uint8, device="cuda"))
    qsa.qsa_check_device_status()
    a, b = ids_full.cpu().numpy(), ids_small.cpu().numpy()
    np.testing.assert_array_equal(a, b)
    toks = np.arange(0, T, max(1, T // 10), dtype=np.int32)
    _, ref_ids, _, _ = oracle.prefill(inp, T, pos0, toks=toks)
    np.testing.assert_array_equal(b[toks], ref_ids)

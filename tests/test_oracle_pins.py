"""Pins of the CPU oracle against things other than itself (no GPU needed).

Each test checks the oracle against a fixed point that the layer's definition or plain
mathematics gives: exact rational arithmetic, brute-force dense attention through a
library routine, closed forms, the merge identity, invariants of the selection and of the
quantiser, and the IEEE binary16 format as numpy implements it.
"""
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from int8_kv_top_gb300 import synth

HD, HPG, NG = 256, 12, 2


def dequant(codes, scales):
    """k^ = code * scale of its 64-element block (float64)."""
    return codes.astype(np.float64) * np.repeat(scales.astype(np.float64), 64, axis=-1)


def tiny_inputs(T, n, seed=11):
    return synth.layer_inputs(T, n, seed=seed)


# ------------------------------------------------------------------ binary16 format
def test_half_decode_matches_numpy_for_every_finite_pattern():
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    finite = np.isfinite(ref)
    got = np.array([oracle.half_to_double(int(b)) for b in bits[finite][::7]])
    np.testing.assert_array_equal(got, ref[finite][::7])


def test_float_to_half_rounds_to_nearest_even_like_numpy():
    rng = np.random.default_rng(3)
    xs = np.concatenate([
        rng.standard_normal(3000).astype(np.float32) * 10.0,
        (rng.uniform(-1, 1, 2000) * 1e-5).astype(np.float32),       # subnormal range
        np.array([65504, 65519, 65520, 1e9, -0.0, 2.0 ** -25, 2.0 ** -24 * 1.5, 1 + 2 ** -11, 1 + 3 * 2 ** -11],
                 dtype=np.float32),
    ])
    got = np.array([oracle.float_to_half_bits(float(x)) for x in xs], dtype=np.uint16)
    with np.errstate(over="ignore"):
        ref = xs.astype(np.float16).view(np.uint16)
    np.testing.assert_array_equal(got, ref)


# ------------------------------------------------------------------ attention (identity)
@pytest.mark.parametrize("T,pos0", [(8, 0), (6, 40), (1, 0)])
def test_identity_attention_matches_library_sdpa(T, pos0):
    n = pos0 + T
    inp = tiny_inputs(T, n, seed=T + pos0)
    out, ids, n_set, _ = oracle.prefill(inp, T, pos0)
    q = torch.from_numpy(inp["q"].astype(np.float64))                   # [T][24][256]
    k = torch.from_numpy(dequant(inp["kq"], inp["ksc"]))                # [n][2][256]
    v = torch.from_numpy(dequant(inp["vq"], inp["vsc"]))
    # query head h reads group h // 12; causal: token t sees cells 0 .. pos0 + t
    kk = k[:, torch.arange(24) // 12, :].permute(1, 0, 2)               # [24][n][256]
    vv = v[:, torch.arange(24) // 12, :].permute(1, 0, 2)
    mask = torch.arange(n)[None, :] <= (pos0 + torch.arange(T))[:, None]
    ref = torch.nn.functional.scaled_dot_product_attention(q.permute(1, 0, 2), kk, vv, attn_mask=mask,
                                                           scale=1 / 16).permute(1, 0, 2)
    np.testing.assert_allclose(out, ref.numpy(), rtol=1e-12, atol=1e-12)
    assert (ids == -1).all()
    assert (n_set == (pos0 + np.arange(T) + 1)[:, None]).all()


def test_single_cell_gives_its_value_row():
    inp = tiny_inputs(1, 1)
    out, *_ = oracle.prefill(inp, 1, 0)
    vhat = dequant(inp["vq"], inp["vsc"])[0]                           # [2][256]
    np.testing.assert_allclose(out[0], vhat[np.arange(24) // 12], rtol=0, atol=1e-15)


def test_zero_query_gives_mean_of_values():
    inp = tiny_inputs(1, 37)
    inp["q"][:] = 0
    out, *_ = oracle.prefill(inp, 1, 36)
    vhat = dequant(inp["vq"], inp["vsc"]).mean(axis=0)                 # [2][256]
    np.testing.assert_allclose(out[0], vhat[np.arange(24) // 12], rtol=1e-13, atol=1e-15)


def test_equal_keys_give_mean_of_values():
    inp = tiny_inputs(1, 20)
    inp["kq"][:] = inp["kq"][0]
    inp["ksc"][:] = inp["ksc"][0]
    out, *_ = oracle.prefill(inp, 1, 19)
    vhat = dequant(inp["vq"], inp["vsc"]).mean(axis=0)
    np.testing.assert_allclose(out[0], vhat[np.arange(24) // 12], rtol=1e-13, atol=1e-15)


def test_dominant_logit_selects_its_value_row():
    inp = tiny_inputs(1, 30)
    inp["q"][:] = 0
    inp["q"][0, :, :] = 1.0
    inp["kq"][:] = 0
    inp["kq"][17] = 127
    inp["ksc"][17] = 0.02                                              # logit 256*127*0.02/16 = 40.6
    out, *_ = oracle.prefill(inp, 1, 29)
    vhat = dequant(inp["vq"], inp["vsc"])[17]
    np.testing.assert_allclose(out[0], vhat[np.arange(24) // 12], rtol=0, atol=1e-14)


# ------------------------------------------------------------------ selection
def exact_scores(q_tok, kq, ksc, g, n):
    """sum over the group's 12 heads of q . k^ as exact rationals (the 1/16 is a positive factor)."""
    qs = [[Fraction(float(x)) for x in q_tok[g * HPG + h]] for h in range(HPG)]
    qsum = [sum(qs[h][d] for h in range(HPG)) for d in range(HD)]
    out = []
    for c in range(n):
        s = Fraction(0)
        for b in range(4):
            sc = Fraction(float(ksc[c, g, b]))
            s += sc * sum(qsum[d] * int(kq[c, g, d]) for d in range(64 * b, 64 * b + 64))
        out.append(s)
    return out


@pytest.mark.parametrize("n_kv,topk,idmax,seed", [(12, 4, 7, 1), (9, 4, 7, 2), (31, 5, 8, 3), (8, 4, 7, 4)])
def test_selection_matches_brute_force_exact_sort(n_kv, topk, idmax, seed):
    inp = tiny_inputs(1, n_kv, seed=seed)
    for g in range(NG):
        cells, _ = oracle.cell_set(inp["q"][0], inp["kq"], inp["ksc"], n_kv, g, topk=topk, identity_max=idmax)
        sc = exact_scores(inp["q"][0], inp["kq"], inp["ksc"], g, n_kv)
        order = sorted(range(n_kv), key=lambda c: (-sc[c], c))
        np.testing.assert_array_equal(cells, np.sort(order[:topk]))


def test_exact_key_equals_rational_score():
    inp = tiny_inputs(1, 6, seed=9)
    for g in range(NG):
        sc = exact_scores(inp["q"][0], inp["kq"], inp["ksc"], g, 6)
        for c in range(6):
            key = oracle.exact_key(inp["q"][0], inp["kq"], inp["ksc"], c, g)
            assert Fraction(key, 2 ** 48) == sc[c]


def test_identity_threshold_boundary():
    inp = tiny_inputs(1, 10, seed=5)
    cells, _ = oracle.cell_set(inp["q"][0], inp["kq"], inp["ksc"], 7, 0, topk=4, identity_max=7)
    np.testing.assert_array_equal(cells, np.arange(7))                # n_kv == identity_max: all cells
    cells, _ = oracle.cell_set(inp["q"][0], inp["kq"], inp["ksc"], 8, 0, topk=4, identity_max=7)
    assert len(cells) == 4                                            # one more cell: top-k


def test_exact_ties_go_to_the_lower_index():
    inp = tiny_inputs(1, 40, seed=6)
    inp["kq"][:] = inp["kq"][5]
    inp["ksc"][:] = inp["ksc"][5]
    for g in range(NG):
        cells, _ = oracle.cell_set(inp["q"][0], inp["kq"], inp["ksc"], 40, g, topk=6, identity_max=9)
        np.testing.assert_array_equal(cells, np.arange(6))
    # duplicates of a winning cell placed above and below it: all copies tie
    inp = tiny_inputs(1, 40, seed=7)
    sc = exact_scores(inp["q"][0], inp["kq"], inp["ksc"], 0, 40)
    best = max(range(40), key=lambda c: (sc[c], -c))
    for dup in (2, 30, 39):
        inp["kq"][dup] = inp["kq"][best]
        inp["ksc"][dup] = inp["ksc"][best]
    copies = sorted({best, 2, 30, 39})
    cells, _ = oracle.cell_set(inp["q"][0], inp["kq"], inp["ksc"], 40, 0, topk=2, identity_max=9)
    np.testing.assert_array_equal(cells, copies[:2])


def test_selection_invariants_at_full_budget():
    n_kv = 2600
    inp = tiny_inputs(1, n_kv, seed=8)
    q = inp["q"][0].astype(np.float64)
    k = dequant(inp["kq"], inp["ksc"])
    for g in range(NG):
        cells, differs = oracle.cell_set(inp["q"][0], inp["kq"], inp["ksc"], n_kv, g, with_f64_check=True)
        assert len(cells) == 2048 and np.all(np.diff(cells) > 0) and cells[0] >= 0 and cells[-1] < n_kv
        score = (q[g * 12:(g + 1) * 12] @ k[:, g, :].T).sum(axis=0) / 16   # float64, independent of the C code
        kept = np.zeros(n_kv, bool)
        kept[cells] = True
        assert score[kept].min() >= score[~kept].max() - 1e-9
        assert not differs


# ------------------------------------------------------------------ partials and merge
def test_single_chunk_partials_match_numpy():
    inp = tiny_inputs(1, 50, seed=12)
    cells = np.arange(50, dtype=np.int32)
    q = inp["q"][0].astype(np.float64)
    k = dequant(inp["kq"], inp["ksc"])
    v = dequant(inp["vq"], inp["vsc"])
    for g in range(NG):
        part = oracle.partials(inp["q"][0], inp["kq"], inp["vq"], inp["ksc"], inp["vsc"], g, cells)
        assert part.shape == (1, 12, 258)
        s = q[g * 12:(g + 1) * 12] @ k[:, g, :].T / 16                    # [12][50]
        m = s.max(axis=1)
        e = np.exp(s - m[:, None])
        np.testing.assert_allclose(part[0, :, 256], m, rtol=1e-14)
        np.testing.assert_allclose(part[0, :, 257], e.sum(axis=1), rtol=1e-13)
        np.testing.assert_allclose(part[0, :, :256], e @ v[:, g, :], rtol=1e-12, atol=1e-13)


def test_merge_of_any_split_equals_unsplit_attention():
    rng = np.random.default_rng(4)
    inp = tiny_inputs(1, 300, seed=13)
    cells = np.sort(rng.choice(300, size=170, replace=False)).astype(np.int32)
    for g in range(NG):
        direct = oracle.attend(inp["q"][0], inp["kq"], inp["vq"], inp["ksc"], inp["vsc"], g, cells)
        # chunked by 64 (the layer's split) and by random cut points (each piece <= 64 cells)
        part64 = oracle.partials(inp["q"][0], inp["kq"], inp["vq"], inp["ksc"], inp["vsc"], g, cells)
        np.testing.assert_allclose(oracle.merge_group(part64), direct, rtol=1e-12, atol=1e-13)
        cuts = np.sort(rng.choice(np.arange(1, 170), size=5, replace=False))
        pieces = np.split(cells, cuts)
        pieces = [p for p in pieces if len(p)]
        parts = np.concatenate([oracle.partials(inp["q"][0], inp["kq"], inp["vq"], inp["ksc"], inp["vsc"], g, p)
                                for p in pieces])
        np.testing.assert_allclose(oracle.merge_group(parts), direct, rtol=1e-12, atol=1e-13)


def test_merge_closed_form_two_chunks():
    part = np.full((1, 2, 24, 258), np.nan, dtype=np.float32)
    o1 = np.linspace(-1, 1, 256, dtype=np.float32)
    o2 = np.linspace(2, 3, 256, dtype=np.float32)
    part[0, 0, :, :256], part[0, 0, :, 256], part[0, 0, :, 257] = o1, 0.0, 1.0
    part[0, 1, :, :256], part[0, 1, :, 256], part[0, 1, :, 257] = o2, np.float32(np.log(2.0)), 1.0
    out = oracle.merge_f32(part, [2])
    m2 = float(np.float32(np.log(2.0)))
    w1 = np.exp(0.0 - m2)                       # chunk 1 relative to the max m = ln 2
    expect = (w1 * o1.astype(np.float64) + o2) / (w1 + 1.0)
    np.testing.assert_allclose(out[0], np.broadcast_to(expect, (24, 256)), rtol=1e-14)


def test_merge_ignores_slots_past_the_chunk_count():
    part = synth.merge_partials([3, 1], chunk_cap=4, seed=2)
    out = oracle.merge_f32(part, [3, 1])
    assert np.isfinite(out).all()
    np.testing.assert_allclose(out[1], part[1, 0, :, :256] / part[1, 0, :, 257:258], rtol=1e-6)


def test_decode_driver_is_consistent_with_prefill_driver():
    P, N = 70, 3
    inp = tiny_inputs(N, P + N, seed=14)
    part, n_chunks, merged, direct, ids = oracle.decode(inp, N, P, topk=40, identity_max=71)
    out, ids_p, n_set, _ = oracle.prefill(inp, N, P, topk=40, identity_max=71)
    np.testing.assert_allclose(merged, direct, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(direct, out, rtol=0, atol=0)
    np.testing.assert_array_equal(ids, ids_p)
    assert list(n_set[:, 0]) == [71, 40, 40]                        # 71 = identity, then top-40
    assert list(n_chunks) == [2, 1, 1]


# ------------------------------------------------------------------ quantiser
def test_quantize_hand_worked_block():
    # a = 1.0 -> a/127 = 0.0078740157 -> fp16 0x2008 = 2^-7 * (1 + 8/1024) = 0.00787353515625
    # codes: 1.0/s = 127.007 -> 127; -0.5/s = -63.50 -> -64; 0.25/s = 31.75 -> 32; 0.75/s = 95.25 -> 95
    x = np.zeros((1, 256), np.float16)
    x[0, :4] = [1.0, -0.5, 0.25, 0.75]
    xq, xsc = oracle.quantize(x)
    assert xsc.view(np.uint16)[0, 0] == 0x2008
    assert list(xq[0, :4]) == [127, -64, 32, 95]
    assert (xq[0, 64:] == 0).all() and (xsc.view(np.uint16)[0, 1:] == 0).all()   # zero blocks: +0 scale


def test_quantize_roundtrip_bounds():
    x = synth.fp16_rows(200, seed=3)
    xq, xsc = oracle.quantize(x)
    xs = x.astype(np.float64).reshape(200, 2, 4, 64)
    s = xsc.astype(np.float64)[..., None]
    codes = xq.astype(np.float64).reshape(200, 2, 4, 64)
    assert np.abs(codes).max() <= 127
    assert (np.abs(codes).max(axis=-1) == 127).all()                  # the absmax element maps to +-127
    # |x - code * scale| <= scale / 2 up to the fp32 rounding of x / scale
    assert (np.abs(xs - codes * s) <= s * (0.5 + 2.0 ** -20)).all()
    # the scale is the fp16 rounding of absmax / 127
    a = np.abs(xs).max(axis=-1)
    np.testing.assert_array_equal(xsc.reshape(200, 2, 4), (a.astype(np.float32) / np.float32(127)).astype(np.float16))


def test_quantize_rounds_exact_halves_away_from_zero():
    # absmax 127 * 2^-8 makes the scale exactly 2^-8 (a / 127 and its fp16 rounding are exact),
    # so x = (k + 1/2) * 2^-8 gives x / scale = k + 1/2 exactly: a true tie for even and odd k.
    # Round-half-away-from-zero sends k + 1/2 to k + 1 and -(k + 1/2) to -(k + 1); a
    # ties-to-even rule would send the even k down instead.
    ks = np.array([0, 1, 2, 3, 10, 11, 62, 63, 124, 125], dtype=np.float64)
    vals = np.concatenate([[127.0], ks + 0.5, -(ks + 0.5)])          # in units of the scale
    x = np.zeros((1, 256), np.float16)
    x[0, :len(vals)] = (vals * 2.0 ** -8).astype(np.float16)
    assert np.array_equal(x[0, :len(vals)].astype(np.float64), vals * 2.0 ** -8)  # every value exact in fp16
    xq, xsc = oracle.quantize(x)
    assert xsc.view(np.uint16)[0, 0] == np.float16(2.0 ** -8).view(np.uint16)
    expect = (np.sign(vals) * np.floor(np.abs(vals) + 0.5)).astype(np.int64)
    np.testing.assert_array_equal(xq[0, :len(vals)].astype(np.int64), expect)
    assert list(expect[1:5]) == [1, 2, 3, 4] and list(expect[11:15]) == [-1, -2, -3, -4]


def test_decode_part_layout_is_per_group_partials_in_head_order():
    # oracle.decode's part [N][cap][24][258] must hold, for token t, chunk k and query head
    # 12 g + h, the partial of group g's head h over chunk k of the token's ascending set
    # ("round 27 track b - qsa prep and merge", correctness: head stride 258, chunk stride
    # 24 * 258); slots past the chunk count are left untouched.
    P, N, topk, idmax = 150, 3, 40, 151
    inp = tiny_inputs(N, P + N, seed=15)
    part, n_chunks, merged, _, ids = oracle.decode(inp, N, P, topk=topk, identity_max=idmax)
    cap = part.shape[1]
    for t in range(N):
        n_kv = P + t + 1
        for g in range(NG):
            cells, _ = oracle.cell_set(inp["q"][t], inp["kq"], inp["ksc"], n_kv, g, topk=topk, identity_max=idmax)
            gp = oracle.partials(inp["q"][t], inp["kq"], inp["vq"], inp["ksc"], inp["vsc"], g, cells)
            nc = gp.shape[0]
            assert n_chunks[t] == nc
            np.testing.assert_array_equal(part[t, :nc, g * HPG:(g + 1) * HPG, :], gp)
            assert np.isnan(part[t, nc:cap, g * HPG:(g + 1) * HPG, :]).all()
    assert list(n_chunks) == [3, 1, 1]    # 151 identity cells (3 chunks), then top-40 (1 chunk)


def test_batched_decode_oracle_is_per_sequence_decode_on_its_slice():
    # three sequences in one pool: the batch oracle must give each sequence exactly what a
    # decode of that sequence's own cache and tokens gives (no cell or token of another leaks in)
    rng = np.random.default_rng(4)
    lens = [(90, 85, 2), (40, 37, 3), (130, 120, 1)]          # (n_cells, pos0, tokens)
    pieces = [tiny_inputs(nt, n, seed=30 + i) for i, (n, p0, nt) in enumerate(lens)]
    pool = {k: np.concatenate([pc[k] for pc in pieces], axis=0) for k in ("q", "kq", "vq", "ksc", "vsc")}
    seqs, c0, t0 = [], 0, 0
    for n, p0, nt in lens:
        seqs.append((c0, n, p0, t0))
        c0 += n
        t0 += nt
    out, ids = oracle.decode_batch(pool, seqs, topk=40, identity_max=71)
    t0 = 0
    for (n, p0, nt), pc in zip(lens, pieces):
        _, _, merged, direct, sid = oracle.decode(pc, nt, p0, topk=40, identity_max=71)
        np.testing.assert_array_equal(out[t0:t0 + nt], merged)
        np.testing.assert_array_equal(ids[t0:t0 + nt], sid)
        np.testing.assert_allclose(merged, direct, rtol=1e-12, atol=1e-13)   # merge identity per sequence
        t0 += nt
    del rng



def test_batched_prefill_oracle_matches_brute_force_over_the_pool():
    # three sequences at different pool offsets (one with an unused gap of cells before it, one
    # with no tokens): every token's set is found from the pool rows by brute force (identity
    # range, or the exact rational top-k with ties to the lower index), then plain float64 softmax
    # attention of its 12 heads; the batch oracle must agree to rounding
    topk, idmax = 4, 7
    lens = [(9, 3, 4), (12, 10, 2), (5, 5, 0), (20, 6, 3)]         # (n_cells, pos0, tokens)
    gap = 6
    pieces = [tiny_inputs(max(nt, 1), n, seed=40 + i) for i, (n, p0, nt) in enumerate(lens)]
    q = np.concatenate([pc["q"][:nt] for pc, (n, p0, nt) in zip(pieces, lens)], axis=0)
    pool, seqs, c0, t0 = {k: [] for k in ("kq", "vq", "ksc", "vsc")}, [], 0, 0
    for i, ((n, p0, nt), pc) in enumerate(zip(lens, pieces)):
        if i == 1:   # unused pool cells before sequence 1
            filler = tiny_inputs(1, gap, seed=99)
            for k in pool:
                pool[k].append(filler[k])
            c0 += gap
        for k in pool:
            pool[k].append(pc[k])
        seqs.append((c0, n, p0, t0))
        c0 += n
        t0 += nt
    pool = {k: np.concatenate(v, axis=0) for k, v in pool.items()}
    pool["q"] = q
    out, ids = oracle.prefill_batch(pool, seqs, topk=topk, identity_max=idmax)
    k_all, v_all = dequant(pool["kq"], pool["ksc"]), dequant(pool["vq"], pool["vsc"])
    n_tok = q.shape[0]
    for r in range(n_tok):
        s = max(i for i, e in enumerate(seqs) if e[3] <= r and (i + 1 == len(seqs) or seqs[i + 1][3] > r))
        cfirst, _, p0, tfirst = seqs[s]
        n_kv = p0 + (r - tfirst) + 1
        for g in range(NG):
            if n_kv <= idmax:
                cells = np.arange(n_kv)
                assert (ids[r, g] == -1).all()
            else:
                sub_kq = pool["kq"][cfirst:cfirst + n_kv]
                sub_ksc = pool["ksc"][cfirst:cfirst + n_kv]
                sc = exact_scores(q[r], sub_kq, sub_ksc, g, n_kv)
                cells = np.sort(sorted(range(n_kv), key=lambda c: (-sc[c], c))[:topk])
                np.testing.assert_array_equal(ids[r, g], cells)
            kk, vv = k_all[cfirst + cells, g], v_all[cfirst + cells, g]
            for h in range(HPG):
                logit = (kk @ q[r, g * HPG + h].astype(np.float64)) / 16
                w = np.exp(logit - logit.max())
                np.testing.assert_allclose(out[r, g * HPG + h], (w / w.sum()) @ vv, rtol=1e-12, atol=1e-13)


# ------------------------------------------------------------------ output gate
def test_gate_zero_halves_and_symmetric_gates_sum_to_the_output():
    rng = np.random.default_rng(8)
    out = rng.standard_normal((3, 24, 256))
    zero = np.zeros((3, 24, 256), np.float16)
    np.testing.assert_array_equal(oracle.apply_gate(out, zero), out / 2)        # sigmoid(0) = 1/2 exactly
    g = synth.gate_input(3, seed=9)
    both = oracle.apply_gate(out, g) + oracle.apply_gate(out, -g)              # sigmoid(x) + sigmoid(-x) = 1
    np.testing.assert_allclose(both, out, rtol=1e-14, atol=1e-15)


def test_gate_matches_the_library_logistic_function():
    from scipy.special import expit
    rng = np.random.default_rng(10)
    out = rng.standard_normal((2, 24, 256))
    g = synth.gate_input(2, seed=11, spread=6.0)
    ref = out * expit(g.astype(np.float64))
    np.testing.assert_allclose(oracle.apply_gate(out, g), ref, rtol=1e-13, atol=0)
    big = np.full((1, 24, 256), 30.0, np.float16)                              # a fully open gate
    np.testing.assert_allclose(oracle.apply_gate(out[:1], big), out[:1], rtol=1e-12)
    np.testing.assert_allclose(oracle.apply_gate(out[:1], -big), 0.0, atol=1e-12)



# ------------------------------------------------------------------ fused prep (norm, rope)
def prep_case(T=3, seed=12):
    return synth.prep_inputs(T, seed=seed)


def test_prep_at_position_zero_is_the_library_rms_norm():
    # theta = 0 at position 0: the rotation is the identity, leaving torch's rms_norm with weight
    inp = prep_case()
    qc, kc = oracle.prep(inp["q_raw"], inp["k_raw"], inp["q_gamma"], inp["k_gamma"], 1, 0)
    x = torch.from_numpy(inp["q_raw"][:1].astype(np.float64))
    ref = torch.nn.functional.rms_norm(x, (256,), torch.from_numpy(inp["q_gamma"].astype(np.float64)), eps=1e-6)
    np.testing.assert_allclose(qc, ref.numpy(), rtol=1e-12, atol=1e-12)
    xk = torch.from_numpy(inp["k_raw"][:1].astype(np.float64))
    refk = torch.nn.functional.rms_norm(xk, (256,), torch.from_numpy(inp["k_gamma"].astype(np.float64)), eps=1e-6)
    np.testing.assert_allclose(kc, refk.numpy(), rtol=1e-12, atol=1e-12)


def test_prep_rotation_is_multiplication_by_exp_i_theta():
    # RoFormer's definition: the pair (y_i, y_{i+128}) read as y_i + i y_{i+128} is multiplied by
    # e^{i p theta_i}, theta_i = base^(-2i/256); the rotated rows against the normed rows at p = 0
    inp = prep_case(T=4)
    T, pos0 = 4, 1000
    qc, kc = oracle.prep(inp["q_raw"], inp["k_raw"], inp["q_gamma"], inp["k_gamma"], T, pos0)
    for t in range(T):
        one = {k: v[t:t + 1] for k, v in inp.items() if k.endswith("raw")}
        q0, k0 = oracle.prep(one["q_raw"], one["k_raw"], inp["q_gamma"], inp["k_gamma"], 1, 0)
        theta = (pos0 + t) * 10000.0 ** (-2.0 * np.arange(128) / 256)
        z = (q0[0, :, :128] + 1j * q0[0, :, 128:]) * np.exp(1j * theta)
        np.testing.assert_allclose(qc[t, :, :128], z.real, rtol=0, atol=1e-11)
        np.testing.assert_allclose(qc[t, :, 128:], z.imag, rtol=0, atol=1e-11)


def test_prep_rotation_keeps_pair_norms_and_depends_only_on_relative_position():
    inp = prep_case(T=1, seed=13)
    dots = []
    for m, n in [(5, 2), (1005, 1002), (60005, 60002)]:
        qa, _ = oracle.prep(inp["q_raw"], inp["k_raw"], inp["q_gamma"], inp["k_gamma"], 1, m)
        _, kb = oracle.prep(inp["q_raw"], inp["k_raw"], inp["q_gamma"], inp["k_gamma"], 1, n)
        dots.append(np.einsum("hd,d->h", qa[0], kb[0, 0]))
        q0, _ = oracle.prep(inp["q_raw"], inp["k_raw"], inp["q_gamma"], inp["k_gamma"], 1, 0)
        np.testing.assert_allclose(qa[0, :, :128] ** 2 + qa[0, :, 128:] ** 2, q0[0, :, :128] ** 2 + q0[0, :, 128:] ** 2,
                                   rtol=1e-12)
    np.testing.assert_allclose(dots[1], dots[0], rtol=1e-9, atol=1e-9)
    np.testing.assert_allclose(dots[2], dots[0], rtol=1e-7, atol=1e-7)


def test_prep_mrope_with_equal_positions_is_rope_and_sections_pick_components():
    inp = prep_case(T=2, seed=14)
    pos3 = np.array([[70, 70, 70], [71, 71, 71]], np.int32)
    a = oracle.prep(inp["q_raw"], inp["k_raw"], inp["q_gamma"], inp["k_gamma"], 2, 70)
    b = oracle.prep(inp["q_raw"], inp["k_raw"], inp["q_gamma"], inp["k_gamma"], 2, 0, pos3=pos3)
    np.testing.assert_array_equal(a[0], b[0])
    np.testing.assert_array_equal(a[1], b[1])
    # pairs of section 0 follow component 0 only: changing components 1 and 2 leaves them alone
    c = oracle.prep(inp["q_raw"], inp["k_raw"], inp["q_gamma"], inp["k_gamma"], 2, 0,
                    pos3=np.array([[70, 3, 9], [71, 4, 8]], np.int32))
    np.testing.assert_array_equal(c[0][..., :32], a[0][..., :32])
    np.testing.assert_array_equal(c[0][..., 128:160], a[0][..., 128:160])
    assert not np.allclose(c[0][..., 32:128], a[0][..., 32:128])


def test_prep_partial_rotary_leaves_the_tail_unrotated():
    inp = prep_case(T=1, seed=15)
    q64, _ = oracle.prep(inp["q_raw"], inp["k_raw"], inp["q_gamma"], inp["k_gamma"], 1, 500, rotary_dim=64)
    q0, _ = oracle.prep(inp["q_raw"], inp["k_raw"], inp["q_gamma"], inp["k_gamma"], 1, 0)
    np.testing.assert_array_equal(q64[..., 64:], q0[..., 64:])
    theta = 500 * 10000.0 ** (-2.0 * np.arange(32) / 64)
    z = (q0[0, :, :32] + 1j * q0[0, :, 32:64]) * np.exp(1j * theta)
    np.testing.assert_allclose(q64[0, :, :32], z.real, atol=1e-12)
    np.testing.assert_allclose(q64[0, :, 32:64], z.imag, atol=1e-12)

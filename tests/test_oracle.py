"""Pins for the CPU oracle: closed forms, invariants, brute force and the
numbers printed in the guide. None of these calls the CUDA library."""
import itertools
import math
import os

import numpy as np
import pytest
import torch

from oracle import msa_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
RNG = np.random.default_rng(12345)


def _golden_rows(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(line.split())
    return rows


# --------------------------------------------------------------------------- rounding

def test_bf16_rounding_matches_torch_conversion():
    # torch's float32 -> bfloat16 conversion is round-to-nearest-even
    x = np.concatenate([
        RNG.standard_normal(20000).astype(np.float32),
        (RNG.standard_normal(2000) * 1e-30).astype(np.float32),
        (RNG.standard_normal(2000) * 1e30).astype(np.float32),
        np.array([0.0, -0.0, 1.0, -1.0, 3.0e38, -3.0e38, 1e-40, np.inf, -np.inf], dtype=np.float32),
    ])
    ref = torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()
    got = O.round_to_bf16(x)
    assert np.array_equal(got, ref)


def test_bf16_rounding_ties_to_even():
    ulp = 2.0 ** -7  # bf16 spacing in [1, 2)
    cases = {
        1.0 + ulp / 2: 1.0,                    # tie, 1.0 is even
        1.0 + ulp + ulp / 2: 1.0 + 2 * ulp,    # tie, 1+ulp is odd -> up
        1.0 + ulp / 2 + 2.0 ** -20: 1.0 + ulp,  # just above the tie
        -(1.0 + ulp / 2): -1.0,
    }
    for x, want in cases.items():
        assert O.round_to_bf16(np.float32(x)) == want
    assert np.isnan(O.round_to_bf16(np.float32(np.nan)))


# --------------------------------------------------------------------------- pooling

def test_pool_constant_block_is_exact():
    d = O.HEAD_DIM
    k = np.full((256, d), 0.3125)
    for store in ("bf16", "f32"):
        stored, exact = O.pool_block_keys(k, 256, store)
        assert stored.shape == (4, d)
        assert np.all(stored == 0.3125) and np.all(exact == 0.3125)


def test_pool_closed_form_index_pattern():
    # K[t, d] = 1024*block + (t mod 64) + d  ->  mean = 1024*block + 31.5 + d exactly
    d = O.HEAD_DIM
    t = np.arange(5 * 64 + 17)
    k = (1024.0 * (t // 64))[:, None] + (t % 64)[:, None] + np.arange(d)[None, :]
    stored, exact = O.pool_block_keys(k, len(t), "f32")
    assert stored.shape == (5, d)             # the partial sixth block is not pooled
    want = (1024.0 * np.arange(5))[:, None] + 31.5 + np.arange(d)[None, :]
    assert np.array_equal(stored, want) and np.array_equal(exact, want)


def test_pool_stored_value_within_rounding_bound_of_mean():
    d = O.HEAD_DIM
    k = O.round_to_bf16(RNG.standard_normal((64 * 40, d)).astype(np.float32))
    stored, exact = O.pool_block_keys(k, k.shape[0], "bf16")
    # fp32 sum of 64 terms: |err| <= 63 * 2^-24 * sum|x|; then a half bf16 ulp
    absmean = np.abs(k).reshape(40, 64, d).mean(axis=1)
    bound = 63 * 2.0 ** -24 * absmean + np.abs(exact) * 2.0 ** -8 + 1e-30
    assert np.all(np.abs(stored - exact) <= bound)


def test_mean_pooled_key_score_equals_mean_of_token_scores():
    # the reading of the guide's block pooling used here: scoring the mean key is
    # the mean of the token-level scores (linearity), exact in float64
    d = O.HEAD_DIM
    k = RNG.standard_normal((64 * 8, d))
    q = RNG.standard_normal(d)
    _, exact = O.pool_block_keys(k, k.shape[0], "f32")
    tok = (k @ q).reshape(8, 64).mean(axis=1)
    assert np.allclose(exact @ q, tok, rtol=0, atol=1e-12)


# --------------------------------------------------------------------------- index query

def test_index_query_sums_group_heads():
    d = O.HEAD_DIM
    g = 3
    q = np.zeros((g, d))
    for j in range(g):
        q[j, 5 * j] = 1.0
        q[j, 7] = 2.0
    qi = O.index_query(q)
    want = np.zeros(d)
    want[[0, 5, 10]] = 1.0
    want[7] = 2.0 * g
    assert np.array_equal(qi, want)
    # a prefill tile: rows x heads
    qt = np.ones((64, 8, d))
    assert np.all(O.index_query(qt) == 512.0)


# --------------------------------------------------------------------------- selection

def _brute_force_topk(scores, k):
    """The unique k-subset whose every member beats every non-member under
    (higher score, then lower index)."""
    n = len(scores)
    beats = lambda i, j: scores[i] > scores[j] or (scores[i] == scores[j] and i < j)  # noqa: E731
    found = []
    for sub in itertools.combinations(range(n), min(k, n)):
        s = set(sub)
        if all(beats(i, j) for i in s for j in range(n) if j not in s):
            found.append(sorted(sub))
    assert len(found) == 1
    return found[0]


@pytest.mark.parametrize("trial", range(60))
def test_select_matches_brute_force(trial):
    rng = np.random.default_rng(trial)
    n = int(rng.integers(1, 11))
    k = int(rng.integers(1, 6))
    if trial % 3 == 0:
        scores = rng.integers(-2, 3, size=n).astype(np.float64)   # many exact ties
    else:
        scores = rng.standard_normal(n)
    forced = n if trial % 2 == 0 else None
    k_total = k + 1
    sel = O.select_blocks(scores, k, forced, k_total)
    want = _brute_force_topk(list(scores), k)
    if forced is not None:
        want = sorted(want + [forced])
    want = want + [-1] * (k_total - len(want))
    assert list(sel) == want


def test_select_pads_when_few_candidates():
    sel = O.select_blocks(np.array([0.5, 2.0]), 5, 2, 6)
    assert list(sel) == [0, 1, 2, -1, -1, -1]
    sel = O.select_blocks(np.zeros(0), 3, 0, 4)
    assert list(sel) == [0, -1, -1, -1]


def test_planted_needles_are_selected():
    from synth import make_decode_inputs
    inp = make_decode_inputs([4096], 1, 4, "f32", "contiguous", needles=2, seed=1001)
    q = inp.q[0].double().numpy()
    k = inp.kv_rows(0, 0, "k").double().numpy()
    v = inp.kv_rows(0, 0, "v").double().numpy()
    res = O.decode_unit(q, k, v, 4096, 8, 9, 1 / math.sqrt(128), "f32")
    for b in inp.needles[(0, 0)]:
        assert b in res["selected"]
    assert res["selected"][-1] == 63          # newest block always kept
    assert sorted(res["selected"]) == list(res["selected"])


# --------------------------------------------------------------------------- attention

def test_attend_zero_query_is_mean_of_values():
    d = O.HEAD_DIM
    k = RNG.standard_normal((300, d))
    v = RNG.standard_normal((300, d))
    toks = np.array([3, 10, 11, 299])
    o, lse, p = O.attend(np.zeros((2, d)), k, v, toks, 0.1)
    assert np.allclose(o, v[toks].mean(axis=0), atol=1e-14)
    assert np.allclose(lse, math.log(4), atol=1e-14)
    assert np.allclose(p, 0.25, atol=1e-15)


def test_attend_two_tokens_closed_form():
    d = O.HEAD_DIM
    k = np.zeros((2, d))
    k[0, 0], k[1, 1] = 2.0, -1.0
    v = np.zeros((2, d))
    v[0, 3], v[1, 4] = 1.0, 1.0
    q = np.zeros((1, d))
    q[0, 0], q[0, 1] = 1.5, 0.5
    scale = 0.25
    z0, z1 = 1.5 * 2.0 * scale, 0.5 * -1.0 * scale
    p0 = 1.0 / (1.0 + math.exp(z1 - z0))
    o, lse, _ = O.attend(q, k, v, np.array([0, 1]), scale)
    assert abs(o[0, 3] - p0) < 1e-15 and abs(o[0, 4] - (1 - p0)) < 1e-15
    assert abs(lse[0] - math.log(math.exp(z0) + math.exp(z1))) < 1e-14


def test_attend_invariants():
    d = O.HEAD_DIM
    k = RNG.standard_normal((500, d))
    v = RNG.standard_normal((500, d))
    q = RNG.standard_normal((4, d))
    toks = np.sort(RNG.choice(500, size=130, replace=False))
    o, lse, p = O.attend(q, k, v, toks, 1 / math.sqrt(d))
    assert np.allclose(p.sum(axis=1), 1.0, atol=1e-12)
    perm = RNG.permutation(len(toks))
    o2, lse2, _ = O.attend(q, k, v, toks[perm], 1 / math.sqrt(d))
    assert np.allclose(o, o2, atol=1e-12) and np.allclose(lse, lse2, atol=1e-12)
    vc = np.tile(RNG.standard_normal(d), (500, 1))
    o3, _, _ = O.attend(q, k, vc, toks, 1 / math.sqrt(d))
    assert np.allclose(o3, vc[0], atol=1e-12)
    o4, _, _ = O.attend(q, k, v, np.array([77]), 1 / math.sqrt(d))
    assert np.allclose(o4, v[77], atol=1e-15)


def test_dense_closed_form_zero_query():
    d = O.HEAD_DIM
    v = RNG.standard_normal((200, d))
    k = RNG.standard_normal((200, d))
    o, lse = O.dense_gqa(np.zeros((3, d)), k, v, 150, 0.3)
    assert np.allclose(o, v[:151].mean(axis=0), atol=1e-13)
    assert np.allclose(lse, math.log(151), atol=1e-13)


@pytest.mark.parametrize("seq_len", [64 * 12, 64 * 12 + 1, 64 * 12 + 37])
def test_all_blocks_selected_equals_dense_decode(seq_len):
    d = O.HEAD_DIM
    rng = np.random.default_rng(seq_len)
    k = rng.standard_normal((64 * 13, d))
    v = rng.standard_normal((64 * 13, d))
    q = rng.standard_normal((4, d))
    nb = O.num_blocks(seq_len)
    res = O.decode_unit(q, k, v, seq_len, k_scored=nb, k_total=nb, scale=1 / math.sqrt(d), store="f32")
    assert list(res["selected"]) == list(range(nb))
    od, ld = O.dense_gqa(q, k, v, seq_len - 1, 1 / math.sqrt(d))
    assert np.allclose(res["o"], od, rtol=0, atol=1e-12)
    assert np.allclose(res["lse"], ld, rtol=0, atol=1e-12)


def test_all_blocks_selected_equals_dense_prefill():
    d = O.HEAD_DIM
    rng = np.random.default_rng(7)
    q_start, n_new, g = 128, 70, 2
    total = q_start + n_new
    k = rng.standard_normal((total, d))
    v = rng.standard_normal((total, d))
    q = rng.standard_normal((n_new, g, d))
    pooled, _ = O.pool_block_keys(k, total, "f32")
    for tile in range(2):
        rows = q[tile * 64:(tile + 1) * 64]
        sel = O.prefill_tile_select(rows, tile, q_start, pooled, k_scored=64, k_total=5)
        diag = q_start // 64 + tile
        assert list(sel["selected"][: diag + 1]) == list(range(diag + 1))
        pos = q_start + tile * 64 + np.arange(rows.shape[0])
        o, lse = O.prefill_rows(rows, pos, k, v, total, sel["selected"], 1 / math.sqrt(d))
        for i in range(rows.shape[0]):
            od, ld = O.dense_gqa(rows[i], k, v, pos[i], 1 / math.sqrt(d))
            assert np.allclose(o[i], od, atol=1e-12) and np.allclose(lse[i], ld, atol=1e-12)


def test_prefill_tile_excludes_future_blocks():
    d = O.HEAD_DIM
    rng = np.random.default_rng(3)
    k = rng.standard_normal((64 * 10, d))
    pooled, _ = O.pool_block_keys(k, 64 * 10, "f32")
    q = rng.standard_normal((64, 2, d))
    sel = O.prefill_tile_select(q, 2, 5 * 64, pooled, k_scored=3, k_total=4)
    assert sel["diag"] == 7 and len(sel["scores"]) == 7
    assert sel["selected"][-1] == 7 and all(0 <= b < 7 for b in sel["selected"][:-1])


# --------------------------------------------------------------------------- the guide's numbers

def test_golden_block_arithmetic():
    rows = _golden_rows("block_arithmetic.txt")
    for r in rows[:-1]:
        ctx, bs, want = int(r[0]), int(r[1]), int(r[2])
        assert bs == O.BLOCK and O.num_blocks(ctx) == want
    sp, flo, fhi, tlo, thi = map(float, rows[-1])
    nb = O.num_blocks(1048576)
    touched = 1.0 / sp
    assert flo <= touched <= fhi
    assert tlo <= touched * nb * O.BLOCK <= thi


def test_golden_diagram_groups_share_one_selection():
    """Six heads, two KV heads: heads 1-3 must use I1 and heads 4-6 use I2."""
    rows = _golden_rows("diagram_groups.txt")
    d = O.HEAD_DIM
    rng = np.random.default_rng(11)
    hq, hkv = 6, 2
    grp = hq // hkv
    seq_len = 64 * 16
    k = rng.standard_normal((hkv, seq_len, d))
    v = rng.standard_normal((hkv, seq_len, d))
    q = rng.standard_normal((hq, d))
    # plant a different needle block in each KV head, aligned with its group's mean query
    needles = {0: 3, 1: 11}
    for h, b in needles.items():
        k[h, b * 64:(b + 1) * 64] = 3 * q[h * grp:(h + 1) * grp].mean(axis=0)
    sel = {}
    for h in range(hkv):
        res = O.decode_unit(q[h * grp:(h + 1) * grp], k[h], v[h], seq_len, 2, 3, 1 / math.sqrt(d), "f32")
        sel[h] = res
        assert needles[h] in res["selected"]
    for head1, list1 in rows:
        j, h = int(head1) - 1, int(list1) - 1
        assert j // grp == h
        toks = O.tokens_of_blocks(sel[h]["selected"], seq_len)
        o, _, _ = O.attend(q[j:j + 1], k[h], v[h], toks, 1 / math.sqrt(d))
        assert np.allclose(o[0], sel[h]["o"][j - h * grp], atol=1e-13)
    assert list(sel[0]["selected"]) != list(sel[1]["selected"])


# --------------------------------------------------------------------------- token-level max-pooled score

def test_token_max_equals_summary_score_for_constant_blocks():
    # a block whose 64 index keys are one row r: max_t q.k_t = q.r, the score of
    # the summary key r (pooling 64 copies of r gives r exactly)
    rng = np.random.default_rng(7)
    nb = 5
    r = O.round_to_bf16(rng.standard_normal((nb, O.HEAD_DIM)).astype(np.float32))
    kidx = np.repeat(r, O.BLOCK, axis=0)
    q = rng.standard_normal(O.HEAD_DIM)
    got = O.score_blocks_token_max(q, kidx, nb)
    pooled, _ = O.pool_block_keys(kidx, nb * O.BLOCK, "bf16")
    want = O.score_blocks(q, pooled, nb)
    np.testing.assert_allclose(got, want, rtol=1e-14, atol=0)


def test_token_max_brute_force_and_bounds():
    rng = np.random.default_rng(8)
    nb = 3
    kidx = rng.standard_normal((nb * O.BLOCK, O.HEAD_DIM))
    q = rng.standard_normal(O.HEAD_DIM)
    got = O.score_blocks_token_max(q, kidx, nb)
    for b in range(nb):
        toks = [math.fsum(float(q[d]) * float(kidx[b * O.BLOCK + t, d]) for d in range(O.HEAD_DIM))
                for t in range(O.BLOCK)]
        assert abs(got[b] - max(toks)) <= 1e-12 * max(1.0, abs(max(toks)))
        # the max of the token scores is at least their mean (the summary score)
        assert got[b] >= math.fsum(toks) / O.BLOCK - 1e-12
    # fewer candidates than blocks: only the first n_cand are scored
    assert len(O.score_blocks_token_max(q, kidx, 2)) == 2


def test_token_max_is_invariant_to_token_order_within_blocks():
    rng = np.random.default_rng(9)
    nb = 4
    kidx = rng.standard_normal((nb * O.BLOCK, O.HEAD_DIM))
    q = rng.standard_normal(O.HEAD_DIM)
    perm = np.concatenate([b * O.BLOCK + rng.permutation(O.BLOCK) for b in range(nb)])
    np.testing.assert_array_equal(O.score_blocks_token_max(q, kidx, nb), O.score_blocks_token_max(q, kidx[perm], nb))


def test_token_max_single_hot_token_wins_its_block():
    # one token aligned with the query lifts its block to the top even though the
    # block mean barely moves (the case the guide's max pool is drawn for)
    rng = np.random.default_rng(10)
    nb = 12
    kidx = rng.standard_normal((nb * O.BLOCK + 10, O.HEAD_DIM))
    q_group = rng.standard_normal((4, O.HEAD_DIM))
    q_idx = q_group.sum(axis=0)
    kidx[5 * O.BLOCK + 17] = 3.0 * q_idx / np.linalg.norm(q_idx) * 4.0
    res = O.select_token_max(q_group, kidx, nb * O.BLOCK + 10, 1, 2)
    assert list(res["selected"]) == [5, nb]          # the hot block and the newest (partial) block
    assert res["n_cand"] == nb


def test_index_key_needles_are_selected_by_token_max():
    from synth import make_decode_inputs, make_index_keys
    inp = make_decode_inputs([64 * 40 + 3], 2, 8, "f32", "contiguous", seed=21)
    ik = make_index_keys(inp, needles=3, seed=22)
    kidx = ik.rows(inp, 0).double().numpy()
    for h in range(2):
        q = inp.q[0, 4 * h:4 * h + 4].double().numpy()
        res = O.select_token_max(q, kidx, inp.lens[0], 3, 4)
        assert sorted(ik.needles[(0, h)]) == [b for b in res["selected"] if b != 40]


def test_prefill_token_max_one_token_tile_equals_decode():
    # a prefill tile holding one token at a block start sees exactly what a
    # decode step with that token as its newest sees: the same index query, the
    # same candidates (the blocks before it) and the same kept block
    rng = np.random.default_rng(23)
    q_start = 64 * 9
    kidx = rng.standard_normal((q_start + 64, O.HEAD_DIM))
    q_tok = rng.standard_normal((1, 4, O.HEAD_DIM))
    for k in (1, 4, 9, 12):
        pre = O.prefill_tile_select_token_max(q_tok, 0, q_start, kidx, k, k + 1)
        dec = O.select_token_max(q_tok[0], kidx, q_start + 1, k, k + 1)
        assert list(pre["selected"]) == list(dec["selected"])
        np.testing.assert_array_equal(pre["scores"], dec["scores"])
        assert pre["diag"] == dec["forced"] == 9


def test_prefill_token_max_brute_force():
    # index query = sum over the tile's tokens and heads; score = max token score
    # of each block before the diagonal; a hot token makes its block win
    rng = np.random.default_rng(24)
    q_tile = rng.standard_normal((7, 3, O.HEAD_DIM))
    kidx = rng.standard_normal((64 * 6, O.HEAD_DIM))
    q_idx = q_tile.sum(axis=(0, 1))
    kidx[64 * 2 + 40] = 5.0 * q_idx / np.linalg.norm(q_idx)
    res = O.prefill_tile_select_token_max(q_tile, 1, 64 * 4, kidx, 1, 3)
    assert res["diag"] == 5
    want = [max(math.fsum(float(q_idx[d]) * float(kidx[b * 64 + t, d]) for d in range(O.HEAD_DIM))
                for t in range(64)) for b in range(5)]
    np.testing.assert_allclose(res["scores"], want, rtol=1e-12, atol=1e-12)
    assert list(res["selected"]) == [2, 5, -1]


# --------------------------------------------------------------------------- attention sink

@pytest.mark.parametrize("trial", range(30))
def test_sink_selection_matches_brute_force(trial):
    rng = np.random.default_rng(100 + trial)
    n = int(rng.integers(1, 10))
    k = int(rng.integers(1, 5))
    scores = rng.integers(-2, 3, size=n).astype(np.float64) if trial % 3 == 0 else rng.standard_normal(n)
    forced = n
    sel = O.select_blocks_sink(scores, k, forced, k + 2, True)
    # the best k of blocks 1..n-1 by (score, lower index), found by subset search
    rest = list(range(1, n))
    want = []
    if rest:
        best = _brute_force_topk([scores[b] for b in rest], k)
        want = [rest[i] for i in best]
    want = sorted(want + [0, forced])
    assert list(sel) == want + [-1] * (k + 2 - len(want))


def test_sink_selection_edge_cases():
    # one block that is both the sink and the newest: kept once
    assert list(O.select_blocks_sink(np.zeros(0), 3, 0, 5, True)) == [0, -1, -1, -1, -1]
    # block 0 a high scorer: never counted among the k scored blocks
    sel = O.select_blocks_sink(np.array([9.0, 1.0, 3.0, 2.0]), 2, 4, 4, True)
    assert list(sel) == [0, 2, 3, 4]
    # without the sink flag on the block the same scores select block 0 as a scored block
    assert list(O.select_blocks(np.array([9.0, 1.0, 3.0, 2.0]), 2, 4, 4)) == [0, 2, 4, -1]


# --------------------------------------------------------------------------- small helpers, pinned directly

def test_store_as_matches_torch_storage():
    # the value a float32 takes once stored: torch's own bf16 / fp32 conversions
    rng = np.random.default_rng(5)
    x = (rng.standard_normal(4096) * np.exp2(rng.integers(-20, 20, 4096))).astype(np.float32)
    want_bf16 = torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(O.store_as(x, "bf16"), want_bf16)
    assert np.array_equal(O.store_as(x, "f32"), x.astype(np.float64))
    with pytest.raises(ValueError):
        O.store_as(x, "f16")


@pytest.mark.parametrize("n,full,total", [(0, 0, 0), (1, 0, 1), (63, 0, 1), (64, 1, 1), (65, 1, 2), (128, 2, 2),
                                          (131072, 2048, 2048), (131071, 2047, 2048)])
def test_block_counts_closed_form(n, full, total):
    assert O.num_full_blocks(n) == full
    assert O.num_blocks(n) == total


def test_boundary_gap_definition():
    # the k-th and (k+1)-th largest scores; None when every candidate is kept
    s = np.array([0.5, 3.0, -1.0, 2.0, 2.0, 7.0])
    assert O.boundary_gap(s, 1) == (7.0, 3.0)
    assert O.boundary_gap(s, 3) == (2.0, 2.0)   # a tie at the boundary
    assert O.boundary_gap(s, 5) == (0.5, -1.0)
    assert O.boundary_gap(s, 6) is None
    assert O.boundary_gap(s, 0) is None
    assert O.boundary_gap(np.array([]), 3) is None


# --------------------------------------------------------------------------- the double-precision reading of pooling

def test_bf16_rounding_from_double_in_one_step():
    # 1 + 2^-8 + 2^-30 lies just above the tie between 1 and 1 + 2^-7; a detour
    # through binary32 would land exactly on the tie and round down to 1
    assert O.round_to_bf16(1.0 + 2.0 ** -8 + 2.0 ** -30) == 1.0 + 2.0 ** -7
    assert O.round_to_bf16(1.0 + 2.0 ** -8) == 1.0                      # the tie itself: to even
    assert O.round_to_bf16(2.0 ** -134) == 0.0                          # half the smallest subnormal: to even
    assert O.round_to_bf16(1.5 * 2.0 ** -134) == 2.0 ** -133
    big = (2.0 - 2.0 ** -7) * 2.0 ** 127                                # largest finite bfloat16
    assert O.round_to_bf16(big) == big
    assert O.round_to_bf16(2.0 ** 128 - 2.0 ** 119) == np.inf           # halfway past it
    assert O.round_to_bf16(2.0 ** 128 - 2.0 ** 119 - 2.0 ** 100) == big


def test_pool_sums_in_double_and_rounds_once():
    d = O.HEAD_DIM
    # fp32 storage: one key 1.0 and 63 keys 2^-25. Summed in binary32 the small
    # keys vanish (each is below half a unit of 1.0); the exact mean is
    # 2^-6 + 63 * 2^-31, whose nearest binary32 value is 2^-6 + 2^-25
    k = np.full((64, d), 2.0 ** -25, dtype=np.float32)
    k[0] = 1.0
    stored, exact = O.pool_block_keys(k, 64, "f32")
    assert np.all(exact == 2.0 ** -6 + 63 * 2.0 ** -31)
    assert np.all(stored == 2.0 ** -6 + 2.0 ** -25)
    # bf16 storage: the mean of 32 ones and 32 values 1 + 2^-7 is the tie
    # 1 + 2^-8 (rounds to the even 1.0); one more key on the high side moves the
    # mean above the tie (rounds up)
    k = np.ones((64, d))
    k[:32] = 1.0 + 2.0 ** -7
    stored, exact = O.pool_block_keys(k, 64, "bf16")
    assert np.all(exact == 1.0 + 2.0 ** -8) and np.all(stored == 1.0)
    k[32] = 1.0 + 2.0 ** -7
    stored, _ = O.pool_block_keys(k, 64, "bf16")
    assert np.all(stored == 1.0 + 2.0 ** -7)


def test_pool_reads_bf16_bits_exactly():
    # a bfloat16 tensor and its float64 values give the same summaries
    g = torch.Generator().manual_seed(3)
    k = torch.randn(64 * 5 + 9, O.HEAD_DIM, generator=g).to(torch.bfloat16)
    a = O.pool_block_keys(k, k.shape[0], "bf16")
    b = O.pool_block_keys(k.double().numpy(), k.shape[0], "bf16")
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


# --------------------------------------------------------------------------- unit-parallel functions agree with the per-unit steps

def test_decode_select_units_matches_the_per_unit_steps():
    from synth import make_decode_inputs
    lens = [64 * 37 + 5, 64 * 20, 63, 64, 64 * 9 + 1]
    inp = make_decode_inputs(lens, 2, 8, "bf16", "contiguous", needles=2, seed=41)
    hkv, grp = 2, 4
    cap = inp.k.shape[2]
    for force_local in (1, 0, 3):
        r = O.decode_select_units(inp.q.view(len(lens) * hkv, grp, -1), inp.k.view(len(lens) * hkv, cap, -1),
                                  [n for n in lens for _ in range(hkv)], "bf16", 5, 7, force_local,
                                  want_scores=True, want_pooled=True)
        for s, n in enumerate(lens):
            for h in range(hkv):
                u = s * hkv + h
                qg, kr = inp.q[s, h * grp:(h + 1) * grp], inp.k[s, h]
                pooled, _ = O.pool_block_keys(kr, n, "bf16")
                assert np.array_equal(r["pooled"][u, :pooled.shape[0]], pooled)
                nb, nbf = O.num_blocks(n), O.num_full_blocks(n)
                n_cand = min(nbf, nb - 1) if force_local & 1 else nbf
                n_cand = max(n_cand, 0)
                scores = O.score_blocks(O.index_query(qg), pooled, n_cand)
                assert np.array_equal(r["scores"][u, :n_cand], scores)
                forced = nb - 1 if force_local & 1 and nb > 0 else None
                if force_local & 2:
                    has0 = nb > 0 and forced != 0
                    want = O.select_blocks_sink(scores, 5, forced, 7, has0) if n_cand > 0 else \
                        O.select_blocks(scores, 5, forced, 7) if not has0 else \
                        np.array(sorted({0} | ({forced} if forced is not None else set())) + [-1] * 6)[:7]
                else:
                    want = O.select_blocks(scores, 5, forced, 7)
                assert list(r["selected"][u]) == list(want), (force_local, s, h)
                ranked = scores[1:] if force_local & 2 and n_cand > 0 else scores
                gap = O.boundary_gap(ranked, 5)
                if gap is None:
                    assert np.isnan(r["gap"][u]).all()
                else:
                    assert tuple(r["gap"][u]) == gap


def test_decode_step_units_matches_decode_unit():
    from synth import make_decode_inputs
    lens = [64 * 40 + 17, 64 * 33, 100]
    inp = make_decode_inputs(lens, 2, 16, "bf16", "contiguous", needles=2, seed=7)
    hkv, grp, cap = 2, 8, inp.k.shape[2]
    mb = cap // 64
    pooled = np.full((len(lens) * hkv, mb, O.HEAD_DIM), np.nan)
    for s, n in enumerate(lens):
        for h in range(hkv):
            p, _ = O.pool_block_keys(inp.k[s, h], n, "bf16")
            pooled[s * hkv + h, :p.shape[0]] = p
    sel, o, lse = O.decode_step_units(inp.q.view(-1, grp, O.HEAD_DIM), pooled, inp.k.view(-1, cap, O.HEAD_DIM),
                                      inp.v.view(-1, cap, O.HEAD_DIM), [n for n in lens for _ in range(hkv)], 6, 8,
                                      1 / math.sqrt(128))
    for s, n in enumerate(lens):
        for h in range(hkv):
            u = s * hkv + h
            ref = O.decode_unit(inp.q[s, h * grp:(h + 1) * grp], inp.k[s, h], inp.v[s, h], n, 6, 8,
                                1 / math.sqrt(128), "bf16")
            assert list(sel[u]) == list(ref["selected"])
            np.testing.assert_allclose(o[u], ref["o"], rtol=0, atol=1e-13)
            np.testing.assert_allclose(lse[u], ref["lse"], rtol=0, atol=1e-13)


# --------------------------------------------------------------------------- chunks that start inside a block

@pytest.mark.parametrize("q_start,n_new", [(0, 1), (0, 64), (128, 200), (100, 1), (100, 28), (100, 29),
                                           (100, 300), (63, 2), (4097, 4096)])
def test_prefill_tiles_partition_the_chunk_by_block(q_start, n_new):
    tiles = O.prefill_tiles(q_start, n_new)
    rows = [r for _, lo, hi in tiles for r in range(lo, hi)]
    assert rows == list(range(n_new))                       # every chunk row once, in order
    assert [j for j, _, _ in tiles] == list(range(len(tiles)))
    for j, lo, hi in tiles:
        assert 0 < hi - lo <= 64
        blocks = {(q_start + r) // 64 for r in range(lo, hi)}
        assert blocks == {q_start // 64 + j}                # one block per tile: the diagonal one
    if q_start % 64 == 0:
        assert [(lo, hi) for _, lo, hi in tiles] == [(64 * j, min(n_new, 64 * j + 64)) for j in range(len(tiles))]
    assert O.prefill_tiles(q_start, 0) == []


@pytest.mark.parametrize("pos", [64 * 9, 64 * 9 + 1, 64 * 9 + 37, 64 * 9 + 63])
def test_one_token_chunk_equals_the_decode_step(pos):
    # a chunk of one token at position pos sees what a decode step whose newest
    # token sits at pos sees: same index query, candidates, kept block, output
    rng = np.random.default_rng(pos)
    k = rng.standard_normal((64 * 11, O.HEAD_DIM))
    v = rng.standard_normal((64 * 11, O.HEAD_DIM))
    q = rng.standard_normal((1, 4, O.HEAD_DIM))
    pooled, _ = O.pool_block_keys(k, pos + 1, "f32")
    ((j, lo, hi),) = O.prefill_tiles(pos, 1)
    for kk in (1, 3, 9, 20):
        pre = O.prefill_tile_select(q[lo:hi], j, pos, pooled, kk, kk + 1)
        dec = O.decode_unit(q[0], k, v, pos + 1, kk, kk + 1, 1 / math.sqrt(128), "f32", pooled=pooled)
        assert list(pre["selected"]) == list(dec["selected"]) and pre["diag"] == dec["forced"]
        np.testing.assert_array_equal(pre["scores"], dec["scores"])
        o, lse = O.prefill_rows(q, [pos], k, v, pos + 1, pre["selected"], 1 / math.sqrt(128))
        np.testing.assert_allclose(o[0], dec["o"], rtol=0, atol=1e-14)
        np.testing.assert_allclose(lse[0], dec["lse"], rtol=0, atol=1e-14)


@pytest.mark.parametrize("q_start,n_new", [(100, 90), (63, 70), (130, 5)])
def test_unaligned_chunk_with_every_block_equals_dense(q_start, n_new):
    rng = np.random.default_rng(q_start + n_new)
    total = q_start + n_new
    k = rng.standard_normal((total, O.HEAD_DIM))
    v = rng.standard_normal((total, O.HEAD_DIM))
    q = rng.standard_normal((n_new, 2, O.HEAD_DIM))
    pooled, _ = O.pool_block_keys(k, total, "f32")
    for j, lo, hi in O.prefill_tiles(q_start, n_new):
        sel = O.prefill_tile_select(q[lo:hi], j, q_start, pooled, k_scored=64, k_total=6)
        assert [b for b in sel["selected"] if b >= 0] == list(range(sel["diag"] + 1))
        pos = q_start + np.arange(lo, hi)
        o, lse = O.prefill_rows(q[lo:hi], pos, k, v, total, sel["selected"], 0.125)
        for i in range(hi - lo):
            od, ld = O.dense_gqa(q[lo + i], k, v, pos[i], 0.125)
            np.testing.assert_allclose(o[i], od, rtol=0, atol=1e-12)
            np.testing.assert_allclose(lse[i], ld, rtol=0, atol=1e-12)


def test_chunk_split_at_a_block_boundary_keeps_every_list():
    # a tile's list depends only on its own queries and the summaries before
    # it, so a chunk split at a block boundary gives the same lists
    rng = np.random.default_rng(77)
    q_start, n_new, cut = 100, 250, 28 + 64 * 2        # 100 + 156 = 256: a block boundary
    total = q_start + n_new
    k = rng.standard_normal((total, O.HEAD_DIM))
    q = rng.standard_normal((n_new, 3, O.HEAD_DIM))
    pooled, _ = O.pool_block_keys(k, total, "f32")
    whole = [O.prefill_tile_select(q[lo:hi], j, q_start, pooled, 2, 3)["selected"]
             for j, lo, hi in O.prefill_tiles(q_start, n_new)]
    parts = [O.prefill_tile_select(q[lo:hi], j, q_start, pooled, 2, 3)["selected"]
             for j, lo, hi in O.prefill_tiles(q_start, cut)]
    parts += [O.prefill_tile_select(q[cut + lo:cut + hi], j, q_start + cut, pooled, 2, 3)["selected"]
              for j, lo, hi in O.prefill_tiles(q_start + cut, n_new - cut)]
    assert len(whole) == len(parts)
    for a, b in zip(whole, parts):
        assert list(a) == list(b)


@pytest.mark.parametrize("q_start,n_new", [(128, 150), (100, 90)])
def test_prefill_tile_units_matches_the_per_unit_steps(q_start, n_new):
    rng = np.random.default_rng(q_start)
    hkv, hq = 2, 6
    total = q_start + n_new
    k = rng.standard_normal((hkv, total, O.HEAD_DIM))
    v = rng.standard_normal((hkv, total, O.HEAD_DIM))
    q = rng.standard_normal((n_new, hq, O.HEAD_DIM))
    mb = O.num_blocks(total)
    pooled = np.full((hkv, mb, O.HEAD_DIM), np.nan)
    for h in range(hkv):
        p, _ = O.pool_block_keys(k[h], total, "f32")
        pooled[h, :p.shape[0]] = p
    tiles = O.prefill_tiles(q_start, n_new)
    units = [(j, h) for j, _, _ in tiles for h in range(hkv)]
    sel, o, lse = O.prefill_tile_units(units, q_start, q, pooled, k, v, 2, 3, 0.125)
    part = {j: (lo, hi) for j, lo, hi in tiles}
    for u, (j, h) in enumerate(units):
        lo, hi = part[j]
        grp = hq // hkv
        ref = O.prefill_tile_select(q[lo:hi, h * grp:(h + 1) * grp], j, q_start, pooled[h], 2, 3)
        assert list(sel[u]) == list(ref["selected"])
        ro, rl = O.prefill_rows(q[lo:hi, h * grp:(h + 1) * grp], q_start + np.arange(lo, hi), k[h], v[h], total,
                                ref["selected"], 0.125)
        np.testing.assert_allclose(o[lo:hi, h * grp:(h + 1) * grp], ro, rtol=0, atol=1e-13)
        np.testing.assert_allclose(lse[lo:hi, h * grp:(h + 1) * grp], rl, rtol=0, atol=1e-13)

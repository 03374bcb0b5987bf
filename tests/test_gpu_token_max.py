"""GPU parity of the guide-literal Step 1 (token-level index scores against a
shared index-key head, block max pool) against the CPU oracle, through the C
ABI: msa_select_topk_blocks with MSA_SCORE_TOKEN_MAX, and the whole decode step
(msa_sparse_decode_step) in that mode. Small cases on every unit, a
128K-token x 8 batch on sampled units.
"""
import numpy as np
import pytest
import torch

from oracle import msa_oracle as O
from synth import make_decode_inputs, make_index_keys
from tests.parity import SCALE, SelectionStats, check_lse, check_output, check_selection, to64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev(lib):
    assert torch.cuda.is_available()
    return torch.device("cuda:0")


def run_token_max(inp, ik, k_scored, k_total, step=False, sink=False):
    from sparse_attention_step_gb300 import msa
    dev = inp.q.device
    desc = msa.kv_desc(inp.k, inp.v, inp.seq_lens, inp.page_table)
    hq = inp.num_q_heads
    ops = [msa.MSA_OP_SELECT, msa.MSA_OP_DECODE, msa.MSA_OP_DECODE_STEP]
    ws = msa.Workspace(max(msa.msa_workspace_size(op, desc, hq, 1, k_total) for op in ops), dev)
    b, hkv = inp.batch, inp.num_kv_heads
    max_blocks = desc.max_tokens // 64 if desc.layout == 0 else desc.max_pages_per_seq
    idx = torch.full((b, hkv, k_total), -7, dtype=torch.int32, device=dev)
    scores = torch.full((b * hkv, max_blocks), float("nan"), dtype=torch.float32, device=dev)
    out = torch.full_like(inp.q, float("nan"))
    lse = torch.full((b, hq), float("nan"), dtype=torch.float32, device=dev)
    cfg = msa.select_cfg(k_scored, mode=msa.MSA_SCORE_TOKEN_MAX, sink=sink)
    if step:
        msa.msa_sparse_decode_step(inp.q, hq, ik.kidx, desc, cfg, idx, k_total, SCALE, out, lse, ws.buf, ws.nbytes)
        scores = None
    else:
        msa.msa_select_topk_blocks(inp.q, hq, 1, ik.kidx, desc, cfg, idx, k_total, scores, ws.buf, ws.nbytes)
        msa.msa_sparse_attn_decode(inp.q, hq, desc, idx, k_total, SCALE, out, lse, ws.buf, ws.nbytes)
    torch.cuda.synchronize()
    return dict(idx=idx, scores=scores, out=out, lse=lse, status=msa.msa_read_device_status(ws.buf))


def verify(inp, ik, res, units, k_scored, k_total, stats=None):
    grp = inp.num_q_heads // inp.num_kv_heads
    for s, h in units:
        n = inp.lens[s]
        qg = to64(inp.q[s, h * grp:(h + 1) * grp])
        kidx = to64(ik.rows(inp, s))
        ref = O.select_token_max(qg, kidx, n, k_scored, k_total)
        if res["scores"] is not None and ref["n_cand"] > 0:
            got = to64(res["scores"][s * inp.num_kv_heads + h, :ref["n_cand"]])
            # fp32 dot products (bf16 head + remainder of the index query) vs fp64
            lim = 1e-5 * np.maximum(1.0, np.abs(ref["scores"])) + 1e-5 * np.abs(ref["q_idx"]).sum()
            assert (np.abs(got - ref["scores"]) <= lim).all(), f"token-max scores differ at unit {(s, h)}"
        got_idx = res["idx"][s, h].cpu().numpy()
        check_selection(got_idx, ref["scores"], k_scored, ref["forced"], k_total, stats, ik.needles.get((s, h), []))
        toks = O.tokens_of_blocks(got_idx, n)
        o, lse, _ = O.attend(qg, to64(inp.kv_rows(s, h, "k")), to64(inp.kv_rows(s, h, "v")), toks, SCALE)
        check_output(to64(res["out"][s, h * grp:(h + 1) * grp]), o, inp.dtype, f"unit {(s, h)}")
        check_lse(to64(res["lse"][s, h * grp:(h + 1) * grp]), lse)


@pytest.mark.parametrize("layout", ["contiguous", "paged"])
@pytest.mark.parametrize("hkv,hq", [(2, 16), (1, 8), (8, 64)])
def test_token_max_select_and_attend(dev, layout, hkv, hq):
    inp = make_decode_inputs([64 * 90 + 13, 64 * 33, 64 * 7 + 1], hkv, hq, "bf16", layout, seed=41, device=dev)
    ik = make_index_keys(inp, needles=2, seed=42)
    res = run_token_max(inp, ik, 6, 7)
    assert res["status"] == 0
    verify(inp, ik, res, [(s, h) for s in range(inp.batch) for h in range(hkv)], 6, 7)


@pytest.mark.parametrize("layout", ["contiguous", "paged"])
@pytest.mark.parametrize("hkv,hq", [(4, 32), (2, 8), (1, 8)])
def test_token_max_through_the_decode_step(dev, layout, hkv, hq):
    """The decode step in token-max mode: the scores from their own kernel,
    then the fused step reads them in place of scoring summaries. Its lists
    equal those of the two-kernel form (the same scores and keys) and its
    outputs the oracle's; group sizes 8 and 4, one to four KV heads."""
    inp = make_decode_inputs([64 * 200 + 5, 64 * 64, 64 * 3 + 1], hkv, hq, "bf16", layout, seed=43, device=dev)
    ik = make_index_keys(inp, needles=3, seed=44)
    res = run_token_max(inp, ik, 11, 12, step=True)
    ref = run_token_max(inp, ik, 11, 12)
    assert res["status"] == 0 and ref["status"] == 0
    assert torch.equal(res["idx"], ref["idx"])
    verify(inp, ik, res, [(s, h) for s in range(3) for h in range(hkv)], 11, 12)


def test_token_max_decode_step_sink(dev):
    from tests.test_gpu_sink import check_sink_row
    inp = make_decode_inputs([64 * 150 + 9, 64 * 40], 2, 16, "bf16", "contiguous", seed=47, device=dev)
    ik = make_index_keys(inp, needles=2, seed=48)
    res = run_token_max(inp, ik, 7, 9, step=True, sink=True)
    ref = run_token_max(inp, ik, 7, 9, sink=True)
    assert res["status"] == 0 and ref["status"] == 0
    assert torch.equal(res["idx"], ref["idx"])
    grp = inp.num_q_heads // inp.num_kv_heads
    for s in range(2):
        kidx = to64(ik.rows(inp, s))
        for h in range(2):
            r = O.select_token_max(to64(inp.q[s, h * grp:(h + 1) * grp]), kidx, inp.lens[s], 7, 9)
            check_sink_row(res["idx"][s, h].cpu().numpy(), r["scores"], 7, r["forced"], 9, True)


@pytest.mark.parametrize("step", [False, True])
def test_token_max_short_and_empty_sequences(dev, step):
    # no candidates (one partial block), exactly one complete block, and k above the candidates
    inp = make_decode_inputs([40, 64, 64 * 3 + 2], 2, 16, "bf16", "contiguous", seed=45, device=dev)
    ik = make_index_keys(inp, seed=46)
    res = run_token_max(inp, ik, 5, 6, step=step)
    assert res["status"] == 0
    verify(inp, ik, res, [(s, h) for s in range(3) for h in range(2)], 5, 6)


def test_token_max_decode_128k_sampled(dev):
    """8 sequences x 131072 tokens, 8 KV / 64 query heads, top-31 + newest: the
    benchmark's shape, units sampled across the batch."""
    inp = make_decode_inputs([131072] * 8, 8, 64, "bf16", "contiguous", seed=1006, device=dev)
    ik = make_index_keys(inp, needles=8, seed=1007)
    res = run_token_max(inp, ik, 31, 32)
    assert res["status"] == 0
    stats = SelectionStats()
    verify(inp, ik, res, [(0, 0), (3, 5), (7, 7)], 31, 32, stats)
    # the benchmark's launch: the fused step, its lists equal to the two-kernel form's on every unit
    res_step = run_token_max(inp, ik, 31, 32, step=True)
    assert res_step["status"] == 0
    assert torch.equal(res_step["idx"], res["idx"])
    verify(inp, ik, res_step, [(1, 2), (6, 0)], 31, 32)
    del inp, ik
    torch.cuda.empty_cache()


# --------------------------------------------------------------------------- prefill tiles

def run_token_max_prefill(inp, ik, k_scored, k_total, sink=False):
    from sparse_attention_step_gb300 import msa
    c = inp.cache
    dev = inp.q.device
    desc = msa.kv_desc(c.k, c.v, c.seq_lens, c.page_table)
    hq, hkv = c.num_q_heads, c.num_kv_heads
    n_tiles = msa.varlen_tiles(inp.q_counts, inp.q_starts)
    ws = msa.Workspace(msa.msa_workspace_size(msa.MSA_OP_SELECT_PREFILL, desc, hq, 64 * n_tiles, k_total), dev)
    max_blocks = desc.max_tokens // 64 if desc.layout == 0 else desc.max_pages_per_seq
    idx = torch.full((n_tiles, hkv, k_total), -7, dtype=torch.int32, device=dev)
    scores = torch.full((n_tiles * hkv, max_blocks), float("nan"), dtype=torch.float32, device=dev)
    cfg = msa.select_cfg(k_scored, True, 64, mode=msa.MSA_SCORE_TOKEN_MAX, sink=sink)
    msa.msa_select_topk_blocks_varlen(inp.q, hq, inp.q_starts, inp.q_counts, ik.kidx, desc, cfg, idx, k_total, scores,
                                      ws.buf, ws.nbytes)
    torch.cuda.synchronize()
    return dict(idx=idx, scores=scores, status=msa.msa_read_device_status(ws.buf))


@pytest.mark.parametrize("layout,hq,hkv,shift", [("contiguous", 64, 8, 0), ("paged", 16, 4, 0), ("contiguous", 8, 1, 0),
                                                 ("contiguous", 64, 8, 37), ("paged", 16, 4, 11)])
def test_token_max_prefill_tiles(dev, layout, hq, hkv, shift):
    # ragged chunks over a shared index-key head: one spanning two groups of 16
    # tiles (and two of 8), one from an empty prefix, a 5-token one; with a
    # shift the chunks start inside blocks
    from synth import make_prefill_batch_inputs
    q_starts = [64 * 23 + shift, 0, 64 * 7 + shift, 64 * 40 + shift]
    q_counts = [64 * 2 + 17, 64 * 3, 5, 64 * 17 + 1]
    inp = make_prefill_batch_inputs(q_starts, q_counts, hkv, hq, "bf16", layout, seed=95, device=dev)
    ik = make_index_keys(inp.cache, needles=2, seed=96)
    k_scored, k_total = 6, 7
    res = run_token_max_prefill(inp, ik, k_scored, k_total)
    assert res["status"] == 0
    grp = hq // hkv
    for s, (q0, n) in enumerate(zip(q_starts, q_counts)):
        kidx = to64(ik.rows(inp.cache, s))
        qs = inp.q_rows(s)
        for j, lo, hi in O.prefill_tiles(q0, n):
            g = inp.tile_off[s] + j
            for h in range(hkv):
                q_tile = to64(qs[lo:hi, h * grp:(h + 1) * grp])
                ref = O.prefill_tile_select_token_max(q_tile, j, q0, kidx, k_scored, k_total)
                if ref["diag"] > 0:
                    got = to64(res["scores"][g * hkv + h, :ref["diag"]])
                    lim = 1e-5 * np.maximum(1.0, np.abs(ref["scores"])) + 1e-5 * np.abs(ref["q_idx"]).sum()
                    assert (np.abs(got - ref["scores"]) <= lim).all(), f"token-max scores differ, seq {s} tile {j}"
                check_selection(res["idx"][g, h].cpu().numpy(), ref["scores"], k_scored, ref["diag"], k_total)


def test_token_max_prefill_sink(dev):
    from synth import make_prefill_batch_inputs
    from tests.test_gpu_sink import check_sink_row
    inp = make_prefill_batch_inputs([64 * 12], [64 * 2 + 3], 2, 16, "bf16", "contiguous", seed=97, device=dev)
    ik = make_index_keys(inp.cache, needles=1, seed=98)
    res = run_token_max_prefill(inp, ik, 4, 6, sink=True)
    assert res["status"] == 0
    kidx = to64(ik.rows(inp.cache, 0))
    for j in range(3):
        for h in range(2):
            q_tile = to64(inp.q[64 * j:min(131, 64 * j + 64), 8 * h:8 * h + 8])
            ref = O.prefill_tile_select_token_max(q_tile, j, 64 * 12, kidx, 4, 6)
            check_sink_row(res["idx"][j, h].cpu().numpy(), ref["scores"], 4, ref["diag"], 6, True)


def test_token_max_prefill_8k_on_128k_sampled(dev):
    """The benchmark's chunk (8192 new tokens on a 131072-token prefix, 8 KV /
    64 query heads, top-32 + diagonal) in token-max mode, in the launch the
    benchmark times: the scores and selections of 32 (tile, head) units spread
    over the chunk and the heads against the oracle."""
    from synth import make_prefill_batch_inputs
    from tests.parity import record
    q0, n_new, k_scored, k_total = 131072, 8192, 32, 33
    inp = make_prefill_batch_inputs([q0], [n_new], 8, 64, "bf16", "contiguous", seed=1004, device=dev)
    ik = make_index_keys(inp.cache, needles=0, seed=4007)
    res = run_token_max_prefill(inp, ik, k_scored, k_total)
    assert res["status"] == 0
    kidx = to64(ik.rows(inp.cache, 0))
    qs = inp.q_rows(0)
    tiles = list(O.prefill_tiles(q0, n_new))
    stats = SelectionStats()
    for i in range(32):
        j, lo, hi = tiles[(i * 37) % len(tiles)]
        h = i % 8
        q_tile = to64(qs[lo:hi, 8 * h:8 * h + 8])
        ref = O.prefill_tile_select_token_max(q_tile, j, q0, kidx, k_scored, k_total)
        got = to64(res["scores"][j * 8 + h, :ref["diag"]])
        lim = 1e-5 * np.maximum(1.0, np.abs(ref["scores"])) + 1e-5 * np.abs(ref["q_idx"]).sum()
        assert (np.abs(got - ref["scores"]) <= lim).all(), f"token-max scores differ, tile {j} head {h}"
        check_selection(res["idx"][j, h].cpu().numpy(), ref["scores"], k_scored, ref["diag"], k_total, stats)
    record("prefill_8k_on_128k token-max (sampled)", units=stats.units, near_ties=stats.near_ties)
    del inp, ik, res
    torch.cuda.empty_cache()

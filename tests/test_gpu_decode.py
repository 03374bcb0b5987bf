"""GPU parity of the decode path against the CPU oracle, through the C ABI.

Small cases are compared on every unit. The full-size workloads (128K x 8,
1M x 1, ragged paged x 32), in the launch configuration the benchmark uses,
have their selection checked on every unit (the oracle pools, scores and
ranks all of them) and their attention outputs element by element on 16 units
spread over sequences and heads (all 8 at 1M). Near-tie and summary-difference
counts are printed.
"""
import math

import numpy as np
import pytest
import torch

from oracle import msa_oracle as O
from synth import make_decode_inputs, make_workload, WORKLOADS
from tests.parity import (SCALE, PoolStats, SelectionStats, check_lse, check_output, check_pooled, check_selection,
                          record, to64)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev(lib):
    assert torch.cuda.is_available()
    return torch.device("cuda:0")


def run_decode(inp, k_scored, k_total, force_local=True, want_scores=True, dense=False):
    from sparse_attention_step_gb300 import msa
    dev = inp.q.device
    desc = msa.kv_desc(inp.k, inp.v, inp.seq_lens, inp.page_table)
    hq = inp.num_q_heads
    ops = [msa.MSA_OP_POOL, msa.MSA_OP_SELECT, msa.MSA_OP_DECODE, msa.MSA_OP_DENSE_DECODE]
    need = max(msa.msa_workspace_size(op, desc, hq, 1, k_total) for op in ops)
    ws = msa.Workspace(need, dev)
    pooled = torch.full(msa.pooled_shape(desc), float("nan"), dtype=inp.k.dtype, device=dev)
    b, hkv = inp.batch, inp.num_kv_heads
    idx = torch.full((b, hkv, k_total), -7, dtype=torch.int32, device=dev)
    max_blocks = desc.max_tokens // 64 if desc.layout == 0 else desc.max_pages_per_seq
    scores = torch.empty(b * hkv, max_blocks, dtype=torch.float32, device=dev) if want_scores else None
    out = torch.full_like(inp.q, float("nan"))
    lse = torch.full((b, hq), float("nan"), dtype=torch.float32, device=dev)
    msa.msa_pool_block_keys(desc, 0, -1, pooled, ws.buf, ws.nbytes)
    msa.msa_select_topk_blocks(inp.q, hq, 1, pooled, desc, msa.select_cfg(k_scored, force_local), idx, k_total,
                               scores, ws.buf, ws.nbytes)
    msa.msa_sparse_attn_decode(inp.q, hq, desc, idx, k_total, SCALE, out, lse, ws.buf, ws.nbytes)
    res = dict(pooled=pooled, idx=idx, out=out, lse=lse, scores=scores, desc=desc, ws=ws)
    if dense:
        dout = torch.full_like(inp.q, float("nan"))
        dlse = torch.full((b, hq), float("nan"), dtype=torch.float32, device=dev)
        msa.msa_dense_gqa_decode(inp.q, hq, desc, SCALE, dout, dlse, ws.buf, ws.nbytes)
        res.update(dense_out=dout, dense_lse=dlse)
    torch.cuda.synchronize()
    res["status"] = msa.msa_read_device_status(ws.buf)
    return res


def gpu_pooled_rows(inp, res, s, h):
    n = inp.lens[s] // 64
    return to64(res["pooled"][s, h, :n])


def verify_units(inp, res, units, k_scored, k_total, force_local=True, stats=None, check_dense=False,
                 check_needles=True, pool_stats=None):
    grp = inp.num_q_heads // inp.num_kv_heads
    store = inp.dtype
    for s, h in units:
        n = inp.lens[s]
        qg = inp.q[s, h * grp:(h + 1) * grp].cpu()
        kr = inp.kv_rows(s, h, "k").cpu()
        vr = inp.kv_rows(s, h, "v").cpu()
        ref = O.decode_unit(qg, kr, vr, n, k_scored, k_total, SCALE, store, force_local=force_local)
        # pooled summaries: within one bf16 step of the oracle's double-precision mean
        got_pool = gpu_pooled_rows(inp, res, s, h)
        _, exact = O.pool_block_keys(kr, n, store)
        check_pooled(got_pool, ref["pooled"], exact, store, to64(kr) if store == "f32" else None, pool_stats,
                     f"pooled keys of unit {(s, h)}")
        # raw scores (fp32 dot products of the library's summaries vs double of
        # the oracle's): tight relative agreement, plus what the summaries differ by
        if res["scores"] is not None and ref["n_cand"] > 0:
            nc = ref["n_cand"]
            got_sc = to64(res["scores"][s * inp.num_kv_heads + h, :nc])
            dpool = np.abs(got_pool[:nc] - ref["pooled"][:nc]) @ np.abs(ref["q_idx"])
            lim = 1e-5 * np.maximum(1.0, np.abs(ref["scores"])) + 1e-5 * np.abs(ref["q_idx"]).sum() + dpool
            assert (np.abs(got_sc - ref["scores"]) <= lim).all(), f"scores differ at unit {(s, h)}"
        got_idx = res["idx"][s, h].cpu().numpy()
        needles = inp.needles.get((s, h), []) if check_needles else []
        check_selection(got_idx, ref["scores"], k_scored, ref["forced"], k_total, stats, needles)
        # attention over the GPU's (validated) selection
        toks = O.tokens_of_blocks(got_idx, n)
        o_ref, lse_ref, _ = O.attend(qg, kr, vr, toks, SCALE)
        got = to64(res["out"][s, h * grp:(h + 1) * grp])
        if len(toks) == 0:
            assert np.all(got == 0)
            assert np.all(np.isneginf(to64(res["lse"][s, h * grp:(h + 1) * grp])))
        else:
            check_output(got, o_ref, store, f"decode unit {(s, h)}")
            check_lse(to64(res["lse"][s, h * grp:(h + 1) * grp]), lse_ref)
        if check_dense and n > 0:
            od, ld = O.dense_gqa(qg, kr, vr, n - 1, SCALE)
            check_output(to64(res["dense_out"][s, h * grp:(h + 1) * grp]), od, store, f"dense unit {(s, h)}")
            check_lse(to64(res["dense_lse"][s, h * grp:(h + 1) * grp]), ld, "dense lse")


def seq_unit_rows(inp, s):
    """[Hkv, capacity, D] keys of sequence s in logical token order (on the
    device; paged caches gathered through the page table)."""
    if inp.layout == "contiguous":
        return inp.k[s]
    n_pages = -(-inp.lens[s] // 64)
    pages = inp.page_table[s, :n_pages].long()
    return inp.k[pages].permute(1, 0, 2, 3).reshape(inp.num_kv_heads, n_pages * 64, -1)


def verify_selection_all_units(inp, idx, k_scored, k_total, force_local=1, stats=None):
    """The selection rule on every (sequence, KV head) unit: the oracle pools
    each unit's keys, scores its candidates and ranks them; the library's list
    must match exactly, or hold a valid near-tie set."""
    grp = inp.num_q_heads // inp.num_kv_heads
    idx = idx.cpu().numpy()
    hkv = inp.num_kv_heads
    for s in range(inp.batch):
        q = inp.q[s].view(hkv, grp, -1).cpu()
        k = seq_unit_rows(inp, s).cpu()
        r = O.decode_select_units(q, k, [inp.lens[s]] * hkv, inp.dtype, k_scored, k_total, force_local,
                                  want_scores=True)
        nb = -(-inp.lens[s] // 64)
        for h in range(hkv):
            n_cand = min(inp.lens[s] // 64, nb - 1) if force_local & 1 else inp.lens[s] // 64
            scores = r["scores"][h, :max(n_cand, 0)]
            forced = nb - 1 if (force_local & 1) and nb > 0 else None
            check_selection(idx[s, h], scores, k_scored, forced, k_total, stats, inp.needles.get((s, h), []))
            assert list(r["selected"][h]) == list(O.select_blocks(scores, k_scored, forced, k_total))


def spread_units(inp, n=16):
    """Up to n distinct (sequence, head) units spread over sequences and heads."""
    b, hkv = inp.batch, inp.num_kv_heads
    units = []
    for i in range(b * hkv):
        u = ((i * 7) % b, (i + i // b) % hkv) if b > 1 else (0, i % hkv)
        if u not in units:
            units.append(u)
        if len(units) == n:
            break
    return units


def all_units(inp):
    return [(s, h) for s in range(inp.batch) for h in range(inp.num_kv_heads)]


# --------------------------------------------------------------------------- small cases, every unit

@pytest.mark.parametrize("layout", ["contiguous", "paged"])
@pytest.mark.parametrize("hq,hkv", [(16, 2), (8, 8), (8, 2)])
def test_decode_small_bf16(dev, layout, hq, hkv):
    lens = [64 * 37 + 5, 64 * 20, 63, 64, 64 * 300 + 1]
    inp = make_decode_inputs(lens, hkv, hq, "bf16", layout, needles=2, seed=11 + hq, device=dev)
    res = run_decode(inp, 5, 6, dense=True)
    assert res["status"] == 0
    stats = SelectionStats()
    verify_units(inp, res, all_units(inp), 5, 6, stats=stats, check_dense=True)


def test_decode_tiny_f32_workload(dev):
    """The 4096-token fp32 workload (1 KV head, 4 query heads, top-8 + last)."""
    w = WORKLOADS["tiny_decode"]
    inp = make_workload("tiny_decode", device=dev)
    res = run_decode(inp, w["k_scored"], w["k_total"], dense=True)
    assert res["status"] == 0
    verify_units(inp, res, all_units(inp), w["k_scored"], w["k_total"], check_dense=True)


def test_decode_f32_ragged_paged(dev):
    lens = [64 * 9 + 3, 200, 64 * 12]
    inp = make_decode_inputs(lens, 2, 8, "f32", "paged", needles=1, seed=5, device=dev)
    res = run_decode(inp, 3, 5, dense=True)
    assert res["status"] == 0
    verify_units(inp, res, all_units(inp), 3, 5, check_dense=True)


def test_decode_many_splits_and_chunks(dev):
    """Spans several scorer chunks and several attention splits per unit."""
    lens = [64 * 700 + 13, 64 * 1100]
    inp = make_decode_inputs(lens, 2, 16, "bf16", "contiguous", needles=6, seed=3, device=dev)
    res = run_decode(inp, 40, 48, dense=True)
    assert res["status"] == 0
    verify_units(inp, res, all_units(inp), 40, 48, check_dense=True)


@pytest.mark.parametrize("layout", ["contiguous", "paged"])
def test_decode_long_lists_few_units(dev, layout):
    """Few units with long lists: each unit's list over a 16-CTA cluster with
    a long slice per CTA (the two-quartet attention kernel), ragged lengths."""
    lens = [64 * 2000 + 29]
    inp = make_decode_inputs(lens, 8, 64, "bf16", layout, needles=4, seed=41, device=dev)
    res = run_decode(inp, 300, 301, dense=True)
    assert res["status"] == 0
    verify_units(inp, res, all_units(inp), 300, 301, check_dense=True)


@pytest.mark.parametrize("k_scored", [0, 1, 10_000])
def test_decode_k_extremes(dev, k_scored):
    lens = [64 * 30 + 7, 64 * 5]
    inp = make_decode_inputs(lens, 2, 8, "bf16", "contiguous", seed=9, device=dev)
    k_total = min(k_scored, 64 * 31) + 1
    res = run_decode(inp, k_scored, k_total, dense=True)
    assert res["status"] == 0
    verify_units(inp, res, all_units(inp), k_scored, k_total, check_dense=True)
    if k_scored >= 10_000:  # every block selected: sparse output equals dense
        d = (res["out"].float() - res["dense_out"].float()).abs().max().item()
        assert d <= 2e-2


@pytest.mark.parametrize("layout", ["contiguous", "paged"])
def test_decode_one_workspace_for_every_step(dev, layout):
    """Select keeps its scores in the workspace (no scores_out) and decode
    then uses the same workspace, twice in a row: the split-K counters must
    survive the scorer's scratch and reset themselves."""
    lens = [64 * 300 + 5, 64 * 77, 64 * 1024]
    inp = make_decode_inputs(lens, 2, 16, "bf16", layout, needles=3, seed=31, device=dev)
    for _ in range(2):
        res = run_decode(inp, 47, 48, want_scores=False, dense=True)
        assert res["status"] == 0
        verify_units(inp, res, all_units(inp), 47, 48, check_dense=True)


def test_decode_without_forced_block(dev):
    lens = [64 * 20, 64 * 20 + 9]
    inp = make_decode_inputs(lens, 2, 8, "bf16", "contiguous", needles=2, seed=4, device=dev)
    res = run_decode(inp, 4, 4, force_local=False)
    assert res["status"] == 0
    verify_units(inp, res, all_units(inp), 4, 4, force_local=False)


def test_decode_empty_sequence(dev):
    lens = [0, 64 * 3]
    inp = make_decode_inputs(lens, 1, 4, "bf16", "contiguous", seed=1, device=dev, max_tokens=256)
    res = run_decode(inp, 2, 3, dense=True)
    assert res["status"] == 0
    assert res["idx"][0].cpu().tolist() == [[-1, -1, -1]]
    assert torch.all(res["out"][0] == 0)
    assert torch.all(torch.isneginf(res["lse"][0]))
    verify_units(inp, res, [(1, 0)], 2, 3, check_dense=True)


def test_gqa_diagram_structure(dev):
    """Six query heads over two KV heads (the diagram): heads 1-3 use list I1,
    heads 4-6 use I2, and each list holds its own group's needle."""
    inp = make_decode_inputs([64 * 40], 2, 6, "bf16", "contiguous", needles=1, seed=21, device=dev)
    res = run_decode(inp, 3, 4)
    idx = res["idx"][0].cpu().numpy()
    assert inp.needles[(0, 0)][0] in idx[0] and inp.needles[(0, 1)][0] in idx[1]
    verify_units(inp, res, all_units(inp), 3, 4)


def test_device_status_bad_page(dev):
    from sparse_attention_step_gb300 import msa
    inp = make_decode_inputs([64 * 8, 64 * 4], 1, 4, "bf16", "paged", seed=2, device=dev)
    inp.page_table[1, 2] = inp.k.shape[0] + 5  # out of range: skipped and reported
    res = run_decode(inp, 2, 3)
    assert res["status"] == msa.MSA_ERR_DEVICE_BOUNDS
    res2 = run_decode(make_decode_inputs([64 * 8], 1, 4, "bf16", "paged", seed=2, device=dev), 2, 3)
    assert res2["status"] == 0


def test_device_status_length_over_capacity(dev):
    from sparse_attention_step_gb300 import msa
    inp = make_decode_inputs([64 * 8], 1, 4, "bf16", "contiguous", seed=2, device=dev)
    inp.seq_lens[0] = 64 * 8 + 100  # beyond the cache capacity: clamped and reported
    res = run_decode(inp, 2, 3)
    assert res["status"] == msa.MSA_ERR_DEVICE_BOUNDS


def test_bounded_wait_gives_up_and_reports(dev):
    # a wait on a barrier that nothing signals gives up after its limit and
    # records MSA_ERR_TIMEOUT (no fault, no trap); the context stays usable
    from sparse_attention_step_gb300 import msa
    ws = msa.Workspace(4096, dev)
    msa.msa_selftest_wait_timeout(ws.buf, ws.nbytes, 2_000_000)  # about a millisecond
    torch.cuda.synchronize()
    assert msa.msa_read_device_status(ws.buf) == msa.MSA_ERR_TIMEOUT
    assert msa.msa_read_device_status(ws.buf) == 0  # reading clears the word
    res = run_decode(make_decode_inputs([64 * 8 + 3], 1, 4, "bf16", "contiguous", seed=4, device=dev), 2, 3)
    assert res["status"] == 0
    with pytest.raises(msa.MsaError):
        msa.msa_selftest_wait_timeout(ws.buf, ws.nbytes, 10)  # below the smallest limit


# --------------------------------------------------------------------------- full-size workloads, sampled units

def _full(name):
    w = WORKLOADS[name]
    dev = torch.device("cuda:0")
    inp = make_workload(name, device=dev)
    # scores stay in the workspace, as in the benchmark
    res = run_decode(inp, w["k_scored"], w["k_total"], dense=True, want_scores=False)
    assert res["status"] == 0
    stats, pstats = SelectionStats(), PoolStats()
    verify_selection_all_units(inp, res["idx"], w["k_scored"], w["k_total"], stats=stats)
    verify_units(inp, res, spread_units(inp), w["k_scored"], w["k_total"], check_dense=True, pool_stats=pstats)
    record(f"{name} (select + attend)", units=stats.units, near_ties=stats.near_ties,
           summary_elements=pstats.elements, summary_one_step=pstats.differ)
    del inp, res
    torch.cuda.empty_cache()


def test_full_decode_128k(dev):
    _full("decode_128k")


def test_full_decode_1m(dev):
    _full("decode_1m")


def test_full_ragged_paged_decode(dev):
    _full("ragged_paged_decode")


# --------------------------------------------------------------------------- the fused decode step

def run_step(inp, k_scored, k_total, force_local=True):
    """Pool, then msa_sparse_decode_step (selection + attention in one call)."""
    from sparse_attention_step_gb300 import msa
    dev = inp.q.device
    desc = msa.kv_desc(inp.k, inp.v, inp.seq_lens, inp.page_table)
    hq = inp.num_q_heads
    need = max(msa.msa_workspace_size(op, desc, hq, 1, k_total) for op in (msa.MSA_OP_POOL, msa.MSA_OP_DECODE_STEP))
    ws = msa.Workspace(need, dev)
    pooled = torch.full(msa.pooled_shape(desc), float("nan"), dtype=inp.k.dtype, device=dev)
    b, hkv = inp.batch, inp.num_kv_heads
    idx = torch.full((b, hkv, k_total), -7, dtype=torch.int32, device=dev)
    out = torch.full_like(inp.q, float("nan"))
    lse = torch.full((b, hq), float("nan"), dtype=torch.float32, device=dev)
    msa.msa_pool_block_keys(desc, 0, -1, pooled, ws.buf, ws.nbytes)
    for _ in range(2):  # twice: nothing may depend on state left by a previous call
        msa.msa_sparse_decode_step(inp.q, hq, pooled, desc, msa.select_cfg(k_scored, force_local), idx, k_total,
                                   SCALE, out, lse, ws.buf, ws.nbytes)
    torch.cuda.synchronize()
    return dict(pooled=pooled, idx=idx, out=out, lse=lse, scores=None, status=msa.msa_read_device_status(ws.buf))


@pytest.mark.parametrize("lens,hkv,hq,k_scored,k_total", [
    ([64 * 300 + 5, 64 * 77, 64 * 1024], 2, 16, 47, 48),   # few units: clusters of 16
    ([64 * 200 + 33] * 20, 4, 32, 31, 32),                  # 80 units: clusters of 2
    ([64 * 40] * 40, 4, 16, 8, 9),                          # 160 units: one CTA per unit
    ([64 * 2048, 64 * 511 + 63], 1, 8, 63, 64),             # long sequence, k = 63
    ([64 * 12, 10, 64], 2, 4, 5, 6),                        # tiny and partial sequences, G = 2
])
def test_fused_step_small(dev, lens, hkv, hq, k_scored, k_total):
    inp = make_decode_inputs(lens, hkv, hq, "bf16", "contiguous", needles=3, seed=sum(lens) % 997, device=dev)
    res = run_step(inp, k_scored, k_total)
    assert res["status"] == 0
    verify_units(inp, res, all_units(inp), k_scored, k_total)


@pytest.mark.parametrize("lens,hkv,hq,k_scored,k_total", [
    ([64 * 300 + 5, 64 * 77, 64 * 1024], 2, 16, 47, 48),   # few units: clusters of 16
    ([64 * 200 + 33] * 20, 4, 32, 31, 32),                  # 80 units: clusters of 2
    ([64 * 12, 10, 64], 2, 4, 5, 6),                        # tiny and partial sequences, G = 2
])
def test_fused_step_paged(dev, lens, hkv, hq, k_scored, k_total):
    """The fused step on a paged cache (shuffled page table): the summaries are
    per sequence, the K/V blocks are gathered through the page table."""
    inp = make_decode_inputs(lens, hkv, hq, "bf16", "paged", needles=3, seed=sum(lens) % 991, device=dev)
    res = run_step(inp, k_scored, k_total)
    assert res["status"] == 0
    verify_units(inp, res, all_units(inp), k_scored, k_total)


def test_fused_step_without_forced_block(dev):
    inp = make_decode_inputs([64 * 100, 64 * 30 + 9], 2, 16, "bf16", "contiguous", needles=2, seed=77, device=dev)
    res = run_step(inp, 6, 6, force_local=False)
    assert res["status"] == 0
    verify_units(inp, res, all_units(inp), 6, 6, force_local=False)


def test_fused_step_flat_scores(dev):
    """Every key row equal, so every summary and every score ties: the
    selection must be the lowest-index candidates (ties go to the lower
    block). With 512 candidate rows per CTA (one unit, clusters of 16) and
    k = 63, far more than 128 keys reach each selection threshold, so both the
    CTA-local and the cluster selection take their sorting-network path."""
    n_full = 6144
    inp = make_decode_inputs([64 * n_full + 17], 1, 8, "bf16", "contiguous", seed=5, device=dev)
    inp.k.copy_(inp.k[:, :, :1, :].expand_as(inp.k))
    res = run_step(inp, 63, 64)
    assert res["status"] == 0
    want = O.select_blocks(np.zeros(n_full), 63, n_full, 64)
    assert res["idx"][0, 0].cpu().tolist() == [int(b) for b in want]
    verify_units(inp, res, [(0, 0)], 63, 64, check_needles=False)


@pytest.mark.parametrize("name", ["decode_128k", "decode_1m"])
def test_fused_step_full(dev, name):
    w = WORKLOADS[name]
    inp = make_workload(name, device=dev)
    res = run_step(inp, w["k_scored"], w["k_total"])
    assert res["status"] == 0
    stats, pstats = SelectionStats(), PoolStats()
    verify_selection_all_units(inp, res["idx"], w["k_scored"], w["k_total"], stats=stats)
    verify_units(inp, res, spread_units(inp), w["k_scored"], w["k_total"], pool_stats=pstats)
    record(f"{name} (fused step)", units=stats.units, near_ties=stats.near_ties,
           summary_elements=pstats.elements, summary_one_step=pstats.differ)
    del inp, res
    torch.cuda.empty_cache()

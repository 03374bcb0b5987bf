"""GPU parity of the decode path against the CPU oracle, through the C ABI.

Small cases are compared on every unit; the full-size workloads (128K x 8,
1M x 1, ragged paged x 32) on sampled units, in the launch configuration the
benchmark uses.
"""
import math

import numpy as np
import pytest
import torch

from oracle import msa_oracle as O
from synth import make_decode_inputs, make_workload, WORKLOADS
from tests.parity import SCALE, SelectionStats, check_lse, check_output, check_selection, to64

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
    p = res["pooled"]
    if inp.layout == "contiguous":
        return to64(p[s, h, :n])
    pages = inp.page_table[s, :n].long()
    return to64(p[pages, h])


def verify_units(inp, res, units, k_scored, k_total, force_local=True, stats=None, check_dense=False,
                 check_needles=True):
    grp = inp.num_q_heads // inp.num_kv_heads
    store = inp.dtype
    for s, h in units:
        n = inp.lens[s]
        qg = to64(inp.q[s, h * grp:(h + 1) * grp])
        kr = to64(inp.kv_rows(s, h, "k"))
        vr = to64(inp.kv_rows(s, h, "v"))
        ref = O.decode_unit(qg, kr, vr, n, k_scored, k_total, SCALE, store, force_local=force_local)
        # pooled summaries: same fp32 row-order sum and rounding -> identical bits
        got_pool = gpu_pooled_rows(inp, res, s, h)
        assert np.array_equal(got_pool, ref["pooled"]), f"pooled keys differ at unit {(s, h)}"
        # raw scores (fp32 dot products vs fp64): tight relative agreement
        if res["scores"] is not None and ref["n_cand"] > 0:
            got_sc = to64(res["scores"][s * inp.num_kv_heads + h, :ref["n_cand"]])
            lim = 1e-5 * np.maximum(1.0, np.abs(ref["scores"])) + 1e-5 * np.abs(ref["q_idx"]).sum()
            assert (np.abs(got_sc - ref["scores"]) <= lim).all(), f"scores differ at unit {(s, h)}"
        got_idx = res["idx"][s, h].cpu().numpy()
        needles = inp.needles.get((s, h), []) if check_needles else []
        check_selection(got_idx, ref["scores"], k_scored, ref["forced"], k_total, stats, needles)
        # attention over the GPU's (validated) selection
        r2 = O.decode_unit(qg, kr, vr, n, k_scored, k_total, SCALE, store, force_local=force_local,
                           selected=got_idx, pooled=ref["pooled"])
        got = to64(res["out"][s, h * grp:(h + 1) * grp])
        if len(r2["tokens"]) == 0:
            assert np.all(got == 0)
            assert np.all(np.isneginf(to64(res["lse"][s, h * grp:(h + 1) * grp])))
        else:
            check_output(got, r2["o"], store, f"decode unit {(s, h)}")
            check_lse(to64(res["lse"][s, h * grp:(h + 1) * grp]), r2["lse"])
        if check_dense and n > 0:
            od, ld = O.dense_gqa(qg, kr, vr, n - 1, SCALE)
            check_output(to64(res["dense_out"][s, h * grp:(h + 1) * grp]), od, store, f"dense unit {(s, h)}")
            check_lse(to64(res["dense_lse"][s, h * grp:(h + 1) * grp]), ld, "dense lse")


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

def _sampled_full(name, units_fn):
    w = WORKLOADS[name]
    dev = torch.device("cuda:0")
    inp = make_workload(name, device=dev)
    # scores stay in the workspace, as in the benchmark
    res = run_decode(inp, w["k_scored"], w["k_total"], dense=True, want_scores=False)
    assert res["status"] == 0
    stats = SelectionStats()
    units = units_fn(inp)
    verify_units(inp, res, units, w["k_scored"], w["k_total"], stats=stats, check_dense=True)
    # every unit (not only the sampled ones) keeps its planted needles and the newest block
    idx = res["idx"].cpu().numpy()
    for (s, h), blocks in inp.needles.items():
        row = set(idx[s, h].tolist())
        assert set(blocks) <= row, f"needles missing in unit {(s, h)}"
        assert (inp.lens[s] + 63) // 64 - 1 in row
    print(name, stats)
    del inp, res
    torch.cuda.empty_cache()


def test_full_decode_128k(dev):
    _sampled_full("decode_128k", lambda inp: [(0, 0), (3, 5), (7, 7)])


def test_full_decode_1m(dev):
    _sampled_full("decode_1m", lambda inp: [(0, 0), (0, 6)])


def test_full_ragged_paged_decode(dev):
    def units(inp):
        lens = np.array(inp.lens)
        return [(int(lens.argmin()), 1), (int(lens.argmax()), 4), (5, 7)]
    _sampled_full("ragged_paged_decode", units)


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


@pytest.mark.parametrize("name,units", [("decode_128k", [(0, 0), (4, 3), (7, 7)]), ("decode_1m", [(0, 1), (0, 7)])])
def test_fused_step_full(dev, name, units):
    w = WORKLOADS[name]
    inp = make_workload(name, device=dev)
    res = run_step(inp, w["k_scored"], w["k_total"])
    assert res["status"] == 0
    verify_units(inp, res, units, w["k_scored"], w["k_total"])
    idx = res["idx"].cpu().numpy()
    for (s, h), blocks in inp.needles.items():
        assert set(blocks) <= set(idx[s, h].tolist()), f"needles missing in unit {(s, h)}"
    del inp, res
    torch.cuda.empty_cache()

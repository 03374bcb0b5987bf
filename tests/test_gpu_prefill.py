"""GPU parity of the chunked-prefill path (tile selection + causal sparse
attention, and the dense comparator) against the CPU oracle."""
import numpy as np
import pytest
import torch

from oracle import msa_oracle as O
from synth import make_prefill_inputs, make_workload, WORKLOADS
from tests.parity import (SCALE, PoolStats, SelectionStats, check_lse, check_output, check_pooled, check_selection,
                          record, to64)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev(lib):
    assert torch.cuda.is_available()
    return torch.device("cuda:0")


def msa_tiles(inp):
    from sparse_attention_step_gb300 import msa
    return msa.chunk_tiles(inp.q_start, inp.n_new)


def run_prefill(inp, k_scored, k_total, dense=False, sparse=True):
    from sparse_attention_step_gb300 import msa
    dev = inp.q.device
    desc = msa.kv_desc(inp.k, inp.v, inp.seq_lens, inp.page_table)
    hq, n = inp.num_q_heads, inp.n_new
    n_tiles = msa.chunk_tiles(inp.q_start, n)
    need = max(msa.msa_workspace_size(msa.MSA_OP_SELECT_PREFILL, desc, hq, n, k_total),
               msa.msa_workspace_size(msa.MSA_OP_PREFILL, desc, hq, n, k_total))
    ws = msa.Workspace(need, dev)
    pooled = torch.full(msa.pooled_shape(desc), float("nan"), dtype=inp.k.dtype, device=dev)
    idx = torch.full((n_tiles, inp.num_kv_heads, k_total), -7, dtype=torch.int32, device=dev)
    max_blocks = desc.max_tokens // 64 if desc.layout == 0 else desc.max_pages_per_seq
    scores = torch.empty(n_tiles * inp.num_kv_heads, max_blocks, dtype=torch.float32, device=dev)
    out = torch.full_like(inp.q, float("nan"))
    lse = torch.full((n, hq), float("nan"), dtype=torch.float32, device=dev)
    msa.msa_pool_block_keys(desc, 0, -1, pooled, ws.buf, ws.nbytes)
    cfg = msa.select_cfg(k_scored, True, 64, inp.q_start)
    msa.msa_select_topk_blocks(inp.q, hq, n, pooled, desc, cfg, idx, k_total, scores, ws.buf, ws.nbytes)
    if sparse:
        msa.msa_sparse_attn_prefill(inp.q, hq, n, inp.q_start, desc, idx, k_total, SCALE, out, lse, ws.buf,
                                    ws.nbytes)
    res = dict(pooled=pooled, idx=idx, scores=scores, out=out, lse=lse)
    if dense:
        dout = torch.full_like(inp.q, float("nan"))
        dlse = torch.full((n, hq), float("nan"), dtype=torch.float32, device=dev)
        msa.msa_dense_gqa_prefill(inp.q, hq, n, inp.q_start, desc, SCALE, dout, dlse, ws.buf, ws.nbytes)
        res.update(dense_out=dout, dense_lse=dlse)
    torch.cuda.synchronize()
    res["status"] = msa.msa_read_device_status(ws.buf)
    return res


def gpu_pooled_head(inp, res, h, n_full):
    return to64(res["pooled"][0, h, :n_full])


def verify_tiles(inp, res, tiles, heads, k_scored, k_total, rows_per_tile=None, stats=None, check_dense=False,
                 check_sparse=True, pool_stats=None):
    """Tiles are the chunk's queries that sit in one 64-token block
    (O.prefill_tiles); tile j's list is idx[j]."""
    grp = inp.num_q_heads // inp.num_kv_heads
    total = inp.q_start + inp.n_new
    part = {j: (lo, hi) for j, lo, hi in O.prefill_tiles(inp.q_start, inp.n_new)}
    for h in heads:
        kr = inp.kv_rows(h, "k").cpu()
        vr = inp.kv_rows(h, "v").cpu()
        pooled, exact = O.pool_block_keys(kr, total, inp.dtype)
        check_pooled(gpu_pooled_head(inp, res, h, total // 64), pooled, exact, inp.dtype,
                     to64(kr) if inp.dtype == "f32" else None, pool_stats, f"pooled keys, head {h}")
        for j in tiles:
            r0, r1 = part[j]
            q_tile = inp.q[r0:r1, h * grp:(h + 1) * grp].cpu()
            sel = O.prefill_tile_select(q_tile, j, inp.q_start, pooled, k_scored, k_total)
            got_idx = res["idx"][j, h].cpu().numpy()
            check_selection(got_idx, sel["scores"], k_scored, sel["diag"], k_total, stats)
            rows = np.arange(r1 - r0) if rows_per_tile is None else \
                np.unique(np.linspace(0, r1 - r0 - 1, rows_per_tile).astype(int))
            pos = inp.q_start + r0 + rows
            if check_sparse:
                o, lse = O.prefill_rows(q_tile[rows], pos, kr, vr, total, got_idx, SCALE)
                got = to64(res["out"][r0 + rows, h * grp:(h + 1) * grp])
                check_output(got, o, inp.dtype, f"prefill tile {j} head {h}")
                check_lse(to64(res["lse"][r0 + rows, h * grp:(h + 1) * grp]), lse)
            if check_dense:
                for i, r in enumerate(rows):
                    od, ld = O.dense_gqa(q_tile[r], kr, vr, pos[i], SCALE)
                    check_output(to64(res["dense_out"][r0 + r, h * grp:(h + 1) * grp]), od, inp.dtype,
                                 f"dense prefill row {r0 + r} head {h}")
                    check_lse(to64(res["dense_lse"][r0 + r, h * grp:(h + 1) * grp]), ld, "dense lse")


def verify_tile_selection_all(inp, res, k_scored, k_total, stats):
    """The selection rule on every (tile, KV head) unit of the chunk."""
    grp = inp.num_q_heads // inp.num_kv_heads
    total = inp.q_start + inp.n_new
    idx = res["idx"].cpu().numpy()
    q = inp.q.cpu()
    for h in range(inp.num_kv_heads):
        pooled, _ = O.pool_block_keys(inp.kv_rows(h, "k").cpu(), total, inp.dtype)
        for j, r0, r1 in O.prefill_tiles(inp.q_start, inp.n_new):
            sel = O.prefill_tile_select(q[r0:r1, h * grp:(h + 1) * grp], j, inp.q_start, pooled, k_scored, k_total)
            check_selection(idx[j, h], sel["scores"], k_scored, sel["diag"], k_total, stats)


@pytest.mark.parametrize("layout", ["contiguous", "paged"])
@pytest.mark.parametrize("prefix,n_new,hq,hkv", [
    (64 * 10 + 37, 64 * 3 + 5, 64, 8),   # tcgen05 kernel: a short first tile, a ragged last tile
    (64 * 10 + 37, 64 * 3 + 5, 16, 2),   # mma.sync kernel, same chunk
    (100, 28, 64, 8),                    # the chunk fills the rest of one block: one tile
    (100, 29, 16, 4),                    # one token into the next block: two tiles
    (63, 1, 64, 8),                      # one token completing block 0
    (64 * 7 + 1, 64 * 2, 32, 4),         # starts one past a block boundary
])
def test_prefill_chunk_starting_inside_a_block(dev, layout, prefix, n_new, hq, hkv):
    """Chunks whose first token is not on a block boundary: the tiles are the
    chunk's queries grouped by block (a shorter first tile), each with its own
    diagonal block; selection and attention against the oracle, dense too."""
    inp = make_prefill_inputs(prefix, n_new, hkv, hq, "bf16", seed=prefix + n_new, device=dev, layout=layout)
    k_scored = 4
    res = run_prefill(inp, k_scored, k_scored + 1, dense=True)
    assert res["status"] == 0
    tiles = O.prefill_tiles(inp.q_start, inp.n_new)
    assert res["idx"].shape[0] == len(tiles)
    verify_tiles(inp, res, [j for j, _, _ in tiles], range(hkv), k_scored, k_scored + 1, check_dense=True)


def test_prefill_unaligned_every_block_equals_dense(dev):
    inp = make_prefill_inputs(64 * 6 + 21, 64 * 2 + 50, 8, 64, "bf16", seed=33, device=dev)
    res = run_prefill(inp, 1000, 1001, dense=True)
    assert res["status"] == 0
    d = (res["out"].float() - res["dense_out"].float()).abs().max().item()
    assert d <= 2e-2


def test_prefill_split_at_a_block_boundary_matches_the_whole_chunk(dev):
    """A chunk split at a block boundary into two calls gives the same index
    lists as the whole chunk (a tile's list depends only on its own queries
    and the blocks before it), and the same outputs within the bf16 tolerance."""
    from sparse_attention_step_gb300 import msa
    inp = make_prefill_inputs(64 * 9 + 40, 24 + 64 * 3 + 10, 8, 64, "bf16", seed=44, device=dev)
    whole = run_prefill(inp, 5, 6)
    cut = 24 + 64  # 64 * 9 + 40 + 88 = 64 * 11: a block boundary
    desc = msa.kv_desc(inp.k, inp.v, inp.seq_lens, inp.page_table)
    hq = inp.num_q_heads
    ws = msa.Workspace(max(msa.msa_workspace_size(msa.MSA_OP_SELECT_PREFILL, desc, hq, inp.n_new, 6),
                           msa.msa_workspace_size(msa.MSA_OP_PREFILL, desc, hq, inp.n_new, 6)), dev)
    msa.msa_pool_block_keys(desc, 0, -1, whole["pooled"], ws.buf, ws.nbytes)
    for lo, hi in ((0, cut), (cut, inp.n_new)):
        q0 = inp.q_start + lo
        q = inp.q[lo:hi].contiguous()
        nt = msa.chunk_tiles(q0, hi - lo)
        idx = torch.full((nt, inp.num_kv_heads, 6), -7, dtype=torch.int32, device=dev)
        out = torch.empty_like(q)
        msa.msa_select_topk_blocks(q, hq, hi - lo, whole["pooled"], desc, msa.select_cfg(5, True, 64, q0), idx, 6,
                                   None, ws.buf, ws.nbytes)
        msa.msa_sparse_attn_prefill(q, hq, hi - lo, q0, desc, idx, 6, SCALE, out, None, ws.buf, ws.nbytes)
        torch.cuda.synchronize()
        t0 = (q0 // 64) - (inp.q_start // 64)
        assert torch.equal(idx, whole["idx"][t0:t0 + nt]), f"lists of rows {lo}..{hi}"
        assert (out.float() - whole["out"][lo:hi].float()).abs().max().item() <= 2e-2
    assert msa.msa_read_device_status(ws.buf) == 0


@pytest.mark.parametrize("hq,hkv", [(16, 2), (8, 8), (16, 4)])
def test_prefill_small(dev, hq, hkv):
    inp = make_prefill_inputs(64 * 10, 64 * 3 + 37, hkv, hq, "bf16", seed=hq + hkv, device=dev)
    res = run_prefill(inp, 4, 5, dense=True)
    assert res["status"] == 0
    n_tiles = msa_tiles(inp)
    verify_tiles(inp, res, range(n_tiles), range(hkv), 4, 5, check_dense=True)


@pytest.mark.parametrize("hq,hkv", [(64, 8), (16, 4)])
def test_prefill_paged_cache(dev, hq, hkv):
    # the same chunked prefill over a paged cache (shuffled pages), tcgen05 and mma.sync kernels
    inp = make_prefill_inputs(64 * 37, 64 * 3 + 21, hkv, hq, "bf16", seed=71, device=dev, layout="paged")
    res = run_prefill(inp, 6, 7, dense=True)
    assert res["status"] == 0
    n_tiles = msa_tiles(inp)
    verify_tiles(inp, res, range(n_tiles), range(hkv), 6, 7, rows_per_tile=9, check_dense=True)


def test_prefill_diagonal_only_list(dev):
    """k_scored = 0: every tile's list is its diagonal block alone (k_total =
    1). 13 tiles x 8 KV heads on the tcgen05 kernel is 208 CTAs, more than
    one per SM, so the CTAs that prefetch for one a wave later reach the
    last unit's one-entry list."""
    inp = make_prefill_inputs(64 * 20 + 9, 64 * 12 + 40, 8, 64, "bf16", seed=17, device=dev)
    res = run_prefill(inp, 0, 1)
    assert res["status"] == 0
    n_tiles = msa_tiles(inp)
    for j in range(n_tiles):
        assert res["idx"][j].cpu().tolist() == [[inp.q_start // 64 + j]] * 8, f"tile {j}"
    verify_tiles(inp, res, range(n_tiles), [0, 7], 0, 1, rows_per_tile=7)


def test_prefill_all_blocks_equals_dense(dev):
    inp = make_prefill_inputs(64 * 6, 64 * 2 + 5, 2, 16, "bf16", seed=3, device=dev)
    res = run_prefill(inp, 1000, 1001, dense=True)
    assert res["status"] == 0
    d = (res["out"].float() - res["dense_out"].float()).abs().max().item()
    assert d <= 2e-2
    verify_tiles(inp, res, range(3), range(2), 1000, 1001, check_dense=True)


def test_prefill_flat_scores(dev):
    """Every key row equal, so every summary score of a tile ties: each tile
    keeps its lowest-index candidates (ties go to the lower block). All keys
    fall in one bin of the binned selection and more than 128 reach the
    threshold, so the top-k runs its full sorting-network path."""
    inp = make_prefill_inputs(64 * 300, 64 * 2 + 11, 2, 16, "bf16", seed=12, device=dev)
    inp.k.copy_(inp.k[:, :, :1, :].expand_as(inp.k))
    res = run_prefill(inp, 32, 33)
    assert res["status"] == 0
    for j in range(3):
        diag = inp.q_start // 64 + j
        want = [int(b) for b in O.select_blocks(np.zeros(diag), 32, diag, 33)]
        for h in range(2):
            assert res["idx"][j, h].cpu().tolist() == want, f"tile {j} head {h}"
    verify_tiles(inp, res, range(3), range(2), 32, 33, rows_per_tile=5)


def test_prefill_from_empty_prefix(dev):
    inp = make_prefill_inputs(0, 64 * 4, 2, 16, "bf16", seed=8, device=dev)
    res = run_prefill(inp, 2, 3, dense=True)
    assert res["status"] == 0
    verify_tiles(inp, res, range(4), range(2), 2, 3, check_dense=True)


def test_full_chunked_prefill(dev):
    """8192 new tokens on a 131072-token prefix, 8 KV heads, 64 query heads,
    top-32 + diagonal: the selection of every (tile, head) unit; outputs on 16
    (tile, head) pairs spread over the chunk and the heads, 6 rows each."""
    w = WORKLOADS["prefill_8k_on_128k"]
    inp = make_workload("prefill_8k_on_128k", device=dev)
    res = run_prefill(inp, w["k_scored"], w["k_total"], dense=True)
    assert res["status"] == 0
    stats, pstats = SelectionStats(), PoolStats()
    verify_tile_selection_all(inp, res, w["k_scored"], w["k_total"], stats)
    n_tiles = msa_tiles(inp)
    for i in range(16):
        tile, head = (i * 37) % n_tiles, i % inp.num_kv_heads
        verify_tiles(inp, res, [tile], [head], w["k_scored"], w["k_total"], rows_per_tile=6,
                     check_dense=(i % 4 == 0), pool_stats=pstats if i < inp.num_kv_heads else None)
    record("prefill_8k_on_128k (select + attend)", units=stats.units, near_ties=stats.near_ties,
           summary_elements=pstats.elements, summary_one_step=pstats.differ)

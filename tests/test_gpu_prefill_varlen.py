"""GPU parity of the batched chunked prefill (several sequences' chunks in one
selection and one attention launch, tokens back to back) through the C ABI:
each sequence's tiles match the CPU oracle, and the batched results equal the
single-sequence calls on that sequence bit for bit."""
import numpy as np
import pytest
import torch

from oracle import msa_oracle as O
from synth import make_prefill_batch_inputs
from tests.parity import SCALE, check_lse, check_output, check_pooled, check_selection, to64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev(lib):
    assert torch.cuda.is_available()
    return torch.device("cuda:0")


def _workspace(msa, desc, hq, n_tiles, k_total, dev):
    need = max(msa.msa_workspace_size(msa.MSA_OP_SELECT_PREFILL, desc, hq, 64 * max(n_tiles, 1), k_total),
               msa.msa_workspace_size(msa.MSA_OP_PREFILL, desc, hq, 1, k_total),
               msa.msa_workspace_size(msa.MSA_OP_POOL, desc, hq, 1, k_total))
    return msa.Workspace(need, dev)


def run_varlen(inp, k_scored, k_total):
    from sparse_attention_step_gb300 import msa
    c = inp.cache
    dev = inp.q.device
    desc = msa.kv_desc(c.k, c.v, c.seq_lens, c.page_table)
    hq, hkv = c.num_q_heads, c.num_kv_heads
    n_tiles = msa.varlen_tiles(inp.q_counts, inp.q_starts)
    ws = _workspace(msa, desc, hq, n_tiles, k_total, dev)
    pooled = torch.full(msa.pooled_shape(desc), float("nan"), dtype=c.k.dtype, device=dev)
    msa.msa_pool_block_keys(desc, 0, -1, pooled, ws.buf, ws.nbytes)
    idx = torch.full((max(n_tiles, 1), hkv, k_total), -7, dtype=torch.int32, device=dev)
    out = torch.full_like(inp.q, float("nan"))
    lse = torch.full((inp.q.shape[0], hq), float("nan"), dtype=torch.float32, device=dev)
    cfg = msa.select_cfg(k_scored, True, 64)
    msa.msa_select_topk_blocks_varlen(inp.q, hq, inp.q_starts, inp.q_counts, pooled, desc, cfg, idx, k_total, None,
                                      ws.buf, ws.nbytes)
    msa.msa_sparse_attn_prefill_varlen(inp.q, hq, inp.q_starts, inp.q_counts, desc, idx, k_total, SCALE, out, lse,
                                       ws.buf, ws.nbytes)
    torch.cuda.synchronize()
    assert msa.msa_read_device_status(ws.buf) == 0
    return dict(pooled=pooled, idx=idx, out=out, lse=lse)


def run_single(inp, s, pooled, k_scored, k_total):
    """Sequence s alone, through the single-sequence entries (a batch-1 view of
    the same cache and summaries)."""
    from sparse_attention_step_gb300 import msa
    c = inp.cache
    dev = inp.q.device
    if c.layout == "contiguous":
        desc = msa.kv_desc(c.k[s:s + 1], c.v[s:s + 1], c.seq_lens[s:s + 1])
    else:
        desc = msa.kv_desc(c.k, c.v, c.seq_lens[s:s + 1], c.page_table[s:s + 1])
    pool_s = pooled[s:s + 1]
    hq, hkv = c.num_q_heads, c.num_kv_heads
    n = inp.q_counts[s]
    n_tiles = msa.chunk_tiles(inp.q_starts[s], n)
    ws = _workspace(msa, desc, hq, n_tiles, k_total, dev)
    q = inp.q_rows(s).contiguous()
    idx = torch.full((n_tiles, hkv, k_total), -7, dtype=torch.int32, device=dev)
    out = torch.full_like(q, float("nan"))
    lse = torch.full((n, hq), float("nan"), dtype=torch.float32, device=dev)
    cfg = msa.select_cfg(k_scored, True, 64, inp.q_starts[s])
    msa.msa_select_topk_blocks(q, hq, n, pool_s, desc, cfg, idx, k_total, None, ws.buf, ws.nbytes)
    msa.msa_sparse_attn_prefill(q, hq, n, inp.q_starts[s], desc, idx, k_total, SCALE, out, lse, ws.buf, ws.nbytes)
    torch.cuda.synchronize()
    assert msa.msa_read_device_status(ws.buf) == 0
    return idx, out, lse


def verify_against_oracle(inp, res, k_scored, k_total, rows_per_tile=7):
    c = inp.cache
    hkv = c.num_kv_heads
    grp = c.num_q_heads // hkv
    for s, (q0, n) in enumerate(zip(inp.q_starts, inp.q_counts)):
        total = q0 + n
        qs = inp.q_rows(s).cpu()
        for h in range(hkv):
            kr, vr = c.kv_rows(s, h, "k").cpu(), c.kv_rows(s, h, "v").cpu()
            pooled, exact = O.pool_block_keys(kr, total, c.dtype)
            nf = total // 64
            got_pool = res["pooled"][s, h, :nf]
            check_pooled(to64(got_pool), pooled, exact, c.dtype, to64(kr) if c.dtype == "f32" else None,
                         what=f"pooled keys seq {s} head {h}")
            for j, r0, r1 in O.prefill_tiles(q0, n):
                g = inp.tile_off[s] + j
                q_tile = qs[r0:r1, h * grp:(h + 1) * grp]
                sel = O.prefill_tile_select(q_tile, j, q0, pooled, k_scored, k_total)
                got_idx = res["idx"][g, h].cpu().numpy()
                check_selection(got_idx, sel["scores"], k_scored, sel["diag"], k_total)
                rows = np.unique(np.linspace(0, r1 - r0 - 1, rows_per_tile).astype(int))
                o, lse = O.prefill_rows(q_tile[rows], q0 + r0 + rows, kr, vr, total, got_idx, SCALE)
                at = inp.q_off[s] + r0 + rows
                check_output(to64(res["out"][at, h * grp:(h + 1) * grp]), o, c.dtype, f"seq {s} tile {j} head {h}")
                check_lse(to64(res["lse"][at, h * grp:(h + 1) * grp]), lse)


@pytest.mark.parametrize("aligned", [True, False])
@pytest.mark.parametrize("layout,hq,hkv", [("contiguous", 64, 8), ("paged", 16, 4), ("contiguous", 16, 2)])
def test_prefill_batch(dev, layout, hq, hkv, aligned):
    # ragged chunks: a long one, one from an empty prefix, a 5-token one, an
    # empty one and one that ends on a tile boundary; unaligned: the same
    # chunks starting inside blocks (as every chunk after the first of a
    # serving loop does)
    q_starts = [64 * 23, 0, 64 * 7, 64 * 3, 64 * 40] if aligned else [64 * 23 + 17, 0, 64 * 7 + 62, 64 * 3 + 5, 64 * 40 + 1]
    q_counts = [64 * 2 + 17, 64 * 3, 5, 0, 64]
    inp = make_prefill_batch_inputs(q_starts, q_counts, hkv, hq, "bf16", layout, seed=91, device=dev)
    k_scored, k_total = 6, 7
    res = run_varlen(inp, k_scored, k_total)
    verify_against_oracle(inp, res, k_scored, k_total)
    # each sequence alone through the single-sequence entries: identical bits
    for s, n in enumerate(q_counts):
        if n == 0:
            continue
        idx, out, lse = run_single(inp, s, res["pooled"], k_scored, k_total)
        t0, t1 = inp.tile_off[s], inp.tile_off[s + 1]
        o0 = inp.q_off[s]
        assert torch.equal(res["idx"][t0:t1], idx), f"selection of sequence {s}"
        assert torch.equal(res["out"][o0:o0 + n], out), f"output of sequence {s}"
        assert torch.equal(res["lse"][o0:o0 + n], lse), f"lse of sequence {s}"


def test_prefill_batch_rejects_bad_batches(dev):
    from sparse_attention_step_gb300 import msa
    inp = make_prefill_batch_inputs([64, 128], [10, 20], 2, 16, "bf16", seed=92, device=dev)
    c = inp.cache
    desc = msa.kv_desc(c.k, c.v, c.seq_lens, c.page_table)
    ws = _workspace(msa, desc, 16, 2, 5, dev)
    idx = torch.zeros(2, 2, 5, dtype=torch.int32, device=dev)
    out = torch.empty_like(inp.q)
    cases = [([64], [10], msa.MSA_ERR_INVALID_ARG),               # one sequence for a batch of two
             ([64, 128], [10, -1], msa.MSA_ERR_INVALID_ARG),      # negative count
             ([-1, 128], [10, 10], msa.MSA_ERR_INVALID_ARG),      # negative start
             ([64, 128], [10, 10 ** 6], msa.MSA_ERR_INVALID_ARG)]  # past the cache's capacity
    for starts, counts, want in cases:
        with pytest.raises(msa.MsaError) as e:
            msa.msa_sparse_attn_prefill_varlen(inp.q, 16, starts, counts, desc, idx, 5, SCALE, out, None, ws.buf,
                                               ws.nbytes)
        assert e.value.status == want, (starts, counts)
    torch.cuda.synchronize()
    assert msa.msa_read_device_status(ws.buf) == 0

"""GPU parity of the attention-sink selection (block 0 always kept, never
scored, alongside the newest / diagonal block) against the CPU oracle, through
the C ABI, on every selection path: the fused decode step (contiguous and
paged caches), the chunked decode selection, the radix top-k (k above 64,
prefill tiles) and the token-max scores."""
import numpy as np
import pytest
import torch

from oracle import msa_oracle as O
from synth import make_decode_inputs, make_index_keys, make_prefill_inputs
from tests.parity import REL_GAP, SCALE, check_lse, check_output, to64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev(lib):
    assert torch.cuda.is_available()
    return torch.device("cuda:0")


def check_sink_row(got_row, scores, k_scored, forced, k_total, has0):
    """Exact match with the oracle's sink selection unless the k-th and
    (k+1)-th scores among blocks 1.. are a near-tie; then the structure is
    checked and the kept scored blocks must lie in the near-tie band or above."""
    want = O.select_blocks_sink(scores, k_scored, forced, k_total, has0)
    got = [int(b) for b in got_row]
    if got == list(want):
        return
    rest = np.asarray(scores, dtype=np.float64)[1:]
    gap = O.boundary_gap(rest, k_scored)
    assert gap is not None, f"selection differs:\n gpu {got}\n ora {list(want)}"
    s_k, s_k1 = gap
    band = REL_GAP * max(abs(s_k), 1e-30)
    assert s_k - s_k1 < band, f"selection differs:\n gpu {got}\n ora {list(want)}"
    kept = [b for b in got if b >= 0]
    assert kept == sorted(kept) and (0 in kept) == has0
    scored = [b for b in kept if b != 0 and b != forced]
    assert len(scored) == min(k_scored, max(len(scores) - 1, 0))
    assert all(scores[b] >= s_k - band for b in scored)


def run_decode_sink(inp, k_scored, k_total, step, kidx=None):
    from sparse_attention_step_gb300 import msa
    dev = inp.q.device
    desc = msa.kv_desc(inp.k, inp.v, inp.seq_lens, inp.page_table)
    hq = inp.num_q_heads
    ops = [msa.MSA_OP_POOL, msa.MSA_OP_SELECT, msa.MSA_OP_DECODE, msa.MSA_OP_DECODE_STEP]
    ws = msa.Workspace(max(msa.msa_workspace_size(op, desc, hq, 1, k_total) for op in ops), dev)
    pooled = torch.zeros(msa.pooled_shape(desc), dtype=inp.k.dtype, device=dev)
    msa.msa_pool_block_keys(desc, 0, -1, pooled, ws.buf, ws.nbytes)
    b, hkv = inp.batch, inp.num_kv_heads
    idx = torch.full((b, hkv, k_total), -7, dtype=torch.int32, device=dev)
    out = torch.empty_like(inp.q)
    lse = torch.empty(b, hq, dtype=torch.float32, device=dev)
    mode = msa.MSA_SCORE_TOKEN_MAX if kidx is not None else None
    cfg = msa.select_cfg(k_scored, sink=True, mode=mode)
    src = kidx if kidx is not None else pooled
    if step:
        msa.msa_sparse_decode_step(inp.q, hq, src, desc, cfg, idx, k_total, SCALE, out, lse, ws.buf, ws.nbytes)
    else:
        msa.msa_select_topk_blocks(inp.q, hq, 1, src, desc, cfg, idx, k_total, None, ws.buf, ws.nbytes)
        msa.msa_sparse_attn_decode(inp.q, hq, desc, idx, k_total, SCALE, out, lse, ws.buf, ws.nbytes)
    torch.cuda.synchronize()
    assert msa.msa_read_device_status(ws.buf) == 0
    return idx, out, lse


@pytest.mark.parametrize("layout,k_scored,step", [
    ("contiguous", 5, True),     # fused decode step
    ("paged", 5, True),          # fused decode step on a paged cache
    ("paged", 5, False),         # chunked selection kernel + attention
    ("contiguous", 70, False),   # radix top-k (k above 64)
    ("paged", 64, False),        # chunked selection at its largest k: the list fills k_total
    ("contiguous", 64, True),    # fused decode step at its largest k
])
def test_decode_sink(dev, layout, k_scored, step):
    lens = [64 * 150 + 7, 64 * 12, 64 + 3, 40]
    inp = make_decode_inputs(lens, 2, 16, "bf16", layout, needles=2, seed=61, device=dev)
    k_total = k_scored + 2
    idx, out, lse = run_decode_sink(inp, k_scored, k_total, step)
    grp = inp.num_q_heads // inp.num_kv_heads
    for s, n in enumerate(lens):
        for h in range(inp.num_kv_heads):
            qg = to64(inp.q[s, h * grp:(h + 1) * grp])
            kr, vr = to64(inp.kv_rows(s, h, "k")), to64(inp.kv_rows(s, h, "v"))
            ref = O.decode_unit(qg, kr, vr, n, k_scored, k_total, SCALE, "bf16")
            got = idx[s, h].cpu().numpy()
            check_sink_row(got, ref["scores"], k_scored, ref["forced"], k_total, True)
            r2 = O.decode_unit(qg, kr, vr, n, k_scored, k_total, SCALE, "bf16", selected=got, pooled=ref["pooled"])
            check_output(to64(out[s, h * grp:(h + 1) * grp]), r2["o"], "bf16", f"unit {(s, h)}")
            check_lse(to64(lse[s, h * grp:(h + 1) * grp]), r2["lse"])


def test_token_max_sink(dev):
    lens = [64 * 90 + 13, 64 * 33]
    inp = make_decode_inputs(lens, 2, 16, "bf16", "contiguous", seed=62, device=dev)
    ik = make_index_keys(inp, needles=2, seed=63)
    idx, out, lse = run_decode_sink(inp, 6, 8, False, kidx=ik.kidx)
    grp = inp.num_q_heads // inp.num_kv_heads
    for s, n in enumerate(lens):
        for h in range(inp.num_kv_heads):
            qg = to64(inp.q[s, h * grp:(h + 1) * grp])
            ref = O.select_token_max(qg, to64(ik.rows(inp, s)), n, 6, 8)
            check_sink_row(idx[s, h].cpu().numpy(), ref["scores"], 6, ref["forced"], 8, True)


def test_prefill_sink(dev):
    from sparse_attention_step_gb300 import msa
    inp = make_prefill_inputs(64 * 20, 64 * 3 + 9, 2, 16, "bf16", seed=64, device=dev)
    desc = msa.kv_desc(inp.k, inp.v, inp.seq_lens)
    hq, n = inp.num_q_heads, inp.n_new
    k_scored, k_total = 4, 6
    ws = msa.Workspace(max(msa.msa_workspace_size(op, desc, hq, n, k_total)
                           for op in (msa.MSA_OP_POOL, msa.MSA_OP_SELECT_PREFILL, msa.MSA_OP_PREFILL)), dev)
    pooled = torch.zeros(msa.pooled_shape(desc), dtype=inp.k.dtype, device=dev)
    msa.msa_pool_block_keys(desc, 0, -1, pooled, ws.buf, ws.nbytes)
    n_tiles = msa.chunk_tiles(inp.q_start, n)
    idx = torch.full((n_tiles, inp.num_kv_heads, k_total), -7, dtype=torch.int32, device=dev)
    cfg = msa.select_cfg(k_scored, True, 64, inp.q_start, sink=True)
    msa.msa_select_topk_blocks(inp.q, hq, n, pooled, desc, cfg, idx, k_total, None, ws.buf, ws.nbytes)
    torch.cuda.synchronize()
    assert msa.msa_read_device_status(ws.buf) == 0
    grp = hq // inp.num_kv_heads
    total = inp.q_start + n
    pooled_h = [O.pool_block_keys(inp.kv_rows(h, "k").cpu(), total, "bf16")[0] for h in range(inp.num_kv_heads)]
    for j in range(n_tiles):
        rows = to64(inp.q[64 * j:64 * (j + 1)])
        for h in range(inp.num_kv_heads):
            q_tile = rows[:, h * grp:(h + 1) * grp]
            ref = O.prefill_tile_select(q_tile, j, inp.q_start, pooled_h[h], k_scored, k_total)
            check_sink_row(idx[j, h].cpu().numpy(), ref["scores"], k_scored, ref["diag"], k_total, True)

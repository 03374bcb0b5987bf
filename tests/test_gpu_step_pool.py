"""A generation loop through msa_sparse_decode_step_pool: the step that also
writes the summary of a block the moment it fills. Checked through the C ABI:
after the step at which a block fills, the summaries equal a full pooling of
the cache at that length bit for bit (other summaries untouched), the outputs
of every step equal msa_sparse_decode_step's, and the next step (which scores
the new block) matches the CPU oracle."""
import numpy as np
import pytest
import torch

from oracle import msa_oracle as O
from synth import make_decode_inputs
from tests.parity import SCALE, check_lse, check_output, check_selection, to64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev(lib):
    assert torch.cuda.is_available()
    return torch.device("cuda:0")


def _pool_full(msa, desc, like, ws):
    pooled = torch.zeros(msa.pooled_shape(desc), dtype=like.dtype, device=like.device)
    msa.msa_pool_block_keys(desc, 0, -1, pooled, ws.buf, ws.nbytes)
    return pooled


@pytest.mark.parametrize("layout,k_scored", [("contiguous", 7), ("contiguous", 100), ("paged", 7)])
def test_generation_loop_keeps_summaries_current(dev, layout, k_scored):
    from sparse_attention_step_gb300 import msa
    # every sequence sits one token short of filling a block; the cache holds
    # the tokens of the next two steps already
    start = [64 * 40 - 1, 64 * 9 - 1, 64 * 130 - 1]
    inp = make_decode_inputs([n + 2 for n in start], 2, 16, "bf16", layout, needles=2, seed=77, device=dev)
    k_total = k_scored + 1
    desc = msa.kv_desc(inp.k, inp.v, inp.seq_lens, inp.page_table)
    hq, b, hkv = inp.num_q_heads, inp.batch, inp.num_kv_heads
    ops = [msa.MSA_OP_POOL, msa.MSA_OP_SELECT, msa.MSA_OP_DECODE, msa.MSA_OP_DECODE_STEP]
    ws = msa.Workspace(max(msa.msa_workspace_size(op, desc, hq, 1, k_total) for op in ops), dev)
    cfg = msa.select_cfg(k_scored)
    grp = hq // hkv

    def set_len(lens):
        inp.seq_lens.copy_(torch.tensor(lens, dtype=torch.int32))
        inp.lens = list(lens)

    set_len(start)
    pooled = _pool_full(msa, desc, inp.k, ws)
    for step in range(3):
        lens = [n + step for n in start]
        set_len(lens)
        before = pooled.clone()
        idx = torch.full((b, hkv, k_total), -7, dtype=torch.int32, device=dev)
        out = torch.empty_like(inp.q)
        lse = torch.empty(b, hq, dtype=torch.float32, device=dev)
        msa.msa_sparse_decode_step_pool(inp.q, hq, pooled, desc, cfg, idx, k_total, SCALE, out, lse, ws.buf,
                                        ws.nbytes)
        # the same step without the summary upkeep, on the summaries it started from
        idx2 = torch.full_like(idx, -7)
        out2 = torch.empty_like(out)
        lse2 = torch.empty_like(lse)
        msa.msa_sparse_decode_step(inp.q, hq, before, desc, cfg, idx2, k_total, SCALE, out2, lse2, ws.buf,
                                   ws.nbytes)
        torch.cuda.synchronize()
        assert msa.msa_read_device_status(ws.buf) == 0
        assert torch.equal(idx, idx2)
        assert torch.equal(out, out2) and torch.equal(lse, lse2)
        # summaries: exactly a full pooling at this length (the new block, bit for bit)
        full = _pool_full(msa, desc, inp.k, ws)
        torch.cuda.synchronize()
        filled = step == 1
        for s, n in enumerate(lens):
            nbf = n // 64
            assert torch.equal(pooled[s, :, :nbf], full[s, :, :nbf]), f"summaries differ, step {step}"
            if filled:
                assert not torch.equal(pooled[s, :, nbf - 1], before[s, :, nbf - 1])
        # oracle: selection over the summaries of this length, attention over the GPU's list
        for s in range(b):
            for h in range(hkv):
                qg = to64(inp.q[s, h * grp:(h + 1) * grp])
                kr = to64(inp.kv_rows(s, h, "k"))
                vr = to64(inp.kv_rows(s, h, "v"))
                ref = O.decode_unit(qg, kr, vr, lens[s], k_scored, k_total, SCALE, "bf16")
                got_idx = idx[s, h].cpu().numpy()
                check_selection(got_idx, ref["scores"], k_scored, ref["forced"], k_total)
                r2 = O.decode_unit(qg, kr, vr, lens[s], k_scored, k_total, SCALE, "bf16", selected=got_idx,
                                   pooled=ref["pooled"])
                check_output(to64(out[s, h * grp:(h + 1) * grp]), r2["o"], "bf16", f"step {step} unit {(s, h)}")
                check_lse(to64(lse[s, h * grp:(h + 1) * grp]), r2["lse"])


def test_step_pool_rejects_token_max_mode(lib):
    import ctypes
    from sparse_attention_step_gb300 import msa
    d = msa.KvDesc()
    d.layout, d.dtype, d.batch, d.num_kv_heads, d.head_dim, d.block_size = 0, 1, 1, 1, 128, 64
    d.k, d.v, d.seq_lens, d.max_tokens = 0x1000, 0x2000, 0x3000, 1024
    cfg = msa.select_cfg(4, mode=msa.MSA_SCORE_TOKEN_MAX)
    st = lib.msa_sparse_decode_step_pool(0x1, 8, 0x1, ctypes.byref(d), ctypes.byref(cfg), 0x1, 5, 0.1, 0x1, None,
                                         0x1, 1 << 20, None)
    assert st == msa.MSA_ERR_UNSUPPORTED

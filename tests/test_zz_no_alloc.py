"""The allocation-free decode entry point (msa_sparse_attn_decode_noalloc).

It exists for callers that cannot allocate device memory themselves, such as
an engine or plugin host that owns every allocation, or a serving loop that
must not call cudaMalloc/cudaFree once running (both can synchronise the
device). Its split-K scratch is a fixed 4 MiB array inside the library.

Checked here through the C ABI: calls in a row give the same outputs as
msa_sparse_attn_decode with a caller workspace, within the tolerances the
parity tests use (bf16 max-abs 2e-2; fp32 1e-3 relative). bf16 combines its
splits inside a thread-block cluster; fp32 combines them through split-K
tickets and partial results kept in the fixed scratch, so the fp32 case runs
many splits per unit and changes shape between calls (stale tickets or
partials would show). fp32 shapes that need more than the fixed scratch are
rejected. This file is collected last and builds everything it needs itself.
"""
import ctypes
import math

import pytest
import torch

from synth import make_decode_inputs

pytestmark = pytest.mark.gpu

SCALE = 1.0 / math.sqrt(128)
BF16_ABS = 2e-2
F32_REL = 1e-3


def _reference(msa, inp, k_scored, k_total):
    """Pool, select and decode with a caller workspace."""
    dev = inp.q.device
    desc = msa.kv_desc(inp.k, inp.v, inp.seq_lens, inp.page_table)
    hq = inp.num_q_heads
    need = max(msa.msa_workspace_size(op, desc, hq, 1, k_total)
               for op in (msa.MSA_OP_POOL, msa.MSA_OP_SELECT, msa.MSA_OP_DECODE))
    ws = msa.Workspace(need, dev)
    pooled = torch.zeros(msa.pooled_shape(desc), dtype=inp.k.dtype, device=dev)
    idx = torch.empty(inp.batch, inp.num_kv_heads, k_total, dtype=torch.int32, device=dev)
    out = torch.empty_like(inp.q)
    lse = torch.empty(inp.batch, hq, dtype=torch.float32, device=dev)
    msa.msa_pool_block_keys(desc, 0, -1, pooled, ws.buf, ws.nbytes)
    msa.msa_select_topk_blocks(inp.q, hq, 1, pooled, desc, msa.select_cfg(k_scored), idx, k_total, None, ws.buf,
                               ws.nbytes)
    msa.msa_sparse_attn_decode(inp.q, hq, desc, idx, k_total, SCALE, out, lse, ws.buf, ws.nbytes)
    torch.cuda.synchronize()
    assert msa.msa_read_device_status(ws.buf) == 0
    return desc, idx, out, lse


@pytest.mark.parametrize("layout", ["contiguous", "paged"])
def test_noalloc_decode_matches_workspace_decode_twice(lib, layout):
    from sparse_attention_step_gb300 import msa
    dev = torch.device("cuda:0")
    # 4 units with a 48-entry list: several splits per unit, combined inside
    # each unit's thread-block cluster
    inp = make_decode_inputs([64 * 300 + 5, 64 * 77], 2, 16, "bf16", layout, needles=3, seed=31, device=dev)
    desc, idx, ref_out, ref_lse = _reference(msa, inp, 47, 48)
    for call in range(2):
        out = torch.full_like(inp.q, float("nan"))
        lse = torch.full_like(ref_lse, float("nan"))
        msa.msa_sparse_attn_decode_noalloc(inp.q, inp.num_q_heads, desc, idx, 48, SCALE, out, lse)
        torch.cuda.synchronize()
        d = (out.float() - ref_out.float()).abs().max().item()
        assert d <= BF16_ABS, f"call {call}: max-abs {d}"
        dl = (lse - ref_lse).abs().max().item()
        assert dl <= 1e-3 * max(1.0, ref_lse.abs().max().item()), f"call {call}: lse differs by {dl}"


def _f32_close(got, ref, what):
    d = (got.double() - ref.double()).abs()
    lim = F32_REL * ref.double().abs().clamp(min=1.0)
    assert bool((d <= lim).all()), f"{what}: max diff {d.max().item():.3e}"


def test_noalloc_f32_split_k_scratch_across_calls_and_shapes(lib):
    """fp32 keeps its split-K tickets and partials in the fixed scratch: the
    4096-token workload shape (one unit, 9 listed blocks, one split per block)
    then a different shape, then the first again; each must match the
    workspace decode."""
    from sparse_attention_step_gb300 import msa
    dev = torch.device("cuda:0")
    a = make_decode_inputs([4096], 1, 4, "f32", "contiguous", needles=2, seed=1001, device=dev)
    b = make_decode_inputs([64 * 9 + 3, 200, 64 * 12], 2, 8, "f32", "paged", needles=1, seed=5, device=dev)
    refs = {id(a): _reference(msa, a, 8, 9) + (9,), id(b): _reference(msa, b, 3, 5) + (5,)}
    for call, inp in enumerate((a, a, b, a)):
        desc, idx, ref_out, ref_lse, k_total = refs[id(inp)]
        out = torch.full_like(inp.q, float("nan"))
        lse = torch.full_like(ref_lse, float("nan"))
        msa.msa_sparse_attn_decode_noalloc(inp.q, inp.num_q_heads, desc, idx, k_total, SCALE, out, lse)
        torch.cuda.synchronize()
        _f32_close(out, ref_out, f"call {call} output")
        _f32_close(lse, ref_lse, f"call {call} lse")


def test_noalloc_rejects_shapes_beyond_the_fixed_scratch(lib):
    from sparse_attention_step_gb300 import msa
    dev = torch.device("cuda:0")
    # fp32, 160 sequences x 8 KV heads: 1280 partial results of 4160 bytes
    # exceed 4 MiB
    inp = make_decode_inputs([128] * 160, 8, 64, "f32", "contiguous", seed=5, device=dev)
    desc = msa.kv_desc(inp.k, inp.v, inp.seq_lens)
    assert msa.msa_workspace_size(msa.MSA_OP_DECODE, desc, 64, 1, 3) > (4 << 20)
    idx = torch.zeros(160, 8, 3, dtype=torch.int32, device=dev)
    out = torch.empty_like(inp.q)
    st = msa.load().msa_sparse_attn_decode_noalloc(inp.q.data_ptr(), 64, ctypes.byref(desc), idx.data_ptr(), 3,
                                                   SCALE, out.data_ptr(), None, torch.cuda.current_stream().cuda_stream)
    assert st == msa.MSA_ERR_WORKSPACE

"""The C-ABI library loads, exports every symbol include/msa.h declares, and
rejects bad arguments on the host before any launch (no GPU needed)."""
import ctypes
import os
import re
import subprocess

import pytest

from sparse_attention_step_gb300 import msa

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "msa.h")


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = set(re.findall(r"\b(msa_[a-z_0-9]+)\s*\(", text))
    return sorted(names)


def test_header_declares_the_binding_exports():
    assert _declared() == sorted(msa.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", msa.library_path()], capture_output=True, text=True,
                         check=True).stdout
    exported = set(re.findall(r"\sT\s(msa_\w+)", out))
    for name in _declared():
        assert name in exported, name
        assert getattr(lib, name) is not None


def test_status_strings(lib):
    for code in range(7):
        assert msa.status_string(code)
    assert msa.status_string(99) == "unknown status"
    assert msa.msa_version() == 0x000100


def _desc(**kw):
    d = msa.KvDesc()
    d.layout, d.dtype, d.batch, d.num_kv_heads, d.head_dim, d.block_size = 0, 1, 2, 2, 128, 64
    d.k, d.v, d.seq_lens = 0x1000, 0x2000, 0x3000
    d.max_tokens = 1024
    for k, v in kw.items():
        setattr(d, k, v)
    return d


@pytest.mark.parametrize("field,value,expect", [
    ("head_dim", 64, msa.MSA_ERR_UNSUPPORTED),
    ("block_size", 32, msa.MSA_ERR_UNSUPPORTED),
    ("max_tokens", 1000, msa.MSA_ERR_INVALID_ARG),
    ("batch", 0, msa.MSA_ERR_INVALID_ARG),
    ("layout", 7, msa.MSA_ERR_INVALID_ARG),
    ("dtype", 5, msa.MSA_ERR_INVALID_ARG),
    ("k", None, msa.MSA_ERR_INVALID_ARG),
])
def test_bad_descriptor_rejected_before_launch(lib, field, value, expect):
    d = _desc(**{field: value})
    st = lib.msa_pool_block_keys(ctypes.byref(d), 0, -1, 0x4000, None, 0, None)
    assert st == expect
    assert lib.msa_workspace_size(msa.MSA_OP_POOL, ctypes.byref(d), 16, 1, 8) == 0


def test_paged_descriptor_needs_a_table(lib):
    d = _desc(layout=1, num_pages=10, max_pages_per_seq=4)
    assert lib.msa_pool_block_keys(ctypes.byref(d), 0, -1, 0x4000, None, 0, None) == msa.MSA_ERR_INVALID_ARG


def test_head_and_selection_arguments(lib):
    d = _desc()
    cfg = msa.select_cfg(4)
    # Hq not a multiple of Hkv
    assert lib.msa_select_topk_blocks(0x10, 15, 1, 0x1, ctypes.byref(d), ctypes.byref(cfg), 0x1, 5, None, 0x1, 1 << 20,
                                      None) == msa.MSA_ERR_INVALID_ARG
    # more than 8 query heads per KV head
    assert lib.msa_select_topk_blocks(0x10, 32, 1, 0x1, ctypes.byref(d), ctypes.byref(cfg), 0x1, 5, None, 0x1, 1 << 20,
                                      None) == msa.MSA_ERR_UNSUPPORTED
    # k_total too small for k_scored + the forced block
    assert lib.msa_select_topk_blocks(0x10, 16, 1, 0x1, ctypes.byref(d), ctypes.byref(cfg), 0x1, 4, None, 0x1, 1 << 20,
                                      None) == msa.MSA_ERR_INVALID_ARG
    bad = msa.select_cfg(4, q_tile=3)
    assert lib.msa_select_topk_blocks(0x10, 16, 1, 0x1, ctypes.byref(d), ctypes.byref(bad), 0x1, 5, None, 0x1, 1 << 20,
                                      None) == msa.MSA_ERR_UNSUPPORTED
    # a chunk may start anywhere, but must fit in the cache (1024 tokens) and not start before it
    d1 = _desc(batch=1)
    for q_start in (1000, -1):
        cfg_p = msa.select_cfg(4, q_tile=64, q_start=q_start)
        assert lib.msa_select_topk_blocks(0x10, 16, 64, 0x1, ctypes.byref(d1), ctypes.byref(cfg_p), 0x1, 5, None, 0x1,
                                          1 << 20, None) == msa.MSA_ERR_INVALID_ARG


def test_decode_and_prefill_arguments(lib):
    d = _desc()
    assert lib.msa_sparse_attn_decode(0x10, 16, ctypes.byref(d), None, 8, 0.1, 0x1, None, 0x1, 1 << 20,
                                      None) == msa.MSA_ERR_INVALID_ARG
    assert lib.msa_sparse_attn_decode(0x10, 16, ctypes.byref(d), 0x1, 8, -1.0, 0x1, None, 0x1, 1 << 20,
                                      None) == msa.MSA_ERR_INVALID_ARG
    # prefill: batch must be 1
    assert lib.msa_sparse_attn_prefill(0x10, 16, 64, 0, ctypes.byref(d), 0x1, 5, 0.1, 0x1, None, 0x1, 1 << 20,
                                       None) == msa.MSA_ERR_UNSUPPORTED
    d1 = _desc(batch=1)
    # any start, but the chunk must fit in the cache's 1024 tokens
    assert lib.msa_dense_gqa_prefill(0x10, 16, 64, 980, ctypes.byref(d1), 0.1, 0x1, None, 0x1, 1 << 20,
                                     None) == msa.MSA_ERR_INVALID_ARG
    assert lib.msa_dense_gqa_prefill(0x10, 16, 2000, 0, ctypes.byref(d1), 0.1, 0x1, None, 0x1, 1 << 20,
                                     None) == msa.MSA_ERR_INVALID_ARG


def test_queries_and_outputs_must_be_16_byte_aligned(lib):
    """q and out move in 16-byte pieces: a misaligned base is an argument
    error, found before any launch."""
    d, d1 = _desc(), _desc(batch=1)
    cfg = msa.select_cfg(4)
    for q, out in ((0x18, 0x20), (0x20, 0x18)):
        assert lib.msa_sparse_attn_decode(q, 16, ctypes.byref(d), 0x40, 8, 0.1, out, None, 0x40, 1 << 20,
                                          None) == msa.MSA_ERR_INVALID_ARG
        assert lib.msa_sparse_attn_decode_noalloc(q, 16, ctypes.byref(d), 0x40, 8, 0.1, out, None,
                                                  None) == msa.MSA_ERR_INVALID_ARG
        assert lib.msa_sparse_decode_step(q, 16, 0x40, ctypes.byref(d), ctypes.byref(cfg), 0x40, 5, 0.1, out, None,
                                          0x40, 1 << 20, None) == msa.MSA_ERR_INVALID_ARG
        assert lib.msa_sparse_attn_prefill(q, 16, 64, 0, ctypes.byref(d1), 0x40, 5, 0.1, out, None, 0x40, 1 << 20,
                                           None) == msa.MSA_ERR_INVALID_ARG
    assert lib.msa_select_topk_blocks(0x18, 16, 1, 0x40, ctypes.byref(d), ctypes.byref(cfg), 0x40, 5, None, 0x40,
                                      1 << 20, None) == msa.MSA_ERR_INVALID_ARG
    # pooled keys and the cache's k, v
    assert lib.msa_select_topk_blocks(0x20, 16, 1, 0x48, ctypes.byref(d), ctypes.byref(cfg), 0x40, 5, None, 0x40,
                                      1 << 20, None) == msa.MSA_ERR_INVALID_ARG
    assert lib.msa_pool_block_keys(ctypes.byref(d), 0, -1, 0x48, None, 0, None) == msa.MSA_ERR_INVALID_ARG
    for field in ("k", "v"):
        bad = _desc(**{field: 0x1008})
        assert lib.msa_pool_block_keys(ctypes.byref(bad), 0, -1, 0x4000, None, 0, None) == msa.MSA_ERR_INVALID_ARG


def _batch(starts, counts):
    n = len(starts)
    return n, (ctypes.c_int64 * n)(*starts), (ctypes.c_int32 * n)(*counts)


@pytest.mark.parametrize("starts,counts,expect", [
    ([64], [10], msa.MSA_ERR_INVALID_ARG),                 # one chunk for a cache of two sequences
    ([64, 1000], [10, 30], msa.MSA_ERR_INVALID_ARG),       # a start inside a block, past the capacity
    ([64, 128], [10, -1], msa.MSA_ERR_INVALID_ARG),        # a negative count
    ([-64, 128], [10, 1], msa.MSA_ERR_INVALID_ARG),        # a negative start
    ([64, 128], [10, 1000], msa.MSA_ERR_INVALID_ARG),      # past the sequence's capacity (1024 tokens)
])
def test_chunk_batch_arguments(lib, starts, counts, expect):
    # both batched-prefill entries check the chunk table on the host, before any launch
    d = _desc()
    n, st, ct = _batch(starts, counts)
    assert lib.msa_sparse_attn_prefill_varlen(0x1, 16, n, st, ct, ctypes.byref(d), 0x1, 5, 0.1, 0x1, None, 0x1,
                                              1 << 20, None) == expect
    cfg = msa.select_cfg(4, True, 64)
    assert lib.msa_select_topk_blocks_varlen(0x1, 16, n, st, ct, 0x1, ctypes.byref(d), ctypes.byref(cfg), 0x1, 5,
                                             None, 0x1, 1 << 20, None) == expect


def test_chunk_batch_needs_tiles_and_tables(lib):
    d = _desc()
    n, st, ct = _batch([0, 64], [64, 64])
    decode_cfg = msa.select_cfg(4)  # q_tile 1: not a tile selection
    assert lib.msa_select_topk_blocks_varlen(0x1, 16, n, st, ct, 0x1, ctypes.byref(d), ctypes.byref(decode_cfg), 0x1,
                                             5, None, 0x1, 1 << 20, None) == msa.MSA_ERR_INVALID_ARG
    cfg = msa.select_cfg(4, True, 64)
    assert lib.msa_select_topk_blocks_varlen(0x1, 16, n, None, ct, 0x1, ctypes.byref(d), ctypes.byref(cfg), 0x1, 5,
                                             None, 0x1, 1 << 20, None) == msa.MSA_ERR_INVALID_ARG
    assert lib.msa_sparse_attn_prefill_varlen(0x1, 16, n, st, ct, ctypes.byref(d), None, 5, 0.1, 0x1, None, 0x1,
                                              1 << 20, None) == msa.MSA_ERR_INVALID_ARG
    # more sequences than one launch's table holds
    big = _desc(batch=65)
    n, st, ct = _batch([0] * 65, [1] * 65)
    assert lib.msa_sparse_attn_prefill_varlen(0x1, 16, n, st, ct, ctypes.byref(big), 0x1, 5, 0.1, 0x1, None, 0x1,
                                              1 << 20, None) == msa.MSA_ERR_UNSUPPORTED

"""Host-side arithmetic of the benchmark and the binding (no GPU): the bytes a
decode step is charged with, the per-step quantiles, and the chunk-batch
helpers of the binding."""
import os
import sys
import types

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from sparse_attention_step_gb300 import msa  # noqa: E402


def test_decode_bytes_counts_candidates_selection_and_io():
    # two sequences, 2 KV heads, 16 query heads, bf16: summaries of the complete
    # blocks before the newest, k_total selected blocks of K and V, q and out
    q = types.SimpleNamespace(numel=lambda: 2 * 16 * 128, element_size=lambda: 2)
    inp = types.SimpleNamespace(lens=[64 * 10 + 5, 64 * 3], num_kv_heads=2, q=q)
    pooled, sel, qo = bench.decode_bytes(inp, 4)
    # candidates: min(full blocks, blocks - 1) = min(10, 10) and min(3, 2)
    assert pooled == (10 + 2) * 2 * 128 * 2
    # selected: min(k_total, blocks) = 4 and 3, each 64 x 128 x 2 bytes of K and of V
    assert sel == (4 + 3) * 2 * 2 * 64 * 128 * 2
    assert qo == 2 * (2 * 16 * 128 * 2)


def test_decode_bytes_of_the_headline_workload():
    # 8 x 131072 tokens, 8 KV heads, 64 query heads, 31 + 1 blocks: 100,909,056 bytes
    q = types.SimpleNamespace(numel=lambda: 8 * 64 * 128, element_size=lambda: 2)
    inp = types.SimpleNamespace(lens=[131072] * 8, num_kv_heads=8, q=q)
    assert sum(bench.decode_bytes(inp, 32)) == 100909056


def test_quantiles():
    q = bench.quantiles_us([0.031, 0.030, 0.032, 0.029, 0.033, 0.030, 0.031, 0.030, 0.034, 0.030])
    assert q == {"p10": 30.0, "p50": 30.5, "p90": 34.0}
    assert bench.quantiles_us([]) is None


def test_chunk_tiles_group_queries_by_block():
    assert msa.chunk_tiles(0, 0) == 0 and msa.chunk_tiles(128, 1) == 1 and msa.chunk_tiles(128, 64) == 1
    assert msa.chunk_tiles(128, 65) == 2 and msa.chunk_tiles(100, 28) == 1 and msa.chunk_tiles(100, 29) == 2
    assert msa.chunk_tile_rows(100, 100) == [(0, 0, 28), (1, 28, 92), (2, 92, 100)]
    assert msa.chunk_tile_rows(64, 130) == [(0, 0, 64), (1, 64, 128), (2, 128, 130)]
    assert msa.varlen_tiles([5, 70], [100, 60]) == 2 + 2


def test_prefill_flop_of_the_benchmark_chunk():
    # 8192 queries on a 131072-token prefix, 64 query heads, top-32 + diagonal:
    # 558.5 GFLOP sparse, 36.28 TFLOP dense (4 * 128 per visible pair)
    sparse, dense = bench.prefill_flop(131072, 8192, 32, 8, 8)
    assert sparse == 4 * 128 * 64 * (8192 * 32 * 64 + 128 * (64 * 65 // 2))
    assert round(sparse / 1e9, 1) == 558.5 and round(dense / 1e12, 2) == 36.28


def test_replicas_keep_inputs_out_of_l2():
    # the other replicas' steps between two uses of one move > 3 x 129 MB
    for step_bytes in (50_362_368, 100_909_056, 642_000_000):
        r = bench.replicas_needed(step_bytes)
        assert (r - 1) * step_bytes > 3 * bench.L2_BYTES and r >= 2
    assert bench.replicas_needed(100_909_056) == 6 and bench.replicas_needed(50_362_368) == 10


def test_chunk_batch_helpers():
    assert msa.varlen_tiles([0, 1, 64, 65, 128]) == 0 + 1 + 1 + 2 + 2
    n, starts, counts = msa._host_batch([0, 64, 128], [5, 0, 70])
    assert n == 3 and list(starts) == [0, 64, 128] and list(counts) == [5, 0, 70]
    with pytest.raises(ValueError):
        msa._host_batch([0, 64], [1])


def test_host_cpu_model_is_named():
    name = bench.host_cpu_model()
    assert isinstance(name, str) and name and name != "unknown"

"""Thin Python binding of the C ABI in include/msa.h (argument marshalling only).

Every function here has the name of the C entry point it calls and forwards
device pointers, sizes and a CUDA stream handle; all computation happens in the
CUDA kernels of ``libmsa.so``. Tensors are torch tensors (used only as device
memory); the stream defaults to torch's current stream.

There is no fallback: if the shared library is missing or fails to load, every
call raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "_lib", "libmsa.so")
_lib = None

MSA_OK, MSA_ERR_INVALID_ARG, MSA_ERR_UNSUPPORTED, MSA_ERR_WORKSPACE, MSA_ERR_CUDA, \
    MSA_ERR_DEVICE_BOUNDS, MSA_ERR_TIMEOUT = range(7)
MSA_DTYPE_F32, MSA_DTYPE_BF16 = 0, 1
MSA_KV_CONTIGUOUS, MSA_KV_PAGED = 0, 1
MSA_SCORE_MEAN_POOLED_KEYS, MSA_SCORE_TOKEN_MAX = 0, 1
(MSA_OP_POOL, MSA_OP_SELECT, MSA_OP_DECODE, MSA_OP_PREFILL, MSA_OP_DENSE_DECODE, MSA_OP_DENSE_PREFILL,
 MSA_OP_SELECT_PREFILL, MSA_OP_DECODE_STEP) = range(8)

# every symbol include/msa.h declares
EXPORTS = ["msa_workspace_size", "msa_workspace_init", "msa_pool_block_keys", "msa_select_topk_blocks",
           "msa_sparse_attn_decode", "msa_sparse_attn_prefill", "msa_dense_gqa_decode", "msa_dense_gqa_prefill",
           "msa_read_device_status", "msa_status_string", "msa_version", "msa_sparse_attn_decode_noalloc",
           "msa_sparse_decode_step", "msa_sparse_decode_step_pool", "msa_select_topk_blocks_varlen",
           "msa_sparse_attn_prefill_varlen", "msa_selftest_wait_timeout"]


class MsaError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)} ({status})")


class KvDesc(ctypes.Structure):
    _fields_ = [("layout", ctypes.c_int32), ("dtype", ctypes.c_int32), ("batch", ctypes.c_int32),
                ("num_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32), ("block_size", ctypes.c_int32),
                ("k", ctypes.c_void_p), ("v", ctypes.c_void_p), ("max_tokens", ctypes.c_int64),
                ("page_table", ctypes.c_void_p), ("max_pages_per_seq", ctypes.c_int32),
                ("num_pages", ctypes.c_int32), ("seq_lens", ctypes.c_void_p)]


class SelectCfg(ctypes.Structure):
    _fields_ = [("k_scored", ctypes.c_int32), ("force_local", ctypes.c_int32), ("q_tile", ctypes.c_int32),
                ("mode", ctypes.c_int32), ("q_start", ctypes.c_int64)]


_P = ctypes.c_void_p
_I32 = ctypes.c_int32
_I64 = ctypes.c_int64
_SZ = ctypes.c_size_t
_DESC = ctypes.POINTER(KvDesc)
_SIGS = {
    "msa_workspace_size": (_SZ, [_I32, _DESC, _I32, _I32, _I32]),
    "msa_workspace_init": (_I32, [_P, _SZ, _P]),
    "msa_pool_block_keys": (_I32, [_DESC, _I64, _I64, _P, _P, _SZ, _P]),
    "msa_select_topk_blocks": (_I32, [_P, _I32, _I32, _P, _DESC, ctypes.POINTER(SelectCfg), _P, _I32, _P, _P,
                                      _SZ, _P]),
    "msa_sparse_attn_decode": (_I32, [_P, _I32, _DESC, _P, _I32, ctypes.c_float, _P, _P, _P, _SZ, _P]),
    "msa_sparse_attn_prefill": (_I32, [_P, _I32, _I32, _I64, _DESC, _P, _I32, ctypes.c_float, _P, _P, _P, _SZ,
                                       _P]),
    "msa_dense_gqa_decode": (_I32, [_P, _I32, _DESC, ctypes.c_float, _P, _P, _P, _SZ, _P]),
    "msa_dense_gqa_prefill": (_I32, [_P, _I32, _I32, _I64, _DESC, ctypes.c_float, _P, _P, _P, _SZ, _P]),
    "msa_read_device_status": (_I32, [_P, _P, ctypes.POINTER(_I32)]),
    "msa_sparse_attn_decode_noalloc": (_I32, [_P, _I32, _DESC, _P, _I32, ctypes.c_float, _P, _P, _P]),
    "msa_sparse_decode_step": (_I32, [_P, _I32, _P, _DESC, ctypes.POINTER(SelectCfg), _P, _I32, ctypes.c_float, _P,
                                      _P, _P, _SZ, _P]),
    "msa_sparse_decode_step_pool": (_I32, [_P, _I32, _P, _DESC, ctypes.POINTER(SelectCfg), _P, _I32, ctypes.c_float,
                                           _P, _P, _P, _SZ, _P]),
    "msa_select_topk_blocks_varlen": (_I32, [_P, _I32, _I32, _P, _P, _P, _DESC, ctypes.POINTER(SelectCfg), _P, _I32,
                                             _P, _P, _SZ, _P]),
    "msa_sparse_attn_prefill_varlen": (_I32, [_P, _I32, _I32, _P, _P, _DESC, _P, _I32, ctypes.c_float, _P, _P, _P,
                                              _SZ, _P]),
    "msa_selftest_wait_timeout": (_I32, [_P, _SZ, _I64, _P]),
    "msa_status_string": (ctypes.c_char_p, [_I32]),
    "msa_version": (_I32, []),
}


def library_path() -> str:
    return _LIB_PATH


def load():
    """Load ``libmsa.so`` (built by ``sparse_attention_step_gb300.build``)."""
    global _lib
    if _lib is None:
        if not os.path.exists(_LIB_PATH):
            raise RuntimeError(f"{_LIB_PATH} is missing: build it with sparse_attention_step_gb300.build.build()")
        lib = ctypes.CDLL(_LIB_PATH)
        for name, (res, args) in _SIGS.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


def status_string(status: int) -> str:
    return load().msa_status_string(int(status)).decode()


def _check(status: int, where: str) -> None:
    if status != MSA_OK:
        raise MsaError(status, where)


def _ptr(t) -> int | None:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return MSA_DTYPE_BF16
    if t.dtype == torch.float32:
        return MSA_DTYPE_F32
    raise ValueError(f"unsupported dtype {t.dtype}")


def kv_desc(k: torch.Tensor, v: torch.Tensor, seq_lens: torch.Tensor, page_table: torch.Tensor | None = None,
            batch: int | None = None) -> KvDesc:
    """Describe a contiguous [B, Hkv, T, 128] or paged [P, Hkv, 64, 128] cache."""
    d = KvDesc()
    d.dtype = dtype_code(k)
    d.head_dim = k.shape[-1]
    d.block_size = 64
    d.k, d.v = _ptr(k), _ptr(v)
    d.seq_lens = _ptr(seq_lens)
    if page_table is None:
        d.layout = MSA_KV_CONTIGUOUS
        d.batch = k.shape[0]
        d.num_kv_heads = k.shape[1]
        d.max_tokens = k.shape[2]
    else:
        d.layout = MSA_KV_PAGED
        d.batch = page_table.shape[0] if batch is None else batch
        d.num_kv_heads = k.shape[1]
        d.block_size = k.shape[2]
        d.page_table = _ptr(page_table)
        d.max_pages_per_seq = page_table.shape[1]
        d.num_pages = k.shape[0]
    return d


def select_cfg(k_scored: int, force_local: bool = True, q_tile: int = 1, q_start: int = 0,
               mode: int = None, sink: bool = False) -> SelectCfg:
    return SelectCfg(int(k_scored), (1 if force_local else 0) | (2 if sink else 0), int(q_tile),
                     MSA_SCORE_MEAN_POOLED_KEYS if mode is None else int(mode), int(q_start))


# --------------------------------------------------------------------------- entry points

def msa_workspace_size(op: int, desc: KvDesc, num_q_heads: int, n_q_tokens: int, k_total: int) -> int:
    return int(load().msa_workspace_size(op, ctypes.byref(desc), num_q_heads, n_q_tokens, k_total))


def msa_workspace_init(ws, nbytes: int, stream=None) -> None:
    _check(load().msa_workspace_init(_ptr(ws), nbytes, _stream(stream)), "msa_workspace_init")


def msa_pool_block_keys(desc: KvDesc, first_block: int, n_blocks: int, pooled, ws=None, ws_bytes: int = 0,
                        stream=None) -> None:
    _check(load().msa_pool_block_keys(ctypes.byref(desc), first_block, n_blocks, _ptr(pooled), _ptr(ws), ws_bytes,
                                      _stream(stream)), "msa_pool_block_keys")


def msa_select_topk_blocks(q, num_q_heads: int, n_q_tokens: int, pooled, desc: KvDesc, cfg: SelectCfg, idx_out,
                           k_total: int, scores_out, ws, ws_bytes: int, stream=None) -> None:
    _check(load().msa_select_topk_blocks(_ptr(q), num_q_heads, n_q_tokens, _ptr(pooled), ctypes.byref(desc),
                                         ctypes.byref(cfg), _ptr(idx_out), k_total, _ptr(scores_out), _ptr(ws),
                                         ws_bytes, _stream(stream)), "msa_select_topk_blocks")


def _host_batch(q_starts, q_counts):
    """Host arrays of a chunk batch: (n_seqs, int64 starts, int32 counts), kept
    alive by the caller for the duration of the call."""
    n = len(q_starts)
    if len(q_counts) != n:
        raise ValueError("q_starts and q_counts differ in length")
    return n, (ctypes.c_int64 * n)(*[int(x) for x in q_starts]), (ctypes.c_int32 * n)(*[int(x) for x in q_counts])


def chunk_tiles(q_start: int, n: int) -> int:
    """Query tiles of a chunk of n new tokens at absolute positions q_start ..
    q_start + n - 1: its queries grouped by the 64-token block they sit in
    (rows of the chunk's index lists)."""
    q_start, n = int(q_start), int(n)
    if n <= 0:
        return 0
    return (q_start + n - 1) // 64 - q_start // 64 + 1


def chunk_tile_rows(q_start: int, n: int) -> list:
    """[(tile, first chunk row, end chunk row)] of a chunk's query tiles."""
    q_start, n = int(q_start), int(n)
    b0 = q_start // 64
    return [(j, max(0, (b0 + j) * 64 - q_start), min(n, (b0 + j + 1) * 64 - q_start))
            for j in range(chunk_tiles(q_start, n))]


def varlen_tiles(q_counts, q_starts=None) -> int:
    """Global query tiles of a chunk batch (rows of the varlen index lists)."""
    if q_starts is None:
        q_starts = [0] * len(q_counts)
    return sum(chunk_tiles(a, c) for a, c in zip(q_starts, q_counts))


def msa_select_topk_blocks_varlen(q, num_q_heads: int, q_starts, q_counts, pooled, desc: KvDesc, cfg: SelectCfg,
                                  idx_out, k_total: int, scores_out, ws, ws_bytes: int, stream=None) -> None:
    n, st, ct = _host_batch(q_starts, q_counts)
    _check(load().msa_select_topk_blocks_varlen(_ptr(q), num_q_heads, n, st, ct, _ptr(pooled), ctypes.byref(desc),
                                                ctypes.byref(cfg), _ptr(idx_out), k_total, _ptr(scores_out),
                                                _ptr(ws), ws_bytes, _stream(stream)), "msa_select_topk_blocks_varlen")


def msa_sparse_attn_prefill_varlen(q, num_q_heads: int, q_starts, q_counts, desc: KvDesc, idx, k_total: int,
                                   scale: float, out, lse, ws, ws_bytes: int, stream=None) -> None:
    n, st, ct = _host_batch(q_starts, q_counts)
    _check(load().msa_sparse_attn_prefill_varlen(_ptr(q), num_q_heads, n, st, ct, ctypes.byref(desc), _ptr(idx),
                                                 k_total, scale, _ptr(out), _ptr(lse), _ptr(ws), ws_bytes,
                                                 _stream(stream)), "msa_sparse_attn_prefill_varlen")


def msa_sparse_attn_decode(q, num_q_heads: int, desc: KvDesc, idx, k_total: int, scale: float, out, lse, ws,
                           ws_bytes: int, stream=None) -> None:
    _check(load().msa_sparse_attn_decode(_ptr(q), num_q_heads, ctypes.byref(desc), _ptr(idx), k_total, scale,
                                         _ptr(out), _ptr(lse), _ptr(ws), ws_bytes, _stream(stream)),
           "msa_sparse_attn_decode")


def msa_sparse_attn_prefill(q, num_q_heads: int, n_q_tokens: int, q_start: int, desc: KvDesc, idx, k_total: int,
                            scale: float, out, lse, ws, ws_bytes: int, stream=None) -> None:
    _check(load().msa_sparse_attn_prefill(_ptr(q), num_q_heads, n_q_tokens, q_start, ctypes.byref(desc), _ptr(idx),
                                          k_total, scale, _ptr(out), _ptr(lse), _ptr(ws), ws_bytes,
                                          _stream(stream)), "msa_sparse_attn_prefill")


def msa_sparse_decode_step(q, num_q_heads: int, pooled, desc: KvDesc, cfg: SelectCfg, idx_out, k_total: int,
                           scale: float, out, lse, ws, ws_bytes: int, stream=None) -> None:
    _check(load().msa_sparse_decode_step(_ptr(q), num_q_heads, _ptr(pooled), ctypes.byref(desc), ctypes.byref(cfg),
                                         _ptr(idx_out), k_total, scale, _ptr(out), _ptr(lse), _ptr(ws), ws_bytes,
                                         _stream(stream)), "msa_sparse_decode_step")


def msa_sparse_decode_step_pool(q, num_q_heads: int, pooled, desc: KvDesc, cfg: SelectCfg, idx_out, k_total: int,
                                scale: float, out, lse, ws, ws_bytes: int, stream=None) -> None:
    _check(load().msa_sparse_decode_step_pool(_ptr(q), num_q_heads, _ptr(pooled), ctypes.byref(desc),
                                              ctypes.byref(cfg), _ptr(idx_out), k_total, scale, _ptr(out), _ptr(lse),
                                              _ptr(ws), ws_bytes, _stream(stream)), "msa_sparse_decode_step_pool")


def msa_dense_gqa_decode(q, num_q_heads: int, desc: KvDesc, scale: float, out, lse, ws, ws_bytes: int,
                         stream=None) -> None:
    _check(load().msa_dense_gqa_decode(_ptr(q), num_q_heads, ctypes.byref(desc), scale, _ptr(out), _ptr(lse),
                                       _ptr(ws), ws_bytes, _stream(stream)), "msa_dense_gqa_decode")


def msa_dense_gqa_prefill(q, num_q_heads: int, n_q_tokens: int, q_start: int, desc: KvDesc, scale: float, out, lse,
                          ws, ws_bytes: int, stream=None) -> None:
    _check(load().msa_dense_gqa_prefill(_ptr(q), num_q_heads, n_q_tokens, q_start, ctypes.byref(desc), scale,
                                        _ptr(out), _ptr(lse), _ptr(ws), ws_bytes, _stream(stream)),
           "msa_dense_gqa_prefill")


def msa_sparse_attn_decode_noalloc(q, num_q_heads: int, desc: KvDesc, idx, k_total: int, scale: float, out, lse,
                                   stream=None) -> None:
    """msa_sparse_attn_decode for callers that cannot allocate device memory:
    the split-K scratch is a fixed 4 MiB array inside the library."""
    _check(load().msa_sparse_attn_decode_noalloc(_ptr(q), num_q_heads, ctypes.byref(desc), _ptr(idx), k_total, scale,
                                                 _ptr(out), _ptr(lse), _stream(stream)),
           "msa_sparse_attn_decode_noalloc")


def msa_selftest_wait_timeout(ws, ws_bytes: int, limit_cycles: int, stream=None) -> None:
    _check(load().msa_selftest_wait_timeout(_ptr(ws), ws_bytes, limit_cycles, _stream(stream)),
           "msa_selftest_wait_timeout")


def msa_read_device_status(ws, stream=None) -> int:
    out = _I32(0)
    _check(load().msa_read_device_status(_ptr(ws), _stream(stream), ctypes.byref(out)), "msa_read_device_status")
    return int(out.value)


def msa_status_string(status: int) -> str:
    return status_string(status)


def msa_version() -> int:
    return int(load().msa_version())


# --------------------------------------------------------------------------- conveniences

class Workspace:
    """A zero-initialised device workspace of at least ``nbytes`` bytes."""

    def __init__(self, nbytes: int, device="cuda"):
        self.nbytes = max(int(nbytes), 256)
        self.buf = torch.empty(self.nbytes, dtype=torch.uint8, device=device)
        msa_workspace_init(self.buf, self.nbytes)

    def ptr(self) -> int:
        return self.buf.data_ptr()


def pooled_shape(desc: KvDesc) -> tuple:
    """Summary keys: one row per (sequence, KV head, logical block), either cache layout."""
    blocks = desc.max_tokens // 64 if desc.layout == MSA_KV_CONTIGUOUS else desc.max_pages_per_seq
    return (desc.batch, desc.num_kv_heads, blocks, desc.head_dim)

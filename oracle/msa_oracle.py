"""Plain CPU oracle for two-stage GQA block-sparse attention (Python binding).

TEST INFRASTRUCTURE. Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this module. The arithmetic lives
in ``oracle/msa_oracle.c`` (scalar C, double accumulation, OpenMP only across
independent units), built by ``oracle/build.py`` into ``oracle/_build``; this
module only passes arrays to it and assembles the per-unit steps in the order
the guide gives them. It imports nothing from the CUDA library and the CUDA
library never calls it: the two share no code.

What it computes follows the "MiniMax Sparse Attention" diagram as described
in the Atlas Cloud guide "MiniMax goes sparse: decoding M3's attention from a
single diagram" (Portuguese, Spanish and French editions):

* Step 1, the index branch (guide §1, "Step 1: index branch"): one index query
  per GQA group, block-level scores, and a top-k that keeps a short list of KV
  blocks per layer and per group.
* Step 2, the sparse branch (guide §1, "Step 2: sparse branch"): ordinary
  softmax attention of every query head of a group over the real, uncompressed
  K/V of the blocks its group selected.

The guide's formulas were lost in extraction, so these readings fill them in:

* Block summary: the mean of the block's 64 keys of the KV head itself,
  summed in double, divided by 64 and rounded to nearest even into the
  storage type (one rounding, from double). Scoring the mean key equals the
  mean over the block of the token-level scores (linearity).
* Index query of a group: the sum of the group's query heads (and, for a
  prefill tile, of the tile's query tokens).
* The block holding the newest token (decode) or the query tile's own
  diagonal block (prefill) is always kept and never scored; ties in the top-k
  go to the lower block index.
* A prefill tile is the set of chunk queries that sit in one 64-token block
  of the sequence; a chunk that starts inside a block has a shorter first
  tile, so each tile has exactly one diagonal block (:func:`prefill_tiles`).

Array arguments may be numpy arrays (float64 or float32) or CPU torch tensors
(float32, float64 or bfloat16); every value is read exactly as its bits encode.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

BLOCK = 64          # tokens per KV block (the guide's assumed block size, §3)
HEAD_DIM = 128

_F64, _F32, _BF16 = 0, 1, 2
_lib = None


def _load():
    global _lib
    if _lib is None:
        from oracle import build as _build
        path = _build.build()
        lib = ctypes.CDLL(path)
        P, I, I64, D = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_double
        sigs = {
            "ora_round_bf16": (D, [D]),
            "ora_store": (D, [D, I]),
            "ora_pool_block_keys": (I64, [P, I, I64, I64, I, P, P]),
            "ora_index_query": (None, [P, I, I64, P]),
            "ora_score_blocks": (None, [P, P, I64, P]),
            "ora_score_blocks_token_max": (None, [P, P, I, I64, I64, P]),
            "ora_select_blocks": (I64, [P, I64, I64, I64, I64, I, I64, P]),
            "ora_attend": (None, [P, I, I64, P, P, I, I64, P, I64, D, P, P, P]),
            "ora_dense_gqa": (None, [P, I, I64, P, P, I, I64, I64, D, P, P]),
            "ora_decode_select_units": (I, [I64, P, I, I, P, I, I64, I64, P, I, I64, I, I64, I64, P, P, P, P]),
            "ora_decode_step_units": (I, [I64, P, I, I, P, I64, P, P, I, I64, I64, P, I64, I, I64, D, P, P, P]),
            "ora_prefill_tile_units": (I, [I64, P, P, P, P, I64, P, I, I, I, P, I64, P, P, I, I64, I64, I64, D, P, P,
                                            P]),
            "ora_num_threads": (I, []),
        }
        for name, (res, args) in sigs.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


class _Src:
    """A read-only array handed to C: pointer, element type, and the owner
    kept alive for the call."""

    def __init__(self, x):
        try:
            import torch
        except ImportError:  # pragma: no cover
            torch = None
        if torch is not None and isinstance(x, torch.Tensor):
            t = x.detach()
            if t.device.type != "cpu":
                t = t.cpu()
            t = t.contiguous()
            if t.dtype == torch.bfloat16:
                self.arr, self.type = t.view(torch.int16).numpy(), _BF16
            elif t.dtype == torch.float32:
                self.arr, self.type = t.numpy(), _F32
            else:
                self.arr, self.type = t.to(torch.float64).numpy(), _F64
        else:
            a = np.asarray(x)
            if a.dtype == np.float32:
                self.arr, self.type = np.ascontiguousarray(a), _F32
            else:
                self.arr, self.type = np.ascontiguousarray(a, dtype=np.float64), _F64
        self.shape = self.arr.shape
        self.ptr = self.arr.ctypes.data


def _src(x) -> _Src:
    return x if isinstance(x, _Src) else _Src(x)


def _f64(x) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def num_threads() -> int:
    """Threads the C oracle's unit-parallel functions use (OpenMP)."""
    return int(_load().ora_num_threads())


# ---------------------------------------------------------------------------
# Rounding into the storage type
# ---------------------------------------------------------------------------

def round_to_bf16(x) -> np.ndarray:
    """Round each value to the nearest bfloat16, ties to even, in one step
    from its exact value (no binary32 rounding on the way). Returns float64."""
    lib = _load()
    a = _f64(x)
    out = np.array([lib.ora_round_bf16(float(v)) for v in a.ravel()], dtype=np.float64)
    return out.reshape(a.shape)


def store_as(x, store: str) -> np.ndarray:
    """Value of ``x`` once written in the storage type ``store`` ("bf16" or
    "f32"), rounded to nearest even."""
    codes = {"bf16": _BF16, "f32": _F32}
    if store not in codes:
        raise ValueError(f"unknown storage type {store!r}")
    lib = _load()
    a = _f64(x)
    out = np.array([lib.ora_store(float(v), codes[store]) for v in a.ravel()], dtype=np.float64)
    return out.reshape(a.shape)


# ---------------------------------------------------------------------------
# Step 1: index branch
# ---------------------------------------------------------------------------

def num_blocks(seq_len: int) -> int:
    """Blocks that hold at least one token: ceil(seq_len / 64)."""
    return -(-int(seq_len) // BLOCK)


def num_full_blocks(seq_len: int) -> int:
    """Blocks whose 64 tokens are all present; only these get a summary key."""
    return int(seq_len) // BLOCK


def pool_block_keys(k_rows, seq_len: int, store: str):
    """Block summary keys of one (sequence, KV head): ``(stored, exact)``,
    each [seq_len // 64, D] float64. exact = mean of the block's 64 keys
    (double sum / 64), stored = exact rounded to nearest even into ``store``.
    Guide §1, Step 1 (block pooling of the index branch; the mean replaces the
    guide's max, see the module notes)."""
    codes = {"bf16": _BF16, "f32": _F32}
    if store not in codes:
        raise ValueError(f"unknown storage type {store!r}")
    src = _src(k_rows)
    nbf = num_full_blocks(seq_len)
    if nbf and src.shape[0] < nbf * BLOCK:
        raise ValueError("fewer key rows than complete blocks")
    stored = np.empty((nbf, HEAD_DIM))
    exact = np.empty((nbf, HEAD_DIM))
    _load().ora_pool_block_keys(src.ptr, src.type, src.shape[1], int(seq_len), codes[store], _ptr(stored),
                                _ptr(exact))
    return stored, exact


def index_query(q_rows) -> np.ndarray:
    """One index query per GQA group: the sum of the group's query vectors.

    ``q_rows``: [..., D] -- the G heads of one group for a decode token, or the
    tokens x G heads of a prefill tile. Guide §1, Step 1 ("Idx Q", one per
    group; six heads share two index queries in the diagram).
    """
    src = _src(q_rows)
    n = int(np.prod(src.shape[:-1])) if len(src.shape) > 1 else 1
    out = np.empty(HEAD_DIM)
    _load().ora_index_query(src.ptr, src.type, n, _ptr(out))
    return out


def score_blocks(q_idx, pooled, n_cand: int) -> np.ndarray:
    """Score of candidate blocks 0..n_cand-1: q_idx . summary_key[b] (double,
    unscaled: a positive scale does not change the ranking). Guide §1, Step 1."""
    q = _f64(q_idx)
    p = _f64(pooled).reshape(-1, HEAD_DIM)
    n = int(n_cand)
    if n > p.shape[0]:
        raise ValueError("more candidates than summaries")
    out = np.empty(n)
    _load().ora_score_blocks(_ptr(q), _ptr(p), n, _ptr(out))
    return out


def _select(scores, k_scored, forced, k_total, first, keep0) -> np.ndarray:
    sc = _f64(scores)
    sel = np.empty(int(k_total), dtype=np.int64)
    got = _load().ora_select_blocks(_ptr(sc), sc.shape[0], int(k_scored), -1 if forced is None else int(forced),
                                    int(first), int(bool(keep0)), int(k_total), _ptr(sel))
    if got < 0:
        raise ValueError("k_total too small for the selection")
    return sel


def select_blocks(scores, k_scored: int, forced: int | None, k_total: int) -> np.ndarray:
    """Top-k of the candidate scores plus the always-kept block: candidates
    ranked by score, highest first, ties to the lower block index; the first
    ``min(k_scored, n)`` kept, the forced block (if any) added, the list sorted
    ascending and padded with -1 to ``k_total``. Guide §1, Step 1 (TopK keeps the
    k best-scoring KV blocks per layer and group; output lists I1, I2)."""
    return _select(scores, k_scored, forced, k_total, 0, False)


def select_blocks_sink(scores, k_scored: int, forced: int | None, k_total: int, has_block0: bool) -> np.ndarray:
    """Selection with an attention sink: block 0 is always kept and never
    scored (the guide, §2, names a sink as one likely replacement for the
    dropped sliding window). Blocks 1..n-1 are ranked, the best
    ``min(k_scored, n - 1)`` kept, then block 0 (when the sequence has it) and
    the forced block, ascending, padded with -1."""
    return _select(scores, k_scored, forced, k_total, 1, has_block0)


def boundary_gap(scores, k_scored: int):
    """(s_k, s_{k+1}) of the ranked candidate scores, or None when all are kept."""
    s = np.sort(_f64(scores))[::-1]
    if k_scored <= 0 or s.shape[0] <= k_scored:
        return None
    return float(s[k_scored - 1]), float(s[k_scored])


def score_blocks_token_max(q_idx, kidx_rows, n_cand: int) -> np.ndarray:
    """Guide-literal block score of candidate blocks 0..n_cand-1 (double):
    token-level scores q_idx . K_idx[t] against a single index-key head shared
    by every group of the layer, then a max over the 64 tokens of each block
    (guide §1, Step 1 as drawn). ``kidx_rows``: [>= 64 n_cand, D]."""
    q = _f64(q_idx)
    src = _src(kidx_rows)
    n = int(n_cand)
    if n and src.shape[0] < n * BLOCK:
        raise ValueError("fewer index-key rows than candidate blocks")
    out = np.empty(n)
    _load().ora_score_blocks_token_max(_ptr(q), src.ptr, src.type, src.shape[1], n, _ptr(out))
    return out


def select_token_max(q_group, kidx_rows, seq_len, k_scored, k_total, force_local=True):
    """Step 1 with the token-level max-pooled score for one (sequence, KV
    head): index query (group sum), token scores against the shared index
    keys, block max, top-k plus the newest block."""
    nb = num_blocks(seq_len)
    nbf = num_full_blocks(seq_len)
    forced = nb - 1 if force_local else None
    n_cand = min(nbf, nb - 1) if force_local else nbf
    n_cand = max(n_cand, 0)
    q_idx = index_query(q_group)
    scores = score_blocks_token_max(q_idx, kidx_rows, n_cand)
    sel = select_blocks(scores, k_scored, forced, k_total)
    return dict(selected=sel, scores=scores, q_idx=q_idx, forced=forced, n_cand=n_cand)


# ---------------------------------------------------------------------------
# Step 2: sparse branch
# ---------------------------------------------------------------------------

def tokens_of_blocks(blocks, seq_len: int, last_pos: int | None = None) -> np.ndarray:
    """Token positions covered by ``blocks`` (ignoring -1), below ``seq_len``
    and, for a causal query at ``last_pos``, not after it."""
    toks = []
    limit = int(seq_len) if last_pos is None else min(int(seq_len), int(last_pos) + 1)
    for b in blocks:
        b = int(b)
        if b < 0:
            continue
        lo = b * BLOCK
        hi = min(lo + BLOCK, limit)
        if hi > lo:
            toks.append(np.arange(lo, hi))
    if not toks:
        return np.zeros(0, dtype=np.int64)
    return np.concatenate(toks).astype(np.int64)


def attend(q_heads, k_rows, v_rows, tokens, scale: float):
    """Softmax attention of each query vector over the token set ``tokens``:
    z_t = (q . K[t]) * scale, p = softmax_t(z), o = sum_t p_t V[t]. Returns
    ``(o [H, D], lse [H], p [H, n])`` with lse = log sum_t exp(z_t). Guide §1,
    Step 2 (the gathered subsets of the real K/V go through ordinary softmax
    attention; every head of a group uses its group's selection)."""
    q = _src(q_heads)
    k = _src(k_rows)
    v = _src(v_rows)
    if k.type != v.type or k.shape != v.shape:
        raise ValueError("k and v must have the same type and shape")
    toks = np.ascontiguousarray(np.asarray(tokens, dtype=np.int64))
    if toks.size and (toks.min() < 0 or toks.max() >= k.shape[0]):
        raise ValueError("token outside the key rows")
    h = int(np.prod(q.shape[:-1])) if len(q.shape) > 1 else 1
    n = toks.shape[0]
    o = np.empty((h, HEAD_DIM))
    lse = np.empty(h)
    p = np.empty((h, n))
    _load().ora_attend(q.ptr, q.type, h, k.ptr, v.ptr, k.type, k.shape[1], _ptr(toks), n, float(scale), _ptr(o),
                       _ptr(lse), _ptr(p) if n else None)
    return o, lse, p


# ---------------------------------------------------------------------------
# Whole units: one decode (sequence, KV head) and one prefill (tile, KV head)
# ---------------------------------------------------------------------------

def decode_unit(q_group, k_rows, v_rows, seq_len, k_scored, k_total, scale, store,
                force_local=True, selected=None, pooled=None):
    """Decode step for one (sequence, KV head): pool, index query, score,
    select, attend. ``q_group``: [G, D] query heads of the group.

    Candidates are the complete blocks, minus the newest block when it is
    forced. ``selected`` overrides the selection (to attend over another
    valid set). Returns a dict with the intermediate values.
    """
    nb = num_blocks(seq_len)
    if pooled is None:
        pooled, _ = pool_block_keys(k_rows, seq_len, store)
    nbf = pooled.shape[0]
    forced = nb - 1 if force_local else None
    n_cand = min(nbf, nb - 1) if force_local else nbf
    n_cand = max(n_cand, 0)
    q_idx = index_query(q_group)
    scores = score_blocks(q_idx, pooled, n_cand)
    sel = select_blocks(scores, k_scored, forced, k_total)
    use = sel if selected is None else np.asarray(selected)
    toks = tokens_of_blocks(use, seq_len)
    o, lse, p = attend(q_group, k_rows, v_rows, toks, scale)
    return dict(selected=sel, scores=scores, q_idx=q_idx, pooled=pooled, o=o, lse=lse, p=p,
                tokens=toks, forced=forced, n_cand=n_cand)


def prefill_tiles(q_start: int, n_new: int):
    """The query tiles of a chunk of ``n_new`` tokens at absolute positions
    q_start .. q_start + n_new - 1: a tile is the chunk's queries that sit in one
    64-token block. Returns [(tile_index, row_lo, row_hi)] over chunk rows; the
    tile's diagonal block is q_start // 64 + tile_index. A 64-aligned q_start
    gives tiles of 64 rows (the last one ragged); an unaligned one a shorter
    first tile."""
    q_start, n_new = int(q_start), int(n_new)
    out = []
    if n_new <= 0:
        return out
    b0 = q_start // BLOCK
    last = (q_start + n_new - 1) // BLOCK
    for j in range(last - b0 + 1):
        lo = max(0, (b0 + j) * BLOCK - q_start)
        hi = min(n_new, (b0 + j + 1) * BLOCK - q_start)
        out.append((j, lo, hi))
    return out


def prefill_tile_select(q_tile, tile_index, q_start, pooled, k_scored, k_total):
    """Selection for one (query tile, KV head) of a chunked prefill.

    ``q_tile``: [R, G, D] (the R <= 64 tokens of the tile, G heads of the
    group). The tile's diagonal block is q_start // 64 + tile_index; candidates
    are the blocks before it. Guide §3 (during prefill the index branch still
    scans the whole input) and §1, Step 1.
    """
    diag = int(q_start) // BLOCK + int(tile_index)
    q_idx = index_query(q_tile)
    scores = score_blocks(q_idx, pooled, diag)
    sel = select_blocks(scores, k_scored, diag, k_total)
    return dict(selected=sel, scores=scores, q_idx=q_idx, diag=diag)


def prefill_tile_select_token_max(q_tile, tile_index, q_start, kidx_rows, k_scored, k_total):
    """Selection for one (query tile, KV head) of a chunked prefill with the
    guide-literal block score: the tile's index query (sum over its tokens and
    the group's heads) against every token of the shared index-key head, max
    over each block's 64 tokens; candidates are the blocks before the tile's
    diagonal block q_start // 64 + tile_index, which is always kept. Guide §1,
    Step 1 as drawn, and §3 (in prefill the index branch scans the whole input).
    """
    diag = int(q_start) // BLOCK + int(tile_index)
    q_idx = index_query(q_tile)
    scores = score_blocks_token_max(q_idx, kidx_rows, diag)
    sel = select_blocks(scores, k_scored, diag, k_total)
    return dict(selected=sel, scores=scores, q_idx=q_idx, diag=diag)


def prefill_rows(q_rows, positions, k_rows, v_rows, seq_len, blocks, scale):
    """Causal attention of prefill query rows over the selected blocks.

    ``q_rows``: [R, G, D] at absolute ``positions`` [R]. Each row sees the
    tokens of ``blocks`` that are not after its own position.
    Returns ``(o [R, G, D], lse [R, G])``.
    """
    k, v = _src(k_rows), _src(v_rows)
    r, g = q_rows.shape[0], q_rows.shape[1]
    o = np.zeros((r, g, HEAD_DIM))
    lse = np.zeros((r, g))
    for i in range(r):
        toks = tokens_of_blocks(blocks, seq_len, last_pos=int(positions[i]))
        oi, li, _ = attend(q_rows[i], k, v, toks, scale)
        o[i], lse[i] = oi, li
    return o, lse


# ---------------------------------------------------------------------------
# Dense causal GQA attention (the full-attention comparator)
# ---------------------------------------------------------------------------

def dense_gqa(q_heads, k_rows, v_rows, position: int, scale: float):
    """Full causal attention of the query heads at ``position`` over tokens
    0..position of their shared KV head: softmax(q K^T * scale) V, written in C
    apart from :func:`attend` (a running-max softmax, no shared code), so the
    sparse path with every block selected can be checked against it. The
    full-attention baseline the guide's speed-ups are quoted against (§3)."""
    q = _src(q_heads)
    k = _src(k_rows)
    v = _src(v_rows)
    if k.type != v.type or k.shape != v.shape:
        raise ValueError("k and v must have the same type and shape")
    if int(position) >= k.shape[0]:
        raise ValueError("position beyond the key rows")
    h = int(np.prod(q.shape[:-1])) if len(q.shape) > 1 else 1
    o = np.empty((h, HEAD_DIM))
    lse = np.empty(h)
    _load().ora_dense_gqa(q.ptr, q.type, h, k.ptr, v.ptr, k.type, k.shape[1], int(position), float(scale), _ptr(o),
                          _ptr(lse))
    return o, lse


# ---------------------------------------------------------------------------
# Many decode units at once (OpenMP across units)
# ---------------------------------------------------------------------------

def decode_select_units(q, k, lens, store, k_scored, k_total, force_local=1, max_blocks=None,
                        want_scores=False, want_pooled=False):
    """Step 1 (pool from the keys, index query, scores, top-k) for U units.

    ``q``: [U, G, D]; ``k``: [U, T, D] (each unit's key rows in token order);
    ``lens``: U lengths. ``force_local`` is the bit set of the library's
    selection config (1: newest block kept; 2: block 0 kept as a sink).
    Returns dict(selected [U, k_total], gap [U, 2] (NaN where every candidate is
    kept), scores [U, max_blocks] and pooled [U, max_blocks, D] if asked; NaN
    past each unit's candidates / complete blocks)."""
    qs, ks = _Src(q), _Src(k)
    u, g = qs.shape[0], qs.shape[1]
    t = ks.shape[1]
    lens64 = np.ascontiguousarray(np.asarray(lens, dtype=np.int64))
    if ks.shape[0] != u or lens64.shape[0] != u or (lens64 > t).any():
        raise ValueError("unit count or lengths do not match the keys")
    mb = int(max_blocks) if max_blocks is not None else num_blocks(t)
    sel = np.empty((u, int(k_total)), dtype=np.int64)
    gap = np.empty((u, 2))
    scores = np.empty((u, mb)) if want_scores else None
    pooled = np.empty((u, mb, HEAD_DIM)) if want_pooled else None
    code = {"bf16": _BF16, "f32": _F32}[store]
    rc = _load().ora_decode_select_units(u, qs.ptr, qs.type, g, ks.ptr, ks.type, t * HEAD_DIM, HEAD_DIM,
                                         _ptr(lens64), code, int(k_scored), int(force_local), int(k_total), mb,
                                         _ptr(sel), None if scores is None else _ptr(scores),
                                         None if pooled is None else _ptr(pooled), _ptr(gap))
    if rc != 0:
        raise ValueError("bad arguments to decode_select_units")
    return dict(selected=sel, gap=gap, scores=scores, pooled=pooled)


def decode_step_units(q, pooled, k, v, lens, k_scored, k_total, scale, force_local=1):
    """A whole decode step for U units from their stored summaries: index
    query, scores, top-k, then softmax attention of the G heads over the
    selected blocks (tokens below each length). ``q`` [U, G, D]; ``pooled``
    [U, max_blocks, D] (float64); ``k``, ``v`` [U, T, D]. Returns
    (selected [U, k_total], o [U, G, D], lse [U, G])."""
    qs, ks, vs = _Src(q), _Src(k), _Src(v)
    u, g = qs.shape[0], qs.shape[1]
    t = ks.shape[1]
    pl = _f64(pooled)
    lens64 = np.ascontiguousarray(np.asarray(lens, dtype=np.int64))
    if ks.type != vs.type or ks.shape != vs.shape or pl.shape[0] != u or (lens64 > t).any():
        raise ValueError("inconsistent decode_step_units arguments")
    sel = np.empty((u, int(k_total)), dtype=np.int64)
    o = np.empty((u, g, HEAD_DIM))
    lse = np.empty((u, g))
    rc = _load().ora_decode_step_units(u, qs.ptr, qs.type, g, _ptr(pl), pl.shape[1], ks.ptr, vs.ptr, ks.type,
                                       t * HEAD_DIM, HEAD_DIM, _ptr(lens64), int(k_scored), int(force_local),
                                       int(k_total), float(scale), _ptr(sel), _ptr(o), _ptr(lse))
    if rc != 0:
        raise ValueError("bad arguments to decode_step_units")
    return sel, o, lse


def prefill_tile_units(units, q_start, q, pooled, k, v, k_scored, k_total, scale):
    """Select and attend for chunked-prefill units of one sequence, in C with
    OpenMP across units. ``units``: [(tile, head)]; tiles follow
    :func:`prefill_tiles`. ``q`` [n_rows, Hq, D]; ``pooled`` [Hkv, max_blocks, D]
    (float64 stored summaries); ``k``, ``v`` [Hkv, T, D]. Returns (selected
    [U, k_total], o [n_rows, Hq, D], lse [n_rows, Hq]) (rows and heads of
    units not listed are NaN)."""
    qs, ks, vs = _Src(q), _Src(k), _Src(v)
    n_rows, hq = qs.shape[0], qs.shape[1]
    hkv, t = ks.shape[0], ks.shape[1]
    g = hq // hkv
    part = {j: (lo, hi) for j, lo, hi in prefill_tiles(q_start, n_rows)}
    tiles = np.ascontiguousarray([u[0] for u in units], dtype=np.int64)
    heads = np.ascontiguousarray([u[1] for u in units], dtype=np.int64)
    lo = np.ascontiguousarray([part[u[0]][0] for u in units], dtype=np.int64)
    hi = np.ascontiguousarray([part[u[0]][1] for u in units], dtype=np.int64)
    pl = _f64(pooled)
    sel = np.empty((len(units), int(k_total)), dtype=np.int64)
    o = np.full((n_rows, hq, HEAD_DIM), np.nan)
    lse = np.full((n_rows, hq), np.nan)
    rc = _load().ora_prefill_tile_units(len(units), _ptr(tiles), _ptr(heads), _ptr(lo), _ptr(hi), int(q_start),
                                        qs.ptr, qs.type, hq, g, _ptr(pl), pl.shape[1], ks.ptr, vs.ptr, ks.type, t,
                                        int(k_scored), int(k_total), float(scale), _ptr(sel), _ptr(o), _ptr(lse))
    if rc != 0:
        raise ValueError("bad arguments to prefill_tile_units")
    return sel, o, lse

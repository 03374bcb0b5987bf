"""Plain CPU oracle for two-stage GQA block-sparse attention.

TEST INFRASTRUCTURE. Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this module. The CUDA library never
calls it, and it imports nothing from the CUDA library: the two share no code.

What it computes follows the "MiniMax Sparse Attention" diagram as described
in the Atlas Cloud guide "MiniMax goes sparse: decoding M3's attention from a
single diagram" (Portuguese, Spanish and French editions):

* Step 1, the index branch (guide §1, "Step 1: index branch"): one index query
  per GQA group, block-level scores, and a top-k that keeps a short list of KV
  blocks per layer and per group.
* Step 2, the sparse branch (guide §1, "Step 2: sparse branch"): ordinary
  softmax attention of every query head of a group over the real, uncompressed
  K/V of the blocks its group selected.

The guide's formulas were lost in extraction, so the readings below fill them
in (each is listed in the design notes):

* Block summary: the mean of the block's 64 keys of the KV head itself.
  Because the score is linear in the key, the mean-pooled key scored against
  the index query equals the mean over the block of token-level scores (the
  guide pools token scores with a max; the mean is the stated choice here).
* Index query of a group: the sum of the group's query heads (and, for a
  prefill tile, of the tile's query tokens). Summing scores over the heads of a
  group equals scoring once with this summed query.
* The block holding the newest token (decode) or the query tile's own diagonal
  block (prefill) is always kept and never scored.
* Ties in the top-k go to the lower block index.
* The stored block summary is a quantised code decided by floating point, so
  the oracle takes that decision in the kernel's precision: fp32 accumulation
  over the 64 rows in row order, one exact scaling by 1/64, then
  round-to-nearest-even into the storage type. Everything else is float64.

Every array argument holds the exact values of the bf16/fp32 inputs as float64.
"""
from __future__ import annotations

import numpy as np

BLOCK = 64          # tokens per KV block (the guide's assumed block size, §3)
HEAD_DIM = 128


# ---------------------------------------------------------------------------
# Rounding into the storage type
# ---------------------------------------------------------------------------

def round_f32_to_bf16(x) -> np.ndarray:
    """Round float32 values to bfloat16 with round-to-nearest-even.

    bfloat16 keeps the upper 16 bits of the IEEE binary32 pattern. Rounding adds
    half a unit of the kept part, plus one when the kept part is odd (ties go
    to even), then truncates. NaN stays NaN. Returned as exact float64 values.
    """
    x32 = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    bits = x32.view(np.uint32).astype(np.uint64)
    lsb = (bits >> np.uint64(16)) & np.uint64(1)
    rounded = (bits + np.uint64(0x7FFF) + lsb) >> np.uint64(16)
    nan = np.isnan(x32)
    rounded = np.where(nan, (bits >> np.uint64(16)) | np.uint64(0x40), rounded)
    out_bits = (rounded.astype(np.uint32) << np.uint32(16)).astype(np.uint32)
    return out_bits.view(np.float32).astype(np.float64)


def store_as(x32: np.ndarray, store: str) -> np.ndarray:
    """Value of float32 ``x32`` once written in the storage type ``store``."""
    if store == "bf16":
        return round_f32_to_bf16(x32)
    if store == "f32":
        return np.asarray(x32, dtype=np.float32).astype(np.float64)
    raise ValueError(f"unknown storage type {store!r}")


# ---------------------------------------------------------------------------
# Step 1: index branch
# ---------------------------------------------------------------------------

def num_blocks(seq_len: int) -> int:
    """Blocks that hold at least one token: ceil(seq_len / 64)."""
    return -(-int(seq_len) // BLOCK)


def num_full_blocks(seq_len: int) -> int:
    """Blocks whose 64 tokens are all present; only these get a summary key."""
    return int(seq_len) // BLOCK


def pool_block_keys(k_rows: np.ndarray, seq_len: int, store: str):
    """Block summary keys of one (sequence, KV head).

    ``k_rows``: [>= seq_len, D] keys of the head. For each complete block b the
    summary is mean_{i<64} K[64 b + i]. Returns ``(stored, exact)``: the value
    written in the storage type (fp32 row-order sum, times 1/64, rounded to
    nearest even) and the float64 mean for diagnostics. Guide §1, Step 1 (block
    pooling of the index branch); the mean replaces the guide's max (see module
    notes).
    """
    nbf = num_full_blocks(seq_len)
    d = k_rows.shape[1]
    blocks = np.asarray(k_rows[: nbf * BLOCK], dtype=np.float64).reshape(nbf, BLOCK, d)
    acc = np.zeros((nbf, d), dtype=np.float32)
    for i in range(BLOCK):  # row order, one fp32 add per row
        acc = (acc + blocks[:, i, :].astype(np.float32)).astype(np.float32)
    mean32 = (acc * np.float32(1.0 / BLOCK)).astype(np.float32)
    stored = store_as(mean32, store)
    exact = blocks.mean(axis=1)
    return stored, exact


def index_query(q_rows: np.ndarray) -> np.ndarray:
    """One index query per GQA group: the sum of the group's query vectors.

    ``q_rows``: [..., D] -- the G heads of one group for a decode token, or the
    64 tokens x G heads of a prefill tile. Guide §1, Step 1 ("Idx Q", one per
    group; six heads share two index queries in the diagram).
    """
    q = np.asarray(q_rows, dtype=np.float64)
    return q.reshape(-1, q.shape[-1]).sum(axis=0)


def score_blocks(q_idx: np.ndarray, pooled: np.ndarray, n_cand: int) -> np.ndarray:
    """Score of candidate blocks 0..n_cand-1: q_idx . summary_key[b] (float64).

    Unscaled: a positive scale does not change the ranking. Guide §1, Step 1
    (scoring of the index query against the index keys).
    """
    return np.asarray(pooled[:n_cand], dtype=np.float64) @ np.asarray(q_idx, dtype=np.float64)


def select_blocks(scores: np.ndarray, k_scored: int, forced: int | None, k_total: int) -> np.ndarray:
    """Top-k of the candidate scores plus the always-kept block.

    Candidates are ranked by score, highest first, ties to the lower block
    index; the first ``min(k_scored, n)`` are kept, the forced block (if any) is
    added, the list is sorted ascending and padded with -1 to ``k_total``.
    Guide §1, Step 1 (TopK keeps the k best-scoring KV blocks per layer and
    group; output is the index list I1, I2).
    """
    scores = np.asarray(scores, dtype=np.float64)
    n = scores.shape[0]
    order = np.lexsort((np.arange(n), -scores))  # primary -score, secondary index
    chosen = [int(b) for b in order[: min(int(k_scored), n)]]
    if forced is not None:
        chosen.append(int(forced))
    chosen.sort()
    if len(chosen) > k_total:
        raise ValueError("k_total too small for the selection")
    return np.array(chosen + [-1] * (k_total - len(chosen)), dtype=np.int64)


def select_blocks_sink(scores: np.ndarray, k_scored: int, forced: int | None, k_total: int,
                       has_block0: bool) -> np.ndarray:
    """Selection with an attention sink: block 0 is always kept and never
    scored (the guide, §2, names a sink as one likely replacement for the
    dropped sliding window). ``scores`` holds candidate blocks 0..n-1; block 0
    is taken out of the ranking, the best ``min(k_scored, n - 1)`` of blocks
    1..n-1 are kept, then block 0 (when the sequence has it) and the forced
    block, ascending, padded with -1."""
    scores = np.asarray(scores, dtype=np.float64)
    n = scores.shape[0]
    rest = np.arange(1, n)
    order = rest[np.lexsort((rest, -scores[1:]))] if n > 1 else rest
    chosen = [int(b) for b in order[: min(int(k_scored), max(n - 1, 0))]]
    if has_block0:
        chosen.append(0)
    if forced is not None and int(forced) not in chosen:
        chosen.append(int(forced))
    chosen.sort()
    if len(chosen) > k_total:
        raise ValueError("k_total too small for the selection")
    return np.array(chosen + [-1] * (k_total - len(chosen)), dtype=np.int64)


def boundary_gap(scores: np.ndarray, k_scored: int):
    """(s_k, s_{k+1}) of the ranked candidate scores, or None when all are kept."""
    s = np.sort(np.asarray(scores, dtype=np.float64))[::-1]
    if k_scored <= 0 or s.shape[0] <= k_scored:
        return None
    return float(s[k_scored - 1]), float(s[k_scored])


def score_blocks_token_max(q_idx: np.ndarray, kidx_rows: np.ndarray, n_cand: int) -> np.ndarray:
    """Guide-literal block score of candidate blocks 0..n_cand-1 (float64).

    Guide §1, Step 1 as drawn: token-level scores q_idx . K_idx[t] against a
    single index-key head shared by every group of the layer, then a max pool
    over the 64 tokens of each block. ``kidx_rows``: [T, D] index keys of the
    sequence. Candidates are complete blocks, so every one has 64 tokens.
    """
    q = np.asarray(q_idx, dtype=np.float64)
    out = np.empty(int(n_cand))
    for b in range(int(n_cand)):
        rows = np.asarray(kidx_rows[b * BLOCK:(b + 1) * BLOCK], dtype=np.float64)
        out[b] = (rows @ q).max()
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
    return np.concatenate(toks)


def attend(q_heads: np.ndarray, k_rows: np.ndarray, v_rows: np.ndarray, tokens: np.ndarray, scale: float):
    """Softmax attention of each query vector over the token set ``tokens``.

    ``q_heads``: [H, D]. z_t = (q . K[t]) * scale, p = softmax_t(z), o = sum p_t V[t].
    Returns ``(o [H, D], lse [H], p [H, n])`` with lse = log sum_t exp(z_t).
    Guide §1, Step 2 (the gathered subsets of the real K/V go through ordinary
    softmax attention; every head of a group uses its group's selection).
    """
    q = np.asarray(q_heads, dtype=np.float64)
    kk = np.asarray(k_rows[tokens], dtype=np.float64)
    vv = np.asarray(v_rows[tokens], dtype=np.float64)
    z = (q @ kk.T) * float(scale)
    m = z.max(axis=1, keepdims=True)
    e = np.exp(z - m)
    denom = e.sum(axis=1, keepdims=True)
    p = e / denom
    o = p @ vv
    lse = (m + np.log(denom))[:, 0]
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
    q_idx = index_query(q_group)
    scores = score_blocks(q_idx, pooled, n_cand)
    sel = select_blocks(scores, k_scored, forced, k_total)
    use = sel if selected is None else np.asarray(selected)
    toks = tokens_of_blocks(use, seq_len)
    o, lse, p = attend(q_group, k_rows, v_rows, toks, scale)
    return dict(selected=sel, scores=scores, q_idx=q_idx, pooled=pooled, o=o, lse=lse, p=p,
                tokens=toks, forced=forced, n_cand=n_cand)


def prefill_tile_select(q_tile, tile_index, q_start, pooled, k_scored, k_total):
    """Selection for one (64-query tile, KV head) of a chunked prefill.

    ``q_tile``: [R, G, D] (R <= 64 tokens of the tile, G heads of the group).
    The tile's diagonal block is q_start/64 + tile_index; candidates are the
    blocks before it. Guide §3 (during prefill the index branch still scans the
    whole input) and §1, Step 1.
    """
    diag = int(q_start) // BLOCK + int(tile_index)
    q_idx = index_query(q_tile)
    scores = score_blocks(q_idx, pooled, diag)
    sel = select_blocks(scores, k_scored, diag, k_total)
    return dict(selected=sel, scores=scores, q_idx=q_idx, diag=diag)


def prefill_tile_select_token_max(q_tile, tile_index, q_start, kidx_rows, k_scored, k_total):
    """Selection for one (64-query tile, KV head) of a chunked prefill with the
    guide-literal block score: the tile's index query (sum over its tokens and
    the group's heads) against every token of the shared index-key head, max
    over each block's 64 tokens; candidates are the blocks before the tile's
    diagonal block q_start/64 + tile_index, which is always kept. Guide §1,
    Step 1 as drawn, and §3 (in prefill the index branch scans the whole
    input).
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
    q_rows = np.asarray(q_rows, dtype=np.float64)
    r, g, d = q_rows.shape
    o = np.zeros((r, g, d))
    lse = np.zeros((r, g))
    for i in range(r):
        toks = tokens_of_blocks(blocks, seq_len, last_pos=int(positions[i]))
        oi, li, _ = attend(q_rows[i], k_rows, v_rows, toks, scale)
        o[i], lse[i] = oi, li
    return o, lse


# ---------------------------------------------------------------------------
# Dense causal GQA attention (the full-attention comparator)
# ---------------------------------------------------------------------------

def dense_gqa(q_heads: np.ndarray, k_rows: np.ndarray, v_rows: np.ndarray, position: int, scale: float):
    """Full causal attention of the query heads at ``position`` over tokens
    0..position of their shared KV head: softmax(q K^T * scale) V.

    Written on its own (no shared code with :func:`attend`) so the sparse path
    with every block selected can be checked against it. This is the
    full-attention baseline the guide's speed-ups are quoted against (§3).
    """
    q = np.asarray(q_heads, dtype=np.float64)
    n = int(position) + 1
    keys = np.asarray(k_rows[:n], dtype=np.float64)
    vals = np.asarray(v_rows[:n], dtype=np.float64)
    out = np.zeros((q.shape[0], vals.shape[1]))
    lse = np.zeros(q.shape[0])
    for h in range(q.shape[0]):
        logits = keys @ q[h] * float(scale)
        top = logits.max()
        w = np.exp(logits - top)
        total = w.sum()
        out[h] = (w[:, None] * vals).sum(axis=0) / total
        lse[h] = top + np.log(total)
    return out, lse

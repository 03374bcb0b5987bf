"""Seeded synthetic inputs shared by the tests, the benchmark and the smoke run.

This module only draws numbers: it holds none of the attention arithmetic. Both
the CUDA library and the CPU oracle receive the tensors it returns, so the two
always see the same bits.

Every tensor comes from its own seeded stream (seed, stream id), so changing
one part of a workload leaves the others unchanged. Values follow the workloads
of the benchmark: Q, K and V ~ N(0, 1) rounded to the KV dtype; "needle" blocks
whose 64 keys are 3 * q_mean + N(0, 0.1^2), where q_mean is the fp32 mean of
the query heads of that (sequence, KV head); ragged lengths log-uniform in a
range; a shuffled page table for the paged layout.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np
import torch

BLOCK = 64
HEAD_DIM = 128

# stream ids
(_S_Q, _S_K, _S_V, _S_NEEDLE_POS, _S_NEEDLE_NOISE, _S_LENS, _S_PAGES, _S_KIDX, _S_KIDX_POS, _S_KIDX_NOISE,
 _S_CHUNK_Q) = range(11)


def _gen(seed: int, stream: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed) * 1009 + int(stream))
    return g


def _randn_into(t: torch.Tensor, g: torch.Generator, chunk: int = 1 << 27) -> None:
    """Fill ``t`` with N(0,1) drawn in fp32 and rounded to ``t.dtype``."""
    flat = t.view(-1)
    for lo in range(0, flat.numel(), chunk):
        hi = min(flat.numel(), lo + chunk)
        flat[lo:hi].copy_(torch.randn(hi - lo, generator=g, device=t.device, dtype=torch.float32))


def torch_dtype(name: str) -> torch.dtype:
    return {"bf16": torch.bfloat16, "f32": torch.float32}[name]


@dataclasses.dataclass
class DecodeInputs:
    q: torch.Tensor                 # [B, Hq, D]
    k: torch.Tensor                 # contiguous [B, Hkv, T, D] or paged [P, Hkv, 64, D]
    v: torch.Tensor
    seq_lens: torch.Tensor          # int32 [B]
    page_table: torch.Tensor | None  # int32 [B, max_pages] (paged only; -1 = unused)
    layout: str                     # "contiguous" | "paged"
    dtype: str                      # "bf16" | "f32"
    num_kv_heads: int
    num_q_heads: int
    needles: dict                   # (s, h) -> sorted list of needle block ids
    lens: list                      # python ints

    @property
    def batch(self) -> int:
        return self.q.shape[0]

    @property
    def max_tokens(self) -> int:
        return self.k.shape[2] if self.layout == "contiguous" else 0

    def kv_rows(self, s: int, h: int, which: str = "k") -> torch.Tensor:
        """[n_tokens_capacity, D] rows of one (sequence, KV head), in logical
        token order (gathered through the page table for the paged layout)."""
        t = self.k if which == "k" else self.v
        if self.layout == "contiguous":
            return t[s, h]
        n_pages = -(-self.lens[s] // BLOCK)
        pages = self.page_table[s, :n_pages].long()
        return t[pages, h].reshape(n_pages * BLOCK, t.shape[-1])


def ragged_lengths(batch: int, lo: int, hi: int, seed: int) -> list:
    """Lengths log-uniform in [lo, hi] (inclusive), drawn from the seed."""
    rng = np.random.default_rng([int(seed), _S_LENS])
    u = rng.uniform(math.log(lo), math.log(hi), size=batch)
    return [int(min(hi, max(lo, round(math.exp(x))))) for x in u]


def make_decode_inputs(lens, num_kv_heads: int, num_q_heads: int, dtype: str = "bf16",
                       layout: str = "contiguous", needles: int = 0, seed: int = 0,
                       device="cpu", max_tokens: int | None = None) -> DecodeInputs:
    """One decode query token per sequence over a KV cache of ``lens`` tokens."""
    lens = [int(x) for x in lens]
    b = len(lens)
    d = HEAD_DIM
    tdt = torch_dtype(dtype)
    q = torch.empty(b, num_q_heads, d, dtype=tdt, device=device)
    _randn_into(q, _gen(seed, _S_Q, device))
    page_table = None
    if layout == "contiguous":
        cap = max_tokens if max_tokens is not None else -(-max(lens) // BLOCK) * BLOCK
        assert cap % BLOCK == 0 and cap >= max(lens)
        shape = (b, num_kv_heads, cap, d)
    elif layout == "paged":
        pages_per = [-(-n // BLOCK) for n in lens]
        num_pages = sum(pages_per)
        perm = np.random.default_rng([int(seed), _S_PAGES]).permutation(num_pages).astype(np.int32)
        max_pages = max(pages_per)
        table = np.full((b, max_pages), -1, dtype=np.int32)
        off = 0
        for s, n in enumerate(pages_per):
            table[s, :n] = perm[off:off + n]
            off += n
        page_table = torch.from_numpy(table).to(device)
        shape = (num_pages, num_kv_heads, BLOCK, d)
    else:
        raise ValueError(layout)
    k = torch.empty(shape, dtype=tdt, device=device)
    v = torch.empty(shape, dtype=tdt, device=device)
    _randn_into(k, _gen(seed, _S_K, device))
    _randn_into(v, _gen(seed, _S_V, device))
    inp = DecodeInputs(q=q, k=k, v=v, seq_lens=torch.tensor(lens, dtype=torch.int32, device=device),
                       page_table=page_table, layout=layout, dtype=dtype, num_kv_heads=num_kv_heads,
                       num_q_heads=num_q_heads, needles={}, lens=lens)
    if needles:
        _plant_needles(inp, needles, seed)
    return inp


def _plant_needles(inp: DecodeInputs, per_head: int, seed: int) -> None:
    """Overwrite ``per_head`` distinct candidate blocks of every (sequence, KV
    head) with keys 3 * q_mean + N(0, 0.1^2). Candidates are the complete
    blocks other than the block holding the newest token."""
    rng = np.random.default_rng([int(seed), _S_NEEDLE_POS])
    g = _gen(seed, _S_NEEDLE_NOISE, inp.q.device)
    hkv = inp.num_kv_heads
    grp = inp.num_q_heads // hkv
    d = inp.q.shape[-1]
    for s, n in enumerate(inp.lens):
        nb = -(-n // BLOCK)
        n_cand = min(n // BLOCK, nb - 1)
        cnt = min(per_head, n_cand)
        if cnt <= 0:
            continue
        qm = inp.q[s].float().view(hkv, grp, d).mean(dim=1)          # [Hkv, D]
        for h in range(hkv):
            blocks = sorted(int(x) for x in rng.choice(n_cand, size=cnt, replace=False))
            inp.needles[(s, h)] = blocks
            noise = torch.randn(cnt, BLOCK, d, generator=g, device=inp.q.device, dtype=torch.float32)
            rows = (3.0 * qm[h] + 0.1 * noise).to(inp.k.dtype)         # [cnt, 64, D]
            if inp.layout == "contiguous":
                idx = torch.tensor(blocks, device=inp.q.device)
                kv = inp.k[s, h].view(-1, BLOCK, d)
                kv[idx] = rows
            else:
                pages = inp.page_table[s, blocks].long()
                inp.k[pages, h] = rows


@dataclasses.dataclass
class IndexKeys:
    kidx: torch.Tensor   # contiguous [B, T, D] or paged [P, 64, D]: one index-key head per sequence
    needles: dict        # (s, h) -> sorted list of needle block ids (one needle token each)
    layout: str

    def rows(self, inp: DecodeInputs, s: int) -> torch.Tensor:
        """[capacity, D] index keys of sequence s in logical token order."""
        if self.layout == "contiguous":
            return self.kidx[s]
        n_pages = -(-inp.lens[s] // BLOCK)
        pages = inp.page_table[s, :n_pages].long()
        return self.kidx[pages].reshape(n_pages * BLOCK, self.kidx.shape[-1])


def make_index_keys(inp: DecodeInputs, needles: int = 0, seed: int = 0) -> IndexKeys:
    """A single index-key head per sequence, laid out like one KV head of the
    cache (contiguous [B, T, D] or paged [P, 64, D] on the same pages), with
    values ~ N(0, 1) in the KV dtype. For every (sequence, KV head), ``needles``
    distinct candidate blocks (distinct across the heads of the sequence) get
    one token whose index key is 3 * q_mean + N(0, 0.1^2), q_mean the fp32 mean
    of that group's query heads."""
    dev = inp.q.device
    d = inp.q.shape[-1]
    if inp.layout == "contiguous":
        shape = (inp.batch, inp.k.shape[2], d)
    else:
        shape = (inp.k.shape[0], BLOCK, d)
    kidx = torch.empty(shape, dtype=inp.k.dtype, device=dev)
    _randn_into(kidx, _gen(seed, _S_KIDX, dev))
    out = IndexKeys(kidx=kidx, needles={}, layout=inp.layout)
    if not needles:
        return out
    rng = np.random.default_rng([int(seed), _S_KIDX_POS])
    g = _gen(seed, _S_KIDX_NOISE, dev)
    hkv = inp.num_kv_heads
    grp = inp.num_q_heads // hkv
    for s, n in enumerate(inp.lens):
        nb = -(-n // BLOCK)
        n_cand = min(n // BLOCK, nb - 1)
        cnt = min(needles, n_cand // hkv)
        if cnt <= 0:
            continue
        chosen = rng.choice(n_cand, size=cnt * hkv, replace=False)
        offs = rng.integers(0, BLOCK, size=cnt * hkv)
        qm = inp.q[s].float().view(hkv, grp, d).mean(dim=1)
        for h in range(hkv):
            blocks = [int(x) for x in chosen[h * cnt:(h + 1) * cnt]]
            out.needles[(s, h)] = sorted(blocks)
            for j, b in enumerate(blocks):
                t = b * BLOCK + int(offs[h * cnt + j])
                row = (3.0 * qm[h] + 0.1 * torch.randn(d, generator=g, device=dev, dtype=torch.float32)).to(kidx.dtype)
                if inp.layout == "contiguous":
                    kidx[s, t] = row
                else:
                    kidx[int(inp.page_table[s, t // BLOCK]), t % BLOCK] = row
    return out


@dataclasses.dataclass
class PrefillInputs:
    q: torch.Tensor        # [N, Hq, D] new query tokens
    k: torch.Tensor        # contiguous [1, Hkv, T, D] or paged [P, Hkv, 64, D]: prefix + new tokens
    v: torch.Tensor
    seq_lens: torch.Tensor  # int32 [1] = q_start + N
    q_start: int
    n_new: int
    num_kv_heads: int
    num_q_heads: int
    dtype: str
    layout: str = "contiguous"
    page_table: torch.Tensor | None = None  # int32 [1, pages] (paged)

    def kv_rows(self, h: int, which: str = "k") -> torch.Tensor:
        """[capacity, D] rows of KV head h in logical token order."""
        t = self.k if which == "k" else self.v
        if self.layout == "contiguous":
            return t[0, h]
        pages = self.page_table[0].long()
        return t[pages, h].reshape(pages.numel() * BLOCK, t.shape[-1])


def make_prefill_inputs(prefix: int, n_new: int, num_kv_heads: int, num_q_heads: int,
                        dtype: str = "bf16", seed: int = 0, device="cpu",
                        max_tokens: int | None = None, layout: str = "contiguous") -> PrefillInputs:
    """A chunk of ``n_new`` query tokens appended to a ``prefix``-token cache
    (contiguous, or paged with a shuffled page table)."""
    total = prefix + n_new
    cap = max_tokens if max_tokens is not None else -(-total // BLOCK) * BLOCK
    tdt = torch_dtype(dtype)
    q = torch.empty(n_new, num_q_heads, HEAD_DIM, dtype=tdt, device=device)
    page_table = None
    if layout == "contiguous":
        k = torch.empty(1, num_kv_heads, cap, HEAD_DIM, dtype=tdt, device=device)
    elif layout == "paged":
        pages = cap // BLOCK
        perm = np.random.default_rng([int(seed), _S_PAGES]).permutation(pages).astype(np.int32)
        page_table = torch.from_numpy(perm.reshape(1, pages)).to(device)
        k = torch.empty(pages, num_kv_heads, BLOCK, HEAD_DIM, dtype=tdt, device=device)
    else:
        raise ValueError(layout)
    v = torch.empty_like(k)
    _randn_into(q, _gen(seed, _S_Q, device))
    _randn_into(k, _gen(seed, _S_K, device))
    _randn_into(v, _gen(seed, _S_V, device))
    return PrefillInputs(q=q, k=k, v=v, seq_lens=torch.tensor([total], dtype=torch.int32, device=device),
                         q_start=prefix, n_new=n_new, num_kv_heads=num_kv_heads,
                         num_q_heads=num_q_heads, dtype=dtype, layout=layout, page_table=page_table)


@dataclasses.dataclass
class PrefillBatchInputs:
    """A batch of prefill chunks: sequence s appends q_counts[s] tokens to a
    q_starts[s]-token prefix. ``cache`` holds every sequence's prefix and new
    tokens (lengths q_starts[s] + q_counts[s], either layout); ``q`` holds the
    chunks' query tokens back to back."""
    cache: DecodeInputs
    q: torch.Tensor      # [sum q_counts, Hq, D]
    q_starts: list
    q_counts: list

    @property
    def q_off(self) -> list:
        return [sum(self.q_counts[:s]) for s in range(len(self.q_counts))]

    @property
    def tile_off(self) -> list:
        """Global index of each sequence's first query tile (tiles group a
        chunk's tokens by the 64-token block they sit in)."""
        def tiles(a, c):
            return 0 if c <= 0 else (a + c - 1) // BLOCK - a // BLOCK + 1
        return [sum(tiles(a, c) for a, c in zip(self.q_starts[:s], self.q_counts[:s]))
                for s in range(len(self.q_counts) + 1)]

    def q_rows(self, s: int) -> torch.Tensor:
        o = self.q_off[s]
        return self.q[o:o + self.q_counts[s]]


def make_prefill_batch_inputs(q_starts, q_counts, num_kv_heads: int, num_q_heads: int, dtype: str = "bf16",
                              layout: str = "contiguous", seed: int = 0, device="cpu") -> PrefillBatchInputs:
    """Chunks of ``q_counts[s]`` new tokens after ``q_starts[s]``-token prefixes,
    one per sequence of a shared cache."""
    q_starts = [int(x) for x in q_starts]
    q_counts = [int(x) for x in q_counts]
    lens = [a + c for a, c in zip(q_starts, q_counts)]
    cache = make_decode_inputs([max(n, 1) for n in lens], num_kv_heads, num_q_heads, dtype, layout, seed=seed,
                               device=device)
    cache.seq_lens.copy_(torch.tensor(lens, dtype=torch.int32))
    cache.lens = lens
    q = torch.empty(sum(q_counts), num_q_heads, HEAD_DIM, dtype=torch_dtype(dtype), device=device)
    _randn_into(q, _gen(seed, _S_CHUNK_Q, device))
    return PrefillBatchInputs(cache=cache, q=q, q_starts=q_starts, q_counts=q_counts)


# ---------------------------------------------------------------------------
# The five benchmark workloads
# ---------------------------------------------------------------------------

WORKLOADS = {
    "tiny_decode": dict(kind="decode", lens=[4096], hkv=1, hq=4, dtype="f32", layout="contiguous",
                        k_scored=8, k_total=9, needles=2, seed=1001),
    "decode_128k": dict(kind="decode", lens=[131072] * 8, hkv=8, hq=64, dtype="bf16",
                        layout="contiguous", k_scored=31, k_total=32, needles=16, seed=1002),
    "decode_1m": dict(kind="decode", lens=[1048576], hkv=8, hq=64, dtype="bf16", layout="contiguous",
                      k_scored=63, k_total=64, needles=32, seed=1003),
    "prefill_8k_on_128k": dict(kind="prefill", prefix=131072, n_new=8192, hkv=8, hq=64, dtype="bf16",
                               k_scored=32, k_total=33, seed=1004),
    "ragged_paged_decode": dict(kind="decode", ragged=(32, 16384, 1048576), hkv=8, hq=64, dtype="bf16",
                                layout="paged", k_scored=47, k_total=48, needles=8, seed=1005),
}


def workload_lens(name: str) -> list:
    w = WORKLOADS[name]
    if "ragged" in w:
        b, lo, hi = w["ragged"]
        return ragged_lengths(b, lo, hi, w["seed"])
    return list(w["lens"])


def make_workload(name: str, device="cpu"):
    w = WORKLOADS[name]
    if w["kind"] == "prefill":
        return make_prefill_inputs(w["prefix"], w["n_new"], w["hkv"], w["hq"], w["dtype"], w["seed"], device)
    return make_decode_inputs(workload_lens(name), w["hkv"], w["hq"], w["dtype"], w["layout"],
                              w["needles"], w["seed"], device)

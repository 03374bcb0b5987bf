"""Benchmark of the two-stage block-sparse GQA attention hot path on GB300.

Default workload: decode over a bf16 KV cache of 8 sequences x 131072 tokens,
8 KV heads / 64 query heads, head dim 128, 64-token blocks, top-31 blocks plus
the newest block. One step = Step 1 (group index query, block scores, top-k)
plus Step 2 (sparse flash-decode with split-K combine) for one query token per
sequence. The summary keys are pooled once beforehand (they change only when a
block fills) and that pass is reported separately.

Timing: W untimed warm-up steps, then K timed steps. The L2 (129 MB) is
flushed before every timed step, outside the timed window: a 512 MB buffer is
written, then a separate 256 MB buffer is read, so the step starts with none of
its inputs cached and with clean lines in L2 (a cache left full of dirty lines
would bill the step for writing back the flush buffer). Each step is bracketed
by CUDA events on the launching stream. Clocks are sampled with nvidia-smi
during the timed region.

Prints ONE JSON line on rank 0. Under torchrun (N > 1) every rank runs an
independent replica on its own GPU (the path shards by sequence and head with
no exchange), the timed region is bracketed by barriers and the slowest rank's
time is reported.

--impl reference times the CPU oracle on the host cores instead (a bounded
sample of the same workload per step, extrapolated to a full step).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "sparse-attn decode µs/step + HBM GB/s at 128K/1M ctx; prefill TFLOP/s"
UNIT = "µs/step"
SCALE = 1.0 / math.sqrt(128)
L2_FLUSH_BYTES = 512 << 20
L2_CLEAN_BYTES = 256 << 20
KV_BLOCK_BYTES = 64 * 128 * 2  # one 64-token K (or V) block in bf16


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-extras", action="store_true", help="time only the headline workload")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU-oracle baseline")
    ap.add_argument("--only", choices=["prefill", "token_max"], default=None,
                    help="time only the chunked-prefill or the token-max decode workload and print its figures "
                         "(profiling)")
    ap.add_argument("--batch", type=int, default=8,
                    help="sequences of the 131072-token decode workload (8 = the benchmark; fewer for profiling)")
    return ap.parse_args()


# --------------------------------------------------------------------------- distributed plumbing

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


class Dist:
    def __init__(self, backend):
        import torch.distributed as dist
        self.world, self.rank, self.local = dist_env()
        self.dist = dist if self.world > 1 else None
        if self.dist is not None:
            os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
            dist.init_process_group(backend)

    def barrier(self):
        if self.dist is not None:
            self.dist.barrier()

    def max(self, x: float) -> float:
        if self.dist is None:
            return x
        import torch
        t = torch.tensor([x], dtype=torch.float64, device="cuda" if self.dist.get_backend() == "nccl" else "cpu")
        self.dist.all_reduce(t, op=self.dist.ReduceOp.MAX)
        return float(t.item())

    def close(self):
        if self.dist is not None:
            self.dist.destroy_process_group()


# --------------------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi samples (200 ms) of the SM clock and throttle reasons."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for nm, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# --------------------------------------------------------------------------- helpers

def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), float(p.get("bf16_tflops_sustained", p["bf16_tflops"])), \
            "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, 1900.0, 1700.0, "fallback"


def kernel_source_hash(name: str) -> str:
    with open(os.path.join(ROOT, "sparse_attention_step_gb300", "csrc", name), "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def recorded_traffic(kernel: str, src: str):
    """DRAM bytes per launch recorded from an ncu capture of this kernel
    (profiles/traffic.json), only while the kernel source is unchanged."""
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            rec = json.load(f)[kernel]
    except (OSError, KeyError, ValueError):
        return None
    if rec.get("source_sha256_16") != kernel_source_hash(src):
        return None
    return rec.get("dram_bytes_per_launch")


class Timer:
    """Per-step CUDA-event timing with an L2 flush before each timed step."""

    def __init__(self, torch):
        self.torch = torch
        self.flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device="cuda")
        self.clean = torch.ones(L2_CLEAN_BYTES // 4, dtype=torch.float32, device="cuda")

    def l2_flush(self):
        self.flush.zero_()
        self.clean.sum()


# --------------------------------------------------------------------------- our arm

def decode_setup(torch, msa, inp, k_scored, k_total):
    desc = msa.kv_desc(inp.k, inp.v, inp.seq_lens, inp.page_table)
    hq = inp.num_q_heads
    need = max(msa.msa_workspace_size(op, desc, hq, 1, k_total)
               for op in (msa.MSA_OP_POOL, msa.MSA_OP_SELECT, msa.MSA_OP_DECODE, msa.MSA_OP_DENSE_DECODE,
                          msa.MSA_OP_DECODE_STEP))
    ws = msa.Workspace(need)
    pooled = torch.empty(msa.pooled_shape(desc), dtype=inp.k.dtype, device="cuda")
    idx = torch.empty(inp.batch, inp.num_kv_heads, k_total, dtype=torch.int32, device="cuda")
    out = torch.empty_like(inp.q)
    lse = torch.empty(inp.batch, hq, dtype=torch.float32, device="cuda")
    cfg = msa.select_cfg(k_scored)
    return dict(desc=desc, ws=ws, pooled=pooled, idx=idx, out=out, lse=lse, cfg=cfg, hq=hq, k_total=k_total)


def decode_select(msa, st, q):
    msa.msa_select_topk_blocks(q, st["hq"], 1, st["pooled"], st["desc"], st["cfg"], st["idx"], st["k_total"], None,
                               st["ws"].buf, st["ws"].nbytes)


def decode_attend(msa, st, q, out=None):
    msa.msa_sparse_attn_decode(q, st["hq"], st["desc"], st["idx"], st["k_total"], SCALE,
                               st["out"] if out is None else out, st["lse"], st["ws"].buf, st["ws"].nbytes)


def decode_bytes(inp, k_total):
    """Algorithmic HBM bytes of one decode step: pooled keys of the candidate
    blocks, the selected K/V blocks (partial last block counted in full), q and
    the output."""
    units_h = inp.num_kv_heads
    d = 128
    pooled = sum(min(n // 64, (n + 63) // 64 - 1) for n in inp.lens) * units_h * d * 2
    sel = sum(min(k_total, (n + 63) // 64) for n in inp.lens) * units_h * 2 * KV_BLOCK_BYTES
    qo = 2 * inp.q.numel() * inp.q.element_size()
    return pooled, sel, qo


def capture(torch, fn):
    """CUDA graph of the library calls in ``fn`` (their first call, which does
    the per-device set-up, has already run outside the capture)."""
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        with torch.cuda.graph(g, stream=side):
            fn()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    return g


def time_graph(torch, timer, g, steps, warmup, dist=None, samples=None):
    """Mean device time of one replay, L2 flushed before each timed replay
    (each replay's time is appended to ``samples`` when given)."""
    for _ in range(warmup):
        g.replay()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    for e0, e1 in ev:
        timer.l2_flush()
        e0.record(stream)
        g.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    times = [a.elapsed_time(b) for a, b in ev]
    if samples is not None:
        samples.extend(times)
    return statistics.mean(times)


def quantiles_us(ms_samples):
    """p10 / median / p90 of per-step times (ms in, microseconds out), this rank."""
    xs = sorted(ms_samples)
    if not xs:
        return None
    pick = lambda f: round(xs[min(len(xs) - 1, int(f * len(xs)))] * 1e3, 3)
    return {"p10": pick(0.1), "p50": round(statistics.median(xs) * 1e3, 3), "p90": pick(0.9)}


def decode_step(msa, st, q, out=None):
    """The whole decode step through msa_sparse_decode_step (one kernel for
    contiguous bf16 caches)."""
    msa.msa_sparse_decode_step(q, st["hq"], st["pooled"], st["desc"], st["cfg"], st["idx"], st["k_total"], SCALE,
                               st["out"] if out is None else out, st["lse"], st["ws"].buf, st["ws"].nbytes)


def time_decode(torch, msa, timer, st, inp, steps, warmup, dist, samples=None):
    """Times the step (msa_sparse_decode_step) as one CUDA graph replay, and
    the two-kernel form (select, then attend; each its own graph) for the
    per-kernel figures."""
    q = inp.q
    for _ in range(max(1, warmup)):
        decode_select(msa, st, q)
        decode_attend(msa, st, q)
        decode_step(msa, st, q)
    torch.cuda.synchronize()
    g_step = capture(torch, lambda: decode_step(msa, st, q))
    g_sel = capture(torch, lambda: decode_select(msa, st, q))
    g_att = capture(torch, lambda: decode_attend(msa, st, q))
    step = time_graph(torch, timer, g_step, steps, warmup, dist, samples)
    sel = time_graph(torch, timer, g_sel, steps, warmup)
    att = time_graph(torch, timer, g_att, steps, warmup)
    return step, sel, att


def time_e2e_decode(torch, msa, timer, st, inp, steps, warmup):
    """Same step through the C ABI with the per-step inputs (the new query
    token of every sequence) in pinned host memory and the output read back."""
    q_host = inp.q.cpu().pin_memory()
    out_host = torch.empty(inp.q.shape, dtype=inp.q.dtype).pin_memory()
    q_dev = torch.empty_like(inp.q)
    stream = torch.cuda.current_stream()
    times = []
    for i in range(warmup + steps):
        timer.l2_flush()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        q_dev.copy_(q_host, non_blocking=True)
        decode_step(msa, st, q_dev)
        out_host.copy_(st["out"], non_blocking=True)
        e1.record(stream)
        e1.synchronize()
        if i >= warmup:
            times.append(e0.elapsed_time(e1))
    nbytes = q_host.numel() * q_host.element_size()
    return statistics.mean(times), nbytes, nbytes


def time_op(torch, timer, fn, steps, warmup):
    """Device time of ``fn`` (library calls only) replayed as a CUDA graph."""
    fn()
    torch.cuda.synchronize()
    return time_graph(torch, timer, capture(torch, fn), steps, warmup)


def extras_decode(torch, msa, timer, name, steps, warmup, hbm):
    from synth import make_workload, WORKLOADS
    w = WORKLOADS[name]
    inp = make_workload(name, device="cuda")
    st = decode_setup(torch, msa, inp, w["k_scored"], w["k_total"])
    msa.msa_pool_block_keys(st["desc"], 0, -1, st["pooled"], st["ws"].buf, st["ws"].nbytes)
    dist = Dist.__new__(Dist)
    dist.dist = None
    step_ms, sel_ms, att_ms = time_decode(torch, msa, timer, st, inp, steps, warmup, dist)
    pooled_b, sel_b, qo_b = decode_bytes(inp, w["k_total"])
    dense_out = torch.empty_like(inp.q)
    dense_ms = time_op(torch, timer, lambda: msa.msa_dense_gqa_decode(
        inp.q, st["hq"], st["desc"], SCALE, dense_out, st["lse"], st["ws"].buf, st["ws"].nbytes),
        max(3, steps // 5), 2)
    dense_bytes = sum(inp.lens) * inp.num_kv_heads * 2 * 128 * 2 + qo_b
    status = msa.msa_read_device_status(st["ws"].buf)
    res = {
        "workload": name, "us_per_step": step_ms * 1e3,
        "two_kernel_select_us": sel_ms * 1e3, "two_kernel_attend_us": att_ms * 1e3,
        "step_GBps": (pooled_b + sel_b + qo_b) / (step_ms * 1e-3) / 1e9,
        "step_roofline_frac": (pooled_b + sel_b + qo_b) / (step_ms * 1e-3) / 1e9 / hbm,
        "bytes_per_step": pooled_b + sel_b + qo_b,
        "dense_us": dense_ms * 1e3, "dense_GBps": dense_bytes / (dense_ms * 1e-3) / 1e9,
        "dense_over_sparse": dense_ms / step_ms, "device_status": status,
    }
    if name == "decode_1m":
        # context point (not the headline): k near the ratio the guide implies
        # (~6.4% of 16384 blocks); k > 64 runs the selection and attention
        # kernels in turn
        k_big = 1050
        st2 = decode_setup(torch, msa, inp, k_big, k_big + 1)
        st2["pooled"] = st["pooled"]
        big_ms = time_op(torch, timer, lambda: decode_step(msa, st2, inp.q), max(5, steps // 2), 2)
        pb2, sb2, qb2 = decode_bytes(inp, k_big + 1)
        res["k1050"] = {"k_scored": k_big, "us_per_step": big_ms * 1e3,
                        "step_GBps": (pb2 + sb2 + qb2) / (big_ms * 1e-3) / 1e9,
                        "step_roofline_frac": (pb2 + sb2 + qb2) / (big_ms * 1e-3) / 1e9 / hbm,
                        "bytes_per_step": pb2 + sb2 + qb2, "dense_over_sparse": dense_ms / big_ms,
                        "device_status": msa.msa_read_device_status(st2["ws"].buf)}
        del st2
    del inp, st
    torch.cuda.empty_cache()
    return res


def extras_token_max(torch, msa, timer, steps, warmup, hbm):
    """The decode step with the guide-literal Step 1 (token-level scores
    against a shared index-key head, block max pool) on the 128K x 8 shape:
    select (token-max scores + top-k) then sparse attention, one CUDA graph."""
    from synth import make_decode_inputs, make_index_keys
    inp = make_decode_inputs([131072] * 8, 8, 64, "bf16", "contiguous", seed=1006, device="cuda")
    ik = make_index_keys(inp, needles=8, seed=1007)
    k_scored, k_total = 31, 32
    st = decode_setup(torch, msa, inp, k_scored, k_total)
    cfg = msa.select_cfg(k_scored, mode=msa.MSA_SCORE_TOKEN_MAX)

    def step():
        msa.msa_sparse_decode_step(inp.q, st["hq"], ik.kidx, st["desc"], cfg, st["idx"], k_total, SCALE,
                                   st["out"], st["lse"], st["ws"].buf, st["ws"].nbytes)

    step_ms = time_op(torch, timer, step, steps, warmup)
    sel_ms = time_op(torch, timer, lambda: msa.msa_select_topk_blocks(
        inp.q, st["hq"], 1, ik.kidx, st["desc"], cfg, st["idx"], k_total, None, st["ws"].buf, st["ws"].nbytes),
        steps, warmup)
    # index keys of every candidate token (read once for all KV heads) + selected K/V + q/out
    kidx_b = sum(min(n // 64, (n + 63) // 64 - 1) * 64 for n in inp.lens) * 128 * 2
    _, sel_b, qo_b = decode_bytes(inp, k_total)
    total = kidx_b + sel_b + qo_b
    status = msa.msa_read_device_status(st["ws"].buf)
    res = {
        "workload": "decode_128k_token_max: 8 x 131072 tokens, 8 KV / 64 query heads, shared bf16 index-key "
                    "head, top-31 + newest, 8 needle tokens per (seq, head)",
        "us_per_step": step_ms * 1e3, "select_us": sel_ms * 1e3,
        "step_GBps": total / (step_ms * 1e-3) / 1e9, "step_roofline_frac": total / (step_ms * 1e-3) / 1e9 / hbm,
        "select_GBps": kidx_b / (sel_ms * 1e-3) / 1e9, "bytes_per_step": total, "device_status": status,
    }
    del inp, ik, st
    torch.cuda.empty_cache()
    return res


def extras_prefill(torch, msa, timer, steps, warmup, tflops_peak):
    from synth import make_workload, WORKLOADS
    w = WORKLOADS["prefill_8k_on_128k"]
    inp = make_workload("prefill_8k_on_128k", device="cuda")
    desc = msa.kv_desc(inp.k, inp.v, inp.seq_lens)
    hq, n = inp.num_q_heads, inp.n_new
    kt = w["k_total"]
    need = max(msa.msa_workspace_size(op, desc, hq, n, kt) for op in (msa.MSA_OP_SELECT_PREFILL, msa.MSA_OP_PREFILL))
    ws = msa.Workspace(need)
    pooled = torch.empty(msa.pooled_shape(desc), dtype=inp.k.dtype, device="cuda")
    n_tiles = (n + 63) // 64
    idx = torch.empty(n_tiles, inp.num_kv_heads, kt, dtype=torch.int32, device="cuda")
    out = torch.empty_like(inp.q)
    cfg = msa.select_cfg(w["k_scored"], True, 64, inp.q_start)
    pool_ms = time_op(torch, timer, lambda: msa.msa_pool_block_keys(desc, 0, -1, pooled, ws.buf, ws.nbytes), 5, 2)
    sel_ms = time_op(torch, timer, lambda: msa.msa_select_topk_blocks(
        inp.q, hq, n, pooled, desc, cfg, idx, kt, None, ws.buf, ws.nbytes), steps, warmup)
    att_ms = time_op(torch, timer, lambda: msa.msa_sparse_attn_prefill(
        inp.q, hq, n, inp.q_start, desc, idx, kt, SCALE, out, None, ws.buf, ws.nbytes), steps, warmup)
    dense_ms = time_op(torch, timer, lambda: msa.msa_dense_gqa_prefill(
        inp.q, hq, n, inp.q_start, desc, SCALE, out, None, ws.buf, ws.nbytes), 3, 1)
    # the guide-literal Step 1 on the same chunk: token scores against one shared
    # bf16 index-key head (N(0,1), seeded), block max pool, top-k
    g_idx = torch.Generator(device="cuda")
    g_idx.manual_seed(4007)
    kidx = torch.randn(1, desc.max_tokens, 128, generator=g_idx, device="cuda").to(torch.bfloat16)
    cfg_tm = msa.select_cfg(w["k_scored"], True, 64, inp.q_start, mode=msa.MSA_SCORE_TOKEN_MAX)
    sel_tm_ms = time_op(torch, timer, lambda: msa.msa_select_topk_blocks(
        inp.q, hq, n, kidx, desc, cfg_tm, idx, kt, None, ws.buf, ws.nbytes), steps, warmup)
    grp = hq // inp.num_kv_heads
    # algorithmic FLOPs: 4 * D per visible (query row, key) pair
    sel_pairs = 0
    diag_pairs = sum(t + 1 for t in range(64))
    for j in range(n_tiles):
        diag = inp.q_start // 64 + j
        sel_pairs += 64 * min(w["k_scored"], diag) * 64 + diag_pairs
    sparse_flop = 4 * 128 * grp * inp.num_kv_heads * sel_pairs
    total = inp.q_start + n
    dense_pairs = sum(inp.q_start + r + 1 for r in range(n))
    dense_flop = 4 * 128 * hq * dense_pairs
    status = msa.msa_read_device_status(ws.buf)
    res = {
        "workload": "prefill_8k_on_128k", "select_us": sel_ms * 1e3, "attend_us": att_ms * 1e3,
        "attend_TFLOPs": sparse_flop / (att_ms * 1e-3) / 1e12,
        "attend_tensor_frac": sparse_flop / (att_ms * 1e-3) / 1e12 / tflops_peak,
        "step_us": (sel_ms + att_ms) * 1e3, "sparse_gflop": sparse_flop / 1e9,
        "dense_us": dense_ms * 1e3, "dense_TFLOPs": dense_flop / (dense_ms * 1e-3) / 1e12,
        "dense_over_sparse_step": dense_ms / (sel_ms + att_ms),
        "pool_us": pool_ms * 1e3, "pool_GBps": total * inp.num_kv_heads * 256 / (pool_ms * 1e-3) / 1e9,
        "select_token_max_us": sel_tm_ms * 1e3,
        "device_status": status,
    }
    del inp, pooled, out, kidx
    torch.cuda.empty_cache()
    return res


def run_ours(args):
    import torch
    from sparse_attention_step_gb300 import build, msa
    from synth import make_workload, WORKLOADS

    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    dist = Dist("nccl")
    if rank == 0 or world == 1:
        build.build()
    dist.barrier()
    msa.load()
    hbm, tf_burst, tf_sus, peak_src = peaks()
    timer = Timer(torch)

    name = "decode_128k"
    w = WORKLOADS[name]
    if args.batch == len(w["lens"]):
        inp = make_workload(name, device="cuda")
    else:
        from synth import make_decode_inputs
        inp = make_decode_inputs(w["lens"][:1] * args.batch, w["hkv"], w["hq"], w["dtype"], w["layout"],
                                 w["needles"], w["seed"], "cuda")
    st = decode_setup(torch, msa, inp, w["k_scored"], w["k_total"])
    pool_ms = time_op(torch, timer, lambda: msa.msa_pool_block_keys(st["desc"], 0, -1, st["pooled"], st["ws"].buf,
                                                                     st["ws"].nbytes), 5, 2)

    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.5)
    step_samples = []
    step_ms, sel_ms, att_ms = time_decode(torch, msa, timer, st, inp, args.steps, args.warmup, dist, step_samples)
    clk = clocks.stop()
    step_ms = dist.max(step_ms)
    att_ms = dist.max(att_ms)
    sel_ms = dist.max(sel_ms)
    status = msa.msa_read_device_status(st["ws"].buf)

    e2e_ms, h2d, d2h = time_e2e_decode(torch, msa, timer, st, inp, max(5, args.steps // 2), 2)
    e2e_ms = dist.max(e2e_ms)

    pooled_b, sel_b, qo_b = decode_bytes(inp, w["k_total"])
    att_bytes = sel_b + qo_b  # the attention kernel reads the selected K/V and q, writes out
    pool_bytes = sum(n for n in inp.lens) * inp.num_kv_heads * 256 * (1 + 1 / 64)
    del inp, st
    torch.cuda.empty_cache()

    extras = {}
    if not args.no_extras and world == 1:
        extras["decode_1m"] = extras_decode(torch, msa, timer, "decode_1m", max(10, args.steps // 2), 3, hbm)
        extras["ragged_paged_decode"] = extras_decode(torch, msa, timer, "ragged_paged_decode",
                                                      max(10, args.steps // 2), 3, hbm)
        extras["prefill_8k_on_128k"] = extras_prefill(torch, msa, timer, max(5, args.steps // 5), 2, tf_burst)
        extras["decode_128k_token_max"] = extras_token_max(torch, msa, timer, max(10, args.steps // 2), 3, hbm)

    cpu = None
    if rank == 0 and not args.no_cpu:
        cpu = cpu_baseline(name, target_seconds=15.0)

    att_gbps = att_bytes / (att_ms * 1e-3) / 1e9
    step_bytes = pooled_b + sel_b + qo_b
    step_gbps = step_bytes / (step_ms * 1e-3) / 1e9
    traffic = recorded_traffic("decode_step_kernel", "step.cu")
    line = {
        "metric": METRIC, "value": round(step_ms * 1e3, 3), "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(step_ms, 6), "higher_is_better": False, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {
            "workload": f"decode_128k: {args.batch} sequences x 131072 tokens, 8 KV heads, 64 query heads, head dim 128, "
                        "64-token blocks, top-31 scored blocks + newest block, 16 needle blocks per (seq, head)",
            "global_batch": args.batch * world, "seq_len": 131072, "parallelism": f"replicas x{world}",
            "l2": "flushed before every timed step (512 MB written, then 256 MB read)",
            "step": "msa_sparse_decode_step (block scores, top-k and sparse attention in one kernel), replayed as a "
                    "CUDA graph; summary keys pooled beforehand",
        },
        "tokens_per_s": round(args.batch * world / (step_ms * 1e-3), 1),
        "step_us_quantiles": quantiles_us(step_samples),
        "step_GBps": round(step_gbps, 1),
        "step_bytes": step_bytes,
        "roofline": {"kernel": "decode_step_kernel (fused scores + top-k + sparse flash-decode)", "bound": "hbm",
                     "achieved": round(step_gbps, 1), "peak": hbm, "unit": "GB/s",
                     "frac": round(step_gbps / hbm, 4), "peak_source": f"{peak_src} (hbm_gbs)",
                     "algorithmic_bytes_per_launch": step_bytes, "traffic": traffic},
        "two_kernel_form": {"select_us": round(sel_ms * 1e3, 3), "attend_us": round(att_ms * 1e3, 3),
                            "attend_GBps": round(att_gbps, 1), "attend_frac": round(att_gbps / hbm, 4)},
        "pool_block_keys": {"us": round(pool_ms * 1e3, 2), "GBps": round(pool_bytes / (pool_ms * 1e-3) / 1e9, 1)},
        "e2e": {"value": round(e2e_ms * 1e3, 3), "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": args.steps,
        "clocks": clk,
        "device_status": status,
    }
    if cpu is not None:
        line["cpu_baseline"] = cpu
    if extras:
        line["extras"] = extras
    if rank == 0:
        print(json.dumps(line), flush=True)
    dist.close()


# --------------------------------------------------------------------------- CPU oracle (baseline and reference arm)

def _oracle_unit(args):
    """One (sequence, KV head) decode unit of the 128K workload on the CPU:
    score + select + attend (summary keys precomputed). Returns seconds."""
    seed, ctx, grp, k_scored, k_total, needles = args
    import numpy as np
    import torch
    from oracle import msa_oracle as O
    from synth import make_decode_inputs
    inp = make_decode_inputs([ctx], 1, grp, "bf16", "contiguous", needles=needles, seed=seed)
    q = inp.q[0].double().numpy()
    k = inp.k[0, 0].double().numpy()
    v = inp.v[0, 0].double().numpy()
    pooled, _ = O.pool_block_keys(k, ctx, "bf16")
    t0 = time.perf_counter()
    O.decode_unit(q, k, v, ctx, k_scored, k_total, SCALE, "bf16", pooled=pooled)
    return time.perf_counter() - t0


def host_cpu_model() -> str:
    """The host CPU's name (x86: /proc/cpuinfo "model name"; Arm: the
    implementer / part codes there), else the machine type."""
    import platform
    try:
        with open("/proc/cpuinfo") as f:
            info = f.read()
        for key in ("model name", "Model Name", "Processor"):
            for line in info.splitlines():
                if line.split(":")[0].strip() == key and ":" in line:
                    return line.split(":", 1)[1].strip()
        fields = {}
        for line in info.splitlines():
            if ":" in line:
                k, v = line.split(":", 1)
                fields.setdefault(k.strip(), v.strip())
        if "CPU part" in fields:
            return f"{platform.machine()} implementer {fields.get('CPU implementer', '?')} part {fields['CPU part']}"
    except OSError:
        pass
    return platform.machine() or "unknown"


class OraclePool:
    """The oracle as it stands, run on decode units of the 128K workload in a
    pool of single-threaded spawned workers, one per host core."""

    def __init__(self, name: str = "decode_128k"):
        import multiprocessing as mp
        from synth import WORKLOADS
        self.w = WORKLOADS[name]
        self.cores = os.cpu_count() or 1
        env_keys = ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS")
        old = {k: os.environ.get(k) for k in env_keys}
        for k in env_keys:
            os.environ[k] = "1"
        try:
            self.pool = mp.get_context("spawn").Pool(self.cores)
        finally:
            for k, v in old.items():
                if v is None:
                    os.environ.pop(k, None)
                else:
                    os.environ[k] = v
        grp = self.w["hq"] // self.w["hkv"]
        self.pool.map(_oracle_unit, [(7, 4096, grp, 8, 9, 1)] * self.cores)  # import warm-up
        self.round = 0

    def step(self) -> tuple:
        """One round: one unit per worker. Returns (extrapolated seconds per
        full step, seconds per unit, wall seconds)."""
        w = self.w
        grp = w["hq"] // w["hkv"]
        seeds = [2000 + self.round * self.cores + i for i in range(self.cores)]
        self.round += 1
        t0 = time.perf_counter()
        per_unit = self.pool.map(_oracle_unit, [(sd, w["lens"][0], grp, w["k_scored"], w["k_total"], w["needles"])
                                                for sd in seeds])
        wall = time.perf_counter() - t0
        unit_s = statistics.mean(per_unit)
        return math.ceil(self.units_per_step / self.cores) * unit_s, unit_s, wall

    @property
    def units_per_step(self) -> int:
        return len(self.w["lens"]) * self.w["hkv"]

    def describe(self, rounds: int) -> str:
        return (f"{rounds} round(s) of {self.cores} (sequence, KV head) units of 131072 tokens, one per "
                f"single-threaded worker (score + top-k + attention, float64 numpy; summary keys precomputed); "
                f"a full step = {self.units_per_step} units = {math.ceil(self.units_per_step / self.cores)} rounds")

    def close(self):
        self.pool.close()
        self.pool.join()


def cpu_baseline(name: str, target_seconds: float = 15.0) -> dict:
    pool = OraclePool(name)
    try:
        vals, t_start, rounds = [], time.perf_counter(), 0
        while rounds < 1 or (time.perf_counter() - t_start < target_seconds and rounds < 8):
            step_s, _, _ = pool.step()
            vals.append(step_s)
            rounds += 1
        return {"value": round(statistics.mean(vals) * 1e6, 1), "unit": UNIT, "cores": pool.cores, "kind": "oracle",
                "cpu_model": host_cpu_model(), "sample": pool.describe(rounds)}
    finally:
        pool.close()


def run_reference(args):
    world, rank, _ = dist_env()
    if world > 1 and rank != 0:
        return
    pool = OraclePool("decode_128k")
    try:
        for _ in range(args.warmup):
            pool.step()
        vals = [pool.step()[0] for _ in range(args.steps)]
    finally:
        pool.close()
    val = statistics.mean(vals) * 1e6
    line = {"metric": METRIC, "value": round(val, 1), "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(val / 1e3, 3), "higher_is_better": False,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic", "impl": "reference",
            "config": {"workload": "decode_128k: 8 sequences x 131072 tokens, 8 KV heads, 64 query heads, "
                                   "head dim 128, 64-token blocks, top-31 scored blocks + newest block",
                       "global_batch": 8, "seq_len": 131072, "parallelism": "CPU oracle"},
            "cpu_baseline": {"value": round(val, 1), "unit": UNIT, "cores": pool.cores, "kind": "oracle",
                             "cpu_model": host_cpu_model(), "sample": pool.describe(args.steps)},
            "e2e": {"value": round(val, 1), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_only(args):
    import torch
    from sparse_attention_step_gb300 import build, msa
    build.build()
    msa.load()
    hbm, tf_burst, _, _ = peaks()
    timer = Timer(torch)
    if args.only == "prefill":
        res = extras_prefill(torch, msa, timer, args.steps, args.warmup, tf_burst)
    else:
        res = extras_token_max(torch, msa, timer, args.steps, args.warmup, hbm)
    print(json.dumps(res), flush=True)


def main():
    args = parse()
    if args.only is not None:
        run_only(args)
        return
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()

"""Benchmark of the two-stage block-sparse GQA attention hot path on GB300.

Headline workload: decode over a bf16 KV cache of 8 sequences x 131072 tokens,
8 KV heads / 64 query heads, head dim 128, 64-token blocks, top-31 blocks plus
the newest block. One step = Step 1 (group index query, block scores, top-k)
plus Step 2 (sparse flash-decode with split-K combine) for one query token per
sequence, through msa_sparse_decode_step. The summary keys are pooled once
beforehand (they change only when a block fills) and that pass is reported
separately.

Timing of the headline value: W untimed warm-up steps, then EXACTLY K steps run
back to back as one CUDA graph and bracketed by CUDA events on the launching
stream (barrier + synchronize on both sides). Step i runs on replica i mod R of
the workload (R independent sets of inputs with the same shapes and recipe,
replica 0 being the workload itself); R is chosen so that the other replicas'
step bytes between two uses of a replica exceed three times the L2 (129 MB),
so no step finds its inputs in L2. The L2 is also flushed before the timed
region. Each step's time is also measured in isolation (L2 flushed before it,
one step between events) and reported as isolated_step_us.

Clocks are sampled with nvidia-smi over the whole headline measurement.

Prints ONE JSON line on rank 0. Under torchrun (N > 1) every rank runs an
independent replica on its own GPU (the path shards by sequence and head with
no exchange), the timed region is bracketed by barriers and the slowest rank's
time is reported.

--impl reference times the CPU oracle (scalar C, OpenMP across units) on the
host cores on a bounded sample of the headline workload's units, scaled to a
full step, and prints the same JSON line with "impl": "reference".
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
L2_BYTES = 129 << 20
L2_FLUSH_BYTES = 512 << 20
L2_CLEAN_BYTES = 256 << 20
KV_BLOCK_BYTES = 64 * 128 * 2  # one 64-token K (or V) block in bf16


def parse(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-extras", action="store_true", help="time only the headline workload")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU-oracle baselines")
    ap.add_argument("--only", choices=["prefill", "token_max", "decode_128k", "decode_1m", "ragged_paged_decode"],
                    default=None, help="time one workload and print its figures (profiling)")
    ap.add_argument("--batch", type=int, default=8,
                    help="sequences of the 131072-token decode workload (8 = the benchmark; fewer for profiling)")
    ap.add_argument("--replicas", type=int, default=0,
                    help="input replicas of --only decode workloads (0 = enough to keep inputs out of L2; 1 for "
                         "small profiling captures)")
    return ap.parse_args(argv)


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


def no_dist():
    d = Dist.__new__(Dist)
    d.dist = None
    return d


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


def headline_config(batch: int, world: int) -> dict:
    """The headline workload's config, identical in both arms."""
    return {
        "workload": f"decode_128k: {batch} sequences x 131072 tokens, 8 KV heads, 64 query heads, head dim 128, "
                    "64-token blocks, top-31 scored blocks + newest block, 16 needle blocks per (seq, head)",
        "global_batch": batch * world, "seq_len": 131072, "parallelism": f"replicas x{world}",
        "l2": "inputs larger than L2: each step runs on one of R replicas in turn, R chosen so that the steps "
              "between two uses of a replica move over 3x the L2; the L2 is also flushed before the timed region",
        "step": "msa_sparse_decode_step (block scores, top-k and sparse attention in one kernel); K steps back to "
                "back in one CUDA graph; summary keys pooled beforehand",
    }


class Timer:
    """L2 flush between measurements: 512 MB written, then 256 MB of another
    buffer read, so no input is cached and no dirty line is left to write back."""

    def __init__(self, torch):
        self.torch = torch
        self.flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device="cuda")
        self.clean = torch.ones(L2_CLEAN_BYTES // 4, dtype=torch.float32, device="cuda")

    def l2_flush(self):
        self.flush.zero_()
        self.clean.sum()


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


def replicas_needed(step_bytes: int) -> int:
    """Replicas so that the other replicas' steps between two uses of one move
    more than three times the L2 (at least 2)."""
    return max(2, 1 + math.ceil(3 * L2_BYTES / max(step_bytes, 1)))


def time_rotating(torch, timer, fns, steps, warmup, dist=None):
    """Device time per step (ms) of EXACTLY ``steps`` steps run back to back,
    step i calling fns[i % len(fns)], captured as one CUDA graph and bracketed
    by CUDA events; ``warmup`` untimed steps first."""
    dist = dist or no_dist()
    r = len(fns)
    g_warm = capture(torch, lambda: [fns[i % r]() for i in range(max(1, warmup))])
    g_timed = capture(torch, lambda: [fns[i % r]() for i in range(steps)])
    g_warm.replay()
    torch.cuda.synchronize()
    dist.barrier()
    timer.l2_flush()
    torch.cuda.synchronize()
    dist.barrier()
    stream = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    g_timed.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    dist.barrier()
    return e0.elapsed_time(e1) / steps


def time_graph(torch, timer, g, steps, warmup, samples=None):
    """Mean device time (ms) of one replay of ``g``, the L2 flushed before each
    timed replay (each replay's time is appended to ``samples`` when given)."""
    for _ in range(warmup):
        g.replay()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for e0, e1 in ev:
        timer.l2_flush()
        e0.record(stream)
        g.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    times = [a.elapsed_time(b) for a, b in ev]
    if samples is not None:
        samples.extend(times)
    return statistics.mean(times)


def time_op(torch, timer, fn, steps, warmup, samples=None):
    """Isolated device time (ms) of ``fn`` (library calls only) replayed as a CUDA graph."""
    fn()
    torch.cuda.synchronize()
    return time_graph(torch, timer, capture(torch, fn), steps, warmup, samples)


def quantiles_us(ms_samples):
    """p10 / median / p90 of per-step times (ms in, microseconds out), this rank."""
    xs = sorted(ms_samples)
    if not xs:
        return None
    pick = lambda f: round(xs[min(len(xs) - 1, int(f * len(xs)))] * 1e3, 3)  # noqa: E731
    return {"p10": pick(0.1), "p50": round(statistics.median(xs) * 1e3, 3), "p90": pick(0.9)}


def empty_launch_us(torch, reps=50):
    """Median time between two events around one replay of a graph holding one
    tiny kernel: the launch-and-event floor inside every isolated figure."""
    x = torch.zeros(1, device="cuda")
    g = capture(torch, lambda: x.add_(1))
    ts = []
    for _ in range(reps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        g.replay()
        e1.record()
        e1.synchronize()
        ts.append(e0.elapsed_time(e1) * 1e3)
    return statistics.median(ts)


# --------------------------------------------------------------------------- decode workloads (our arm)

def make_replica(name, r, device="cuda", lens=None):
    """Replica r of a decode workload: r = 0 is the workload itself; r > 0 the
    same shapes and recipe from another seed."""
    from synth import WORKLOADS, make_decode_inputs, make_workload
    w = WORKLOADS[name]
    if r == 0 and lens is None:
        return make_workload(name, device=device)
    from synth import workload_lens
    lens = lens if lens is not None else workload_lens(name)
    return make_decode_inputs(lens, w["hkv"], w["hq"], w["dtype"], w["layout"], w["needles"], w["seed"] + 7919 * r,
                              device)


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
    msa.msa_pool_block_keys(desc, 0, -1, pooled, ws.buf, ws.nbytes)
    return dict(inp=inp, desc=desc, ws=ws, pooled=pooled, idx=idx, out=out, lse=lse, cfg=cfg, hq=hq, k_total=k_total,
                k_scored=k_scored)


def decode_step(msa, st, q=None, out=None):
    """The whole decode step through msa_sparse_decode_step (one kernel for
    contiguous bf16 caches, select then attend otherwise)."""
    msa.msa_sparse_decode_step(st["inp"].q if q is None else q, st["hq"], st["pooled"], st["desc"], st["cfg"],
                               st["idx"], st["k_total"], SCALE, st["out"] if out is None else out, st["lse"],
                               st["ws"].buf, st["ws"].nbytes)


def decode_select(msa, st):
    msa.msa_select_topk_blocks(st["inp"].q, st["hq"], 1, st["pooled"], st["desc"], st["cfg"], st["idx"],
                               st["k_total"], None, st["ws"].buf, st["ws"].nbytes)


def decode_attend(msa, st):
    msa.msa_sparse_attn_decode(st["inp"].q, st["hq"], st["desc"], st["idx"], st["k_total"], SCALE, st["out"],
                               st["lse"], st["ws"].buf, st["ws"].nbytes)


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


def measure_decode(torch, msa, timer, name, steps, warmup, hbm, dist=None, lens=None, n_rep=0):
    """Back-to-back steady-state step time over rotating replicas, the isolated
    step, the two-kernel form and the dense comparator on the same inputs."""
    from synth import WORKLOADS
    w = WORKLOADS[name]
    st0 = decode_setup(torch, msa, make_replica(name, 0, lens=lens), w["k_scored"], w["k_total"])
    pooled_b, sel_b, qo_b = decode_bytes(st0["inp"], w["k_total"])
    step_bytes = pooled_b + sel_b + qo_b
    n_rep = n_rep or replicas_needed(step_bytes)
    sts = [st0] + [decode_setup(torch, msa, make_replica(name, r, lens=st0["inp"].lens), w["k_scored"], w["k_total"])
                   for r in range(1, n_rep)]
    for st in sts:
        decode_step(msa, st)
    torch.cuda.synchronize()
    step_ms = time_rotating(torch, timer, [lambda st=st: decode_step(msa, st) for st in sts], steps, warmup, dist)
    iso_samples = []
    iso_ms = time_op(torch, timer, lambda: decode_step(msa, st0), max(10, steps // 2), 3, iso_samples)
    decode_select(msa, st0)
    decode_attend(msa, st0)
    sel_ms = time_op(torch, timer, lambda: decode_select(msa, st0), max(10, steps // 2), 3)
    att_ms = time_op(torch, timer, lambda: decode_attend(msa, st0), max(10, steps // 2), 3)
    dense_out = torch.empty_like(st0["inp"].q)
    dense_lse = torch.empty_like(st0["lse"])
    dense_ms = time_op(torch, timer, lambda: msa.msa_dense_gqa_decode(
        st0["inp"].q, st0["hq"], st0["desc"], SCALE, dense_out, dense_lse, st0["ws"].buf, st0["ws"].nbytes),
        max(3, steps // 10), 2)
    inp = st0["inp"]
    dense_bytes = sum(inp.lens) * inp.num_kv_heads * 2 * 128 * 2 + qo_b
    # the step's own outputs on replica 0 (for the CPU leg's parity check)
    decode_step(msa, st0)
    torch.cuda.synchronize()
    status = max(msa.msa_read_device_status(st["ws"].buf) for st in sts)
    res = {
        "workload": name, "us_per_step": step_ms * 1e3, "replicas": n_rep,
        "isolated_step_us": iso_ms * 1e3, "isolated_step_us_quantiles": quantiles_us(iso_samples),
        "step_GBps": step_bytes / (step_ms * 1e-3) / 1e9,
        "step_roofline_frac": step_bytes / (step_ms * 1e-3) / 1e9 / hbm,
        "bytes_per_step": step_bytes, "summary_bytes": pooled_b, "selected_kv_bytes": sel_b,
        "two_kernel_select_us": sel_ms * 1e3, "two_kernel_attend_us": att_ms * 1e3,
        "attend_GBps": (sel_b + qo_b) / (att_ms * 1e-3) / 1e9,
        "dense_us": dense_ms * 1e3, "dense_GBps": dense_bytes / (dense_ms * 1e-3) / 1e9,
        "dense_over_sparse": dense_ms / step_ms, "device_status": status,
    }
    keep = {"inp": inp, "idx": st0["idx"], "out": st0["out"], "lse": st0["lse"], "st": st0}
    del sts
    return res, keep


def extras_k1050(torch, msa, timer, keep, steps, hbm, dense_us):
    """1M context with k near the ratio the guide implies (~6.4% of 16384
    blocks): k > 64 runs the selection and attention kernels in turn."""
    inp = keep["inp"]
    k_big = 1050
    st2 = decode_setup(torch, msa, inp, k_big, k_big + 1)
    big_ms = time_op(torch, timer, lambda: decode_step(msa, st2), max(5, steps // 2), 2)
    pb2, sb2, qb2 = decode_bytes(inp, k_big + 1)
    res = {"k_scored": k_big, "isolated_step_us": big_ms * 1e3,
           "step_GBps": (pb2 + sb2 + qb2) / (big_ms * 1e-3) / 1e9,
           "step_roofline_frac": (pb2 + sb2 + qb2) / (big_ms * 1e-3) / 1e9 / hbm,
           "bytes_per_step": pb2 + sb2 + qb2, "dense_over_sparse": dense_us / (big_ms * 1e3),
           "device_status": msa.msa_read_device_status(st2["ws"].buf)}
    del st2
    return res


def time_e2e_decode(torch, msa, timer, st, steps, warmup):
    """The same step through the C ABI with the per-step inputs (the new query
    token of every sequence) in pinned host memory and the output read back,
    both inside the timed region."""
    inp = st["inp"]
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
        decode_step(msa, st, q=q_dev)
        out_host.copy_(st["out"], non_blocking=True)
        e1.record(stream)
        e1.synchronize()
        if i >= warmup:
            times.append(e0.elapsed_time(e1))
    nbytes = q_host.numel() * q_host.element_size()
    return statistics.mean(times), nbytes, nbytes


def extras_token_max(torch, msa, timer, steps, warmup, hbm):
    """The decode step with the guide-literal Step 1 (token-level scores
    against a shared index-key head, block max pool) on the 128K x 8 shape:
    select (token-max scores + top-k) then sparse attention; back to back over
    input replicas like the other decode workloads, and isolated."""
    from synth import make_decode_inputs, make_index_keys
    k_scored, k_total = 31, 32
    cfg = msa.select_cfg(k_scored, mode=msa.MSA_SCORE_TOKEN_MAX)
    reps = []
    for r in range(3):  # the other replicas move > 3 x L2 between two uses of one
        inp = make_decode_inputs([131072] * 8, 8, 64, "bf16", "contiguous", seed=1006 + 7919 * r, device="cuda")
        ik = make_index_keys(inp, needles=8, seed=1007 + 7919 * r)
        reps.append((inp, ik, decode_setup(torch, msa, inp, k_scored, k_total)))

    def step_of(inp, ik, st):
        return lambda: msa.msa_sparse_decode_step(inp.q, st["hq"], ik.kidx, st["desc"], cfg, st["idx"], k_total,
                                                  SCALE, st["out"], st["lse"], st["ws"].buf, st["ws"].nbytes)

    fns = [step_of(*rep) for rep in reps]
    for fn in fns:
        fn()
    torch.cuda.synchronize()
    b2b_ms = time_rotating(torch, timer, fns, steps, warmup)
    inp, ik, st = reps[0]
    step_ms = time_op(torch, timer, fns[0], max(10, steps // 2), warmup)
    sel_ms = time_op(torch, timer, lambda: msa.msa_select_topk_blocks(
        inp.q, st["hq"], 1, ik.kidx, st["desc"], cfg, st["idx"], k_total, None, st["ws"].buf, st["ws"].nbytes),
        max(10, steps // 2), warmup)
    kidx_b = sum(min(n // 64, (n + 63) // 64 - 1) * 64 for n in inp.lens) * 128 * 2
    _, sel_b, qo_b = decode_bytes(inp, k_total)
    total = kidx_b + sel_b + qo_b
    status = max(msa.msa_read_device_status(rep[2]["ws"].buf) for rep in reps)
    res = {
        "workload": "decode_128k_token_max: 8 x 131072 tokens, 8 KV / 64 query heads, shared bf16 index-key "
                    "head, top-31 + newest, 8 needle tokens per (seq, head)",
        "us_per_step": b2b_ms * 1e3, "replicas": len(reps),
        "step_GBps": total / (b2b_ms * 1e-3) / 1e9, "step_roofline_frac": total / (b2b_ms * 1e-3) / 1e9 / hbm,
        "isolated_step_us": step_ms * 1e3, "select_us": sel_ms * 1e3,
        "select_GBps": kidx_b / (sel_ms * 1e-3) / 1e9, "bytes_per_step": total, "device_status": status,
    }
    del reps, inp, ik, st, fns
    torch.cuda.empty_cache()
    return res


def prefill_flop(q_start, n_new, k_scored, grp, hkv):
    """Algorithmic FLOPs of the sparse chunk: 4 * D per visible (query row, key)
    pair, over each tile's k_scored earlier blocks (all visible) and its causal
    diagonal block; and those of dense causal attention."""
    from sparse_attention_step_gb300.msa import chunk_tile_rows
    sel_pairs = 0
    for j, lo, hi in chunk_tile_rows(q_start, n_new):
        diag = q_start // 64 + j
        sel_pairs += (hi - lo) * min(k_scored, diag) * 64
        sel_pairs += sum((q_start + r) - diag * 64 + 1 for r in range(lo, hi))
    sparse = 4 * 128 * grp * hkv * sel_pairs
    dense = 4 * 128 * grp * hkv * sum(q_start + r + 1 for r in range(n_new))
    return sparse, dense


def extras_prefill(torch, msa, timer, steps, warmup, tflops_peak):
    from synth import WORKLOADS, make_workload
    w = WORKLOADS["prefill_8k_on_128k"]
    inp = make_workload("prefill_8k_on_128k", device="cuda")
    desc = msa.kv_desc(inp.k, inp.v, inp.seq_lens)
    hq, n = inp.num_q_heads, inp.n_new
    kt = w["k_total"]
    need = max(msa.msa_workspace_size(op, desc, hq, n, kt) for op in (msa.MSA_OP_SELECT_PREFILL, msa.MSA_OP_PREFILL))
    ws = msa.Workspace(need)
    pooled = torch.empty(msa.pooled_shape(desc), dtype=inp.k.dtype, device="cuda")
    n_tiles = msa.chunk_tiles(inp.q_start, n)
    idx = torch.empty(n_tiles, inp.num_kv_heads, kt, dtype=torch.int32, device="cuda")
    out = torch.empty_like(inp.q)
    lse = torch.empty(n, hq, dtype=torch.float32, device="cuda")
    cfg = msa.select_cfg(w["k_scored"], True, 64, inp.q_start)
    pool_ms = time_op(torch, timer, lambda: msa.msa_pool_block_keys(desc, 0, -1, pooled, ws.buf, ws.nbytes), 5, 2)
    sel_ms = time_op(torch, timer, lambda: msa.msa_select_topk_blocks(
        inp.q, hq, n, pooled, desc, cfg, idx, kt, None, ws.buf, ws.nbytes), steps, warmup)
    att_ms = time_op(torch, timer, lambda: msa.msa_sparse_attn_prefill(
        inp.q, hq, n, inp.q_start, desc, idx, kt, SCALE, out, lse, ws.buf, ws.nbytes), steps, warmup)
    dense_out = torch.empty_like(inp.q)
    dense_ms = time_op(torch, timer, lambda: msa.msa_dense_gqa_prefill(
        inp.q, hq, n, inp.q_start, desc, SCALE, dense_out, None, ws.buf, ws.nbytes), 3, 1)
    # the guide-literal Step 1 on the same chunk: token scores against one shared
    # bf16 index-key head (N(0,1), seeded), block max pool, top-k
    g_idx = torch.Generator(device="cuda")
    g_idx.manual_seed(4007)
    kidx = torch.randn(1, desc.max_tokens, 128, generator=g_idx, device="cuda").to(torch.bfloat16)
    idx_tm = torch.empty_like(idx)
    cfg_tm = msa.select_cfg(w["k_scored"], True, 64, inp.q_start, mode=msa.MSA_SCORE_TOKEN_MAX)
    sel_tm_ms = time_op(torch, timer, lambda: msa.msa_select_topk_blocks(
        inp.q, hq, n, kidx, desc, cfg_tm, idx_tm, kt, None, ws.buf, ws.nbytes), steps, warmup)
    # the step's own outputs for the CPU leg's parity check
    msa.msa_select_topk_blocks(inp.q, hq, n, pooled, desc, cfg, idx, kt, None, ws.buf, ws.nbytes)
    msa.msa_sparse_attn_prefill(inp.q, hq, n, inp.q_start, desc, idx, kt, SCALE, out, lse, ws.buf, ws.nbytes)
    torch.cuda.synchronize()
    grp = hq // inp.num_kv_heads
    sparse_flop, dense_flop = prefill_flop(inp.q_start, n, w["k_scored"], grp, inp.num_kv_heads)
    total = inp.q_start + n
    status = msa.msa_read_device_status(ws.buf)
    res = {
        "workload": "prefill_8k_on_128k", "select_us": sel_ms * 1e3, "attend_us": att_ms * 1e3,
        "attend_TFLOPs": sparse_flop / (att_ms * 1e-3) / 1e12,
        "attend_tensor_frac": sparse_flop / (att_ms * 1e-3) / 1e12 / tflops_peak,
        "step_us": (sel_ms + att_ms) * 1e3, "sparse_gflop": sparse_flop / 1e9,
        "dense_us": dense_ms * 1e3, "dense_TFLOPs": dense_flop / (dense_ms * 1e-3) / 1e12,
        "dense_over_sparse_step": dense_ms / (sel_ms + att_ms),
        "pool_us": pool_ms * 1e3, "pool_GBps": total * inp.num_kv_heads * 256 / (pool_ms * 1e-3) / 1e9,
        "select_token_max_us": sel_tm_ms * 1e3, "device_status": status,
    }
    keep = {"inp": inp, "idx": idx, "out": out, "lse": lse, "pooled": pooled}
    del kidx, ws
    return res, keep


# --------------------------------------------------------------------------- CPU oracle (baseline and reference arm)

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


def unit_rows(inp, s):
    """[Hkv, capacity, D] keys and values of sequence s in logical token order
    (gathered through the page table for the paged layout), on the host."""
    if inp.layout == "contiguous":
        return inp.k[s].cpu(), inp.v[s].cpu()
    n_pages = -(-inp.lens[s] // 64)
    pages = inp.page_table[s, :n_pages].long()
    hkv = inp.num_kv_heads
    k = inp.k[pages].permute(1, 0, 2, 3).reshape(hkv, n_pages * 64, -1)
    v = inp.v[pages].permute(1, 0, 2, 3).reshape(hkv, n_pages * 64, -1)
    return k.cpu(), v.cpu()


def oracle_decode_units(inp, seqs, k_scored, k_total):
    """Host arrays of the sampled sequences' units for the oracle: q [U, G, D],
    k, v [U, T, D], lens, and the stored summaries (pooled by the oracle,
    outside the timed region: the GPU side also pools beforehand)."""
    import torch
    from oracle import msa_oracle as O
    hkv = inp.num_kv_heads
    grp = inp.num_q_heads // hkv
    qs, ks, vs, lens = [], [], [], []
    t_max = max(-(-inp.lens[s] // 64) * 64 for s in seqs)
    for s in seqs:
        k, v = unit_rows(inp, s)
        pad = t_max - k.shape[1]
        if pad:
            k = torch.nn.functional.pad(k, (0, 0, 0, pad))
            v = torch.nn.functional.pad(v, (0, 0, 0, pad))
        ks.append(k)
        vs.append(v)
        qs.append(inp.q[s].view(hkv, grp, -1).cpu())
        lens += [inp.lens[s]] * hkv
    q = torch.cat(qs)
    k = torch.cat(ks)
    v = torch.cat(vs)
    sel = O.decode_select_units(q, k, lens, inp.dtype, k_scored, k_total, 1, want_scores=True, want_pooled=True)
    return dict(q=q, k=k, v=v, lens=lens, pooled=sel["pooled"], scores=sel["scores"], gap=sel["gap"],
                selected=sel["selected"])


def cpu_decode_baseline(inp, seqs, k_scored, k_total, units_per_step, target_s=10.0, gpu=None):
    """The oracle (C, OpenMP across units) timed on the sampled sequences'
    units: whole decode steps (index query, scores, top-k, attention) from
    summaries pooled beforehand, scaled to a full step. With ``gpu`` (the GPU
    step's idx / out of the same inputs), also the selection rule and output
    parity on those units."""
    from oracle import msa_oracle as O
    d = oracle_decode_units(inp, seqs, k_scored, k_total)
    n_units = len(d["lens"])
    vals, t0 = [], time.perf_counter()
    while not vals or (time.perf_counter() - t0 < target_s and len(vals) < 50):
        t1 = time.perf_counter()
        sel, o, lse = O.decode_step_units(d["q"], d["pooled"], d["k"], d["v"], d["lens"], k_scored, k_total, SCALE)
        vals.append(time.perf_counter() - t1)
    per_step = statistics.median(vals) * units_per_step / n_units
    res = {"value": round(per_step * 1e6, 1), "unit": UNIT, "cores": O.num_threads(), "kind": "oracle",
           "cpu_model": host_cpu_model(),
           "sample": f"{n_units} (sequence, KV head) units of {len(seqs)} sequence(s) of the same workload, "
                     f"{len(vals)} timed runs (median), scaled by {units_per_step}/{n_units} units to a full "
                     f"step; scalar C oracle, double precision, OpenMP across units; summaries pooled beforehand"}
    if gpu is not None:
        res["parity"] = decode_parity(d, sel, o, gpu, seqs, inp, k_scored)
    return res


def decode_parity(d, sel, o, gpu, seqs, inp, k_scored):
    """Selection rule and outputs of the GPU step on the oracle's units."""
    import numpy as np
    hkv = inp.num_kv_heads
    grp = inp.num_q_heads // hkv
    idx = gpu["idx"].cpu().numpy()
    out = gpu["out"].float().cpu().numpy()
    equal = near = bad = 0
    err = 0.0
    for u, s in enumerate([s for s in seqs for _ in range(hkv)]):
        h = u % hkv
        got = idx[s, h]
        if list(got) == list(sel[u]):
            equal += 1
            err = max(err, float(np.abs(out[s, h * grp:(h + 1) * grp] - o[u]).max()))
            continue
        s_k, s_k1 = d["gap"][u]
        if np.isfinite(s_k) and s_k - s_k1 < 1e-3 * max(abs(s_k), 1e-30):
            near += 1
        else:
            bad += 1
    return {"units": len(sel), "lists_equal": equal, "near_ties": near, "mismatches": bad,
            "max_abs_out_err_on_equal_lists": round(err, 6), "tolerance": 2e-2}


def cpu_prefill_baseline(keep, k_scored, k_total, target_s=10.0):
    """The oracle on a sample of (tile, KV head) units of the prefill chunk
    (select + causal attention), scaled to the whole chunk, with the GPU's
    selection and outputs compared on those units."""
    import numpy as np
    import torch
    from oracle import msa_oracle as O
    inp = keep["inp"]
    hkv = inp.num_kv_heads
    total = inp.q_start + inp.n_new
    k = inp.k[0, :, :total].cpu()
    v = inp.v[0, :, :total].cpu()
    q = inp.q.cpu()
    mb = -(-total // 64)
    pooled = np.full((hkv, mb, 128), np.nan)
    for h in range(hkv):
        p, _ = O.pool_block_keys(k[h], total, "bf16")
        pooled[h, :p.shape[0]] = p
    tiles = O.prefill_tiles(inp.q_start, inp.n_new)
    pick = [tiles[i][0] for i in np.linspace(0, len(tiles) - 1, 4).astype(int)]
    units = [(j, h) for j in pick for h in range(hkv)]
    vals, t0 = [], time.perf_counter()
    while not vals or (time.perf_counter() - t0 < target_s and len(vals) < 20):
        t1 = time.perf_counter()
        sel, o, lse = O.prefill_tile_units(units, inp.q_start, q, pooled, k, v, k_scored, k_total, SCALE)
        vals.append(time.perf_counter() - t1)
    n_all = len(tiles) * hkv
    per_chunk = statistics.median(vals) * n_all / len(units)
    idx = keep["idx"].cpu().numpy()
    out = keep["out"].float().cpu().numpy()
    part = {j: (lo, hi) for j, lo, hi in tiles}
    grp = inp.num_q_heads // hkv
    equal = 0
    err = 0.0
    for u, (j, h) in enumerate(units):
        if list(idx[j, h]) == list(sel[u]):
            equal += 1
            lo, hi = part[j]
            err = max(err, float(np.abs(out[lo:hi, h * grp:(h + 1) * grp] - o[lo:hi, h * grp:(h + 1) * grp]).max()))
    return {"value": round(per_chunk * 1e6, 1), "unit": "µs/chunk", "cores": O.num_threads(), "kind": "oracle",
            "cpu_model": host_cpu_model(),
            "sample": f"{len(units)} (tile, KV head) units ({len(pick)} tiles spread over the chunk x {hkv} heads), "
                      f"{len(vals)} timed runs (median), scaled by {n_all}/{len(units)} units to the whole chunk; "
                      "scalar C oracle, double precision, OpenMP across units",
            "parity": {"units": len(units), "lists_equal": equal, "max_abs_out_err_on_equal_lists": round(err, 6),
                       "tolerance": 2e-2}}


# --------------------------------------------------------------------------- our arm

def run_ours(args):
    import torch
    from sparse_attention_step_gb300 import build, msa

    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    dist = Dist("nccl")
    if rank == 0 or world == 1:
        build.build()
    dist.barrier()
    msa.load()
    hbm, tf_burst, tf_sus, peak_src = peaks()
    timer = Timer(torch)

    lens = [131072] * args.batch if args.batch != 8 else None
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.4)
    head, keep = measure_decode(torch, msa, timer, "decode_128k", args.steps, args.warmup, hbm, dist, lens)
    clk = clocks.stop()
    step_ms = dist.max(head["us_per_step"] / 1e3)
    e2e_ms, h2d, d2h = time_e2e_decode(torch, msa, timer, keep["st"], max(5, args.steps // 2), 3)
    e2e_ms = dist.max(e2e_ms)
    floor_us = empty_launch_us(torch)

    cpu = None
    extras = {}
    if rank == 0 and not args.no_cpu:
        cpu = cpu_decode_baseline(keep["inp"], [0, 1][:keep["inp"].batch], 31, 32, keep["inp"].batch * 8,
                                  gpu={"idx": keep["idx"], "out": keep["out"]})
    del keep
    torch.cuda.empty_cache()

    if not args.no_extras and world == 1:
        r1m, k1m = measure_decode(torch, msa, timer, "decode_1m", max(10, args.steps), 3, hbm)
        r1m["k1050"] = extras_k1050(torch, msa, timer, k1m, args.steps, hbm, r1m["dense_us"])
        if not args.no_cpu:
            r1m["cpu_baseline"] = cpu_decode_baseline(k1m["inp"], [0], 63, 64, 8,
                                                      gpu={"idx": k1m["idx"], "out": k1m["out"]})
        extras["decode_1m"] = r1m
        del k1m
        torch.cuda.empty_cache()
        rrg, krg = measure_decode(torch, msa, timer, "ragged_paged_decode", max(10, args.steps // 2), 3, hbm)
        if not args.no_cpu:
            rrg["cpu_baseline"] = cpu_decode_baseline(krg["inp"], [0, 1, 2], 47, 48, 32 * 8, target_s=8.0,
                                                      gpu={"idx": krg["idx"], "out": krg["out"]})
            rrg["cpu_baseline"]["sample"] += "; sequences 0-2 of the ragged batch (their lengths: " + \
                ", ".join(str(krg["inp"].lens[s]) for s in range(3)) + "), scaled by unit count"
        extras["ragged_paged_decode"] = rrg
        del krg
        torch.cuda.empty_cache()
        rpf, kpf = extras_prefill(torch, msa, timer, max(5, args.steps // 5), 2, tf_burst)
        if not args.no_cpu:
            rpf["cpu_baseline"] = cpu_prefill_baseline(kpf, 32, 33)
        extras["prefill_8k_on_128k"] = rpf
        del kpf
        torch.cuda.empty_cache()
        extras["decode_128k_token_max"] = extras_token_max(torch, msa, timer, max(10, args.steps // 2), 3, hbm)

    step_gbps = head["bytes_per_step"] / (step_ms * 1e-3) / 1e9
    traffic = recorded_traffic("decode_step_kernel", "step.cu")
    line = {
        "metric": METRIC, "value": round(step_ms * 1e3, 3), "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(step_ms, 6), "higher_is_better": False, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": headline_config(args.batch, world),
        "tokens_per_s": round(args.batch * world / (step_ms * 1e-3), 1),
        "replicas": head["replicas"],
        "isolated_step_us": round(head["isolated_step_us"], 3),
        "isolated_step_us_quantiles": head["isolated_step_us_quantiles"],
        "empty_launch_event_us": round(floor_us, 3),
        "step_GBps": round(step_gbps, 1),
        "step_bytes": head["bytes_per_step"],
        "roofline": {"kernel": "decode_step_kernel (fused scores + top-k + sparse flash-decode)", "bound": "hbm",
                     "achieved": round(step_gbps, 1), "peak": hbm, "unit": "GB/s",
                     "frac": round(step_gbps / hbm, 4), "peak_source": f"{peak_src} (hbm_gbs)",
                     "algorithmic_bytes_per_launch": head["bytes_per_step"], "traffic": traffic,
                     "launch_time": "mean over the K back-to-back launches of the timed region (CUDA events)"},
        "two_kernel_form": {"select_us": round(head["two_kernel_select_us"], 3),
                            "attend_us": round(head["two_kernel_attend_us"], 3),
                            "attend_GBps": round(head["attend_GBps"], 1)},
        "dense_gqa": {"us": round(head["dense_us"], 2), "GBps": round(head["dense_GBps"], 1),
                      "dense_over_sparse": round(head["dense_over_sparse"], 2)},
        "e2e": {"value": round(e2e_ms * 1e3, 3), "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": args.steps,
        "clocks": clk,
        "device_status": head["device_status"],
    }
    if cpu is not None:
        line["parity"] = cpu.pop("parity")
        line["cpu_baseline"] = cpu
    if extras:
        line["extras"] = extras
    if rank == 0:
        print(json.dumps(line), flush=True)
    dist.close()


# --------------------------------------------------------------------------- reference arm

def run_reference(args):
    """The oracle on the host cores, on the headline config: its first two
    sequences' units (16 (sequence, KV head) units), scaled to a step."""
    world, rank, _ = dist_env()
    if world > 1 and rank != 0:
        return
    import torch
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    from synth import WORKLOADS, make_decode_inputs
    w = WORKLOADS["decode_128k"]
    # the headline workload's first two sequences (the generator draws
    # sequence-major, so these are the same tensors as in our arm when made on
    # the same device)
    inp = make_decode_inputs(w["lens"][:2], w["hkv"], w["hq"], w["dtype"], w["layout"], w["needles"], w["seed"], dev)
    from oracle import msa_oracle as O
    d = oracle_decode_units(inp, [0, 1], w["k_scored"], w["k_total"])
    for _ in range(args.warmup):
        O.decode_step_units(d["q"], d["pooled"], d["k"], d["v"], d["lens"], w["k_scored"], w["k_total"], SCALE)
    vals = []
    for _ in range(args.steps):
        t1 = time.perf_counter()
        O.decode_step_units(d["q"], d["pooled"], d["k"], d["v"], d["lens"], w["k_scored"], w["k_total"], SCALE)
        vals.append(time.perf_counter() - t1)
    units_per_step = args.batch * w["hkv"]
    val = statistics.mean(vals) * units_per_step / len(d["lens"]) * 1e6
    line = {"metric": METRIC, "value": round(val, 1), "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(val / 1e3, 3), "higher_is_better": False,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic", "impl": "reference",
            "config": headline_config(args.batch, world),
            "cpu_baseline": {"value": round(val, 1), "unit": UNIT, "cores": O.num_threads(), "kind": "oracle",
                             "cpu_model": host_cpu_model(),
                             "sample": f"each step: the 16 (sequence, KV head) units of the workload's first two "
                                       f"sequences, scaled by {units_per_step}/16 units; scalar C oracle, double "
                                       "precision, OpenMP across units; summaries pooled beforehand"},
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
        res, _ = extras_prefill(torch, msa, timer, args.steps, args.warmup, tf_burst)
    elif args.only == "token_max":
        res = extras_token_max(torch, msa, timer, args.steps, args.warmup, hbm)
    else:
        lens = [131072] * args.batch if args.only == "decode_128k" and args.batch != 8 else None
        res, _ = measure_decode(torch, msa, timer, args.only, args.steps, args.warmup, hbm, lens=lens,
                                n_rep=args.replicas)
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

#!/usr/bin/env python
"""Benchmark of the block-causal decode step on one GB300 (or N, one rank each).

A step is one call of bca_decode with commit on: the attention of a batch of
64 diffusion blocks (64 masked query tokens each, 32 query / 8 KV heads,
head_dim 128) over completed prefixes of log-uniform length in [128, 32768]
held in a paged cache (pages of 16, physical pages in random order, pool of
twice the need), and the commit of the blocks' K/V into the cache (done by the
epilogue kernel that also merges split-KV partials).
Inputs are resident in HBM; the K/V working set (~1.6 GB) is larger than L2,
so no flush is needed between steps.

Prints one JSON line (rank 0).  --impl reference times the fp64 CPU oracle on
a bounded sample of the same workload instead.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "decode-step attention µs, TFLOP/s, HBM GB/s and % of roofline at B=64"
# device cycles (about 100 us) of busy-waiting queued before each row call, so
# that the events around the call time device work, not host marshalling
HOST_LEAD_CYCLES = 200_000
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "source": "fallback"}


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": float(p["hbm_gbs"]), "bf16_tflops": float(p["bf16_tflops"]),
                "bf16_tflops_sustained": float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                "source": "measured"}
    except Exception:
        return dict(FALLBACK_PEAKS)


def algorithmic(prefix_len, D, Hq, Hkv, d, S):
    """Algorithmic work of one decode step: every visible (query, key) pair
    costs 4d flops per query head; bytes count every input byte once (prefix
    K/V, Q, the block's K/V, page-table entries, lengths), the output, and
    the commit writes."""
    B = len(prefix_len)
    sumP = sum(prefix_len)
    flops = 4.0 * d * D * Hq * (sumP + B * D)
    kv = 2.0 * sumP * Hkv * d * 2
    q = B * D * Hq * d * 2.0
    blk = 2.0 * B * D * Hkv * d * 2
    out = B * D * Hq * d * 2.0
    pt = 4.0 * sum(math.ceil(P / S) for P in prefix_len) + 4.0 * B
    attn_bytes = kv + q + blk + out + pt
    commit_bytes = 2.0 * B * D * Hkv * d * 2  # writes into the pool
    return {"flops": flops, "attn_bytes": attn_bytes, "step_bytes": attn_bytes + commit_bytes,
            "sum_prefix": sumP}


class ClockSampler:
    """nvidia-smi samples (timestamped on the host) during the timed region."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.samples = []
        self.proc = None
        self.gpu = gpu_index
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), [x.strip() for x in line.split(",")]))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=5)

    def summary(self, t0, t1):
        rows = [s for (t, s) in self.samples if t0 <= t <= t1 and len(s) >= 8]
        if not rows:
            rows = [s for (_, s) in self.samples if len(s) >= 8]
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"],
                    "samples": 0}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(r[0]) for r in rows if num(r[0]) is not None]
        mx = [num(r[1]) for r in rows if num(r[1]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[4 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "power_w_max": max((num(r[2]) or 0.0) for r in rows), "samples": len(rows)}


# ---------------------------------------------------------------------------
# the CPU oracle (baseline and reference arm)
# ---------------------------------------------------------------------------

def oracle_on_sequences(seed, prefix_len, D, Hq, Hkv, d, seqs, nthreads):
    """Run the fp64 oracle on the listed sequences of the workload; returns
    (seconds, flops) of the oracle calls only."""
    import oracle
    import workloads
    secs, flops = 0.0, 0.0
    for b in seqs:
        P = prefix_len[b]
        kp, vp = workloads.sequence_prefix_kv(seed, b, P, Hkv, d)
        qb, kb, vb = workloads.sequence_block(seed, b, D, Hq, Hkv, d)
        t = time.perf_counter()
        oracle.decode(qb[None], kb[None], vb[None], [kp], [vp], nthreads=nthreads)
        secs += time.perf_counter() - t
        flops += 4.0 * d * D * Hq * (P + D)
    return secs, flops


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo, else platform)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except Exception:
        pass
    import platform
    return platform.processor() or platform.machine()


def cpu_baseline(seed, prefix_len, D, Hq, Hkv, d):
    """The fp64 oracle on the whole step: every sequence of the batch, all
    host cores, timed once."""
    nthreads = os.cpu_count() or 1
    secs, flops = oracle_on_sequences(seed, prefix_len, D, Hq, Hkv, d, range(len(prefix_len)),
                                      nthreads)
    keys = sum(prefix_len) + D * len(prefix_len)
    return {"value": flops / secs / 1e12, "unit": "TFLOP/s", "cores": nthreads, "kind": "oracle",
            "cpu_model": cpu_model(), "us_per_step": secs * 1e6,
            "sample": f"{len(prefix_len)} of {len(prefix_len)} sequences: the whole step "
                      f"({keys} keys), fp64 oracle with an explicit dense mask, "
                      f"{secs:.1f} s of oracle time"}


def run_reference(args):
    """--impl reference: the fp64 oracle, as it stands, on host cores.

    A whole decode step takes the oracle seconds, so each timed step runs a
    bounded sample of the step's sequences: the timed steps cover the batch
    once, cheapest sequences first and several per step while they fit the
    step's budget, then repeat the cheapest one, so that the whole
    --steps/--warmup run stays within a few minutes.  ``value`` is the
    oracle's measured rate; ``ms_per_step`` is the time a whole step (all 64
    sequences) takes at that rate, and ``sample_ms_per_step`` the time of the
    sample each step actually ran."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    import workloads
    D, Hq, Hkv, d = args.D, 32, 8, 128
    prefix_len = workloads.prefix_loguniform_blocks(64, 128, 32768, 64, args.seed)
    nthreads = os.cpu_count() or 1
    n_steps = args.steps + args.warmup
    budget = 150.0 / max(1, n_steps)      # seconds of oracle work per step
    est_rate = 1.5e10                     # fp64 flop/s on a many-core host (estimate)
    cost = [4.0 * d * D * Hq * (P + D) / est_rate for P in prefix_len]
    order = sorted(range(64), key=lambda b: cost[b])
    # the warm-up steps run the cheapest sequence; the timed steps then cover
    # the batch once (cheapest first, several sequences per step while they
    # fit the step's budget, an expensive one alone), after which each step
    # repeats the cheapest sequence
    step_seqs, nxt = [[order[0]]] * args.warmup, 0
    for _ in range(args.steps):
        picked, t = [], 0.0
        while nxt < 64:
            b = order[nxt]
            if picked and t + cost[b] > budget:
                break
            picked.append(b)
            t += cost[b]
            nxt += 1
        step_seqs.append(picked or [order[0]])
    secs = flops = 0.0
    covered = set()
    for i, seqs in enumerate(step_seqs):
        s, f = oracle_on_sequences(args.seed, prefix_len, D, Hq, Hkv, d, seqs, nthreads)
        if i >= args.warmup:
            secs += s
            flops += f
            covered.update(seqs)
    value = flops / secs / 1e12 if secs > 0 else 0.0
    step_flops = 4.0 * d * D * Hq * (sum(prefix_len) + 64 * D)
    whole_ms = step_flops / (value * 1e12) * 1e3 if value > 0 else None
    sample = (f"each timed step: {min(len(x) for x in step_seqs[args.warmup:])}-"
              f"{max(len(x) for x in step_seqs[args.warmup:])} of the 64 sequences ("
              f"{len(covered)} distinct sequences timed over the run), fp64 oracle with an "
              f"explicit dense mask; ms_per_step is a whole step at the measured rate")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": whole_ms, "sample_ms_per_step": 1e3 * secs / max(1, args.steps),
            "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(args, prefix_len),
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": nthreads,
                             "kind": "oracle", "cpu_model": cpu_model(), "sample": sample},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def kernel_source_hash():
    """Hash of the sources of the decode step's attention kernel (the CTA-pair
    kernel for the benchmarked shape) and what it includes."""
    import hashlib
    h = hashlib.sha256()
    for f in ("attention_pair.cu", "attn_common.cuh", "ptx_sm103.cuh", "bca_internal.h"):
        with open(os.path.join(ROOT, "block_causal_paged_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def committed_traffic(batch, D):
    """DRAM bytes per attention launch from the committed ncu summary, scaled
    to this workload; None if the kernel source changed since the capture."""
    path = os.path.join(ROOT, "profiles", "attention_decode_traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
    except Exception:
        return None, "no committed capture"
    if rec.get("kernel_source_sha256") != kernel_source_hash():
        return None, "kernel changed since the capture"
    if rec.get("batch") == batch and rec.get("D") == D:
        return float(rec["dram_bytes_per_launch"]), rec.get("command", "")
    return None, "capture is for another workload"


def workload_config(args, prefix_len):
    return {"workload": f"serving decode step: batch {args.batch} x 1 block of D={args.D} query tokens, "
                        f"32 q / 8 kv heads, head_dim 128, prefix log-uniform in [128, 32768] "
                        f"rounded to 64 (sum {sum(prefix_len)} tokens, seed {args.seed}), "
                        f"page size 16, pool 2x need in random physical order, KV commit on",
            "batch_per_gpu": args.batch, "global_batch": args.batch * args.gpus, "block_size": args.D,
            "seq_len_max": 32768, "heads": "32/8", "head_dim": 128, "page_size": 16,
            "softmax_scale": "1/sqrt(128)", "inputs": "N(0,1) bf16",
            "l2": "inputs larger than L2 (KV working set ~1.6 GB), no flush",
            "parallelism": f"{args.gpus} independent replicas, each with its own batch "
                           "(no collective on the data path)"}


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------

def rank_seed(base_seed: int, rank: int) -> int:
    """Each rank serves its own batch (weak scaling): a distinct seeded workload."""
    return base_seed + rank


def max_over_ranks(value: float, device=None) -> float:
    """Slowest rank's value (the job's step time); identity without a process group."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device or "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput_tflops(flops_per_rank: float, world: int, ms_max: float) -> float:
    """Whole-job TFLOP/s: the work of every rank over the slowest rank's time."""
    return flops_per_rank * world / (ms_max * 1e-3) / 1e12


def time_steps(torch, fn, steps, stream):
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    start.record(stream)
    for _ in range(steps):
        fn()
    end.record(stream)
    torch.cuda.synchronize()
    return start.elapsed_time(end)


def prefill_row(args, bca, workloads, torch, dev, roof, time_calls, reps, res):
    c = workloads.prefill_4x8192(seed=args.seed)
    d = bca.dims(len(c.seq_lens), c.D, c.Hq, c.Hkv, c.d, c.pool.page_size, c.pool.num_pages,
                 c.pool.max_pages_per_seq)
    q, k, v = c.q.to(dev), c.k.to(dev), c.v.to(dev)
    cu, pt = c.cu_seqlens.to(dev), c.pool.page_table.to(dev)
    kp, vp = c.pool.k_pool.to(dev), c.pool.v_pool.to(dev)
    out = torch.empty_like(q)
    ws = bca.new_workspace(d, bca.OP_PREFILL, device=dev)
    T, L = sum(c.seq_lens), max(c.seq_lens)
    ms = time_calls(lambda: bca.bca_prefill(d, q, k, v, cu, T, L, kp, vp, pt, out, ws), reps(10))
    pairs = sum(c.D * c.D * (L // c.D) * (L // c.D + 1) // 2 for L in c.seq_lens)
    flops = 4.0 * c.d * c.Hq * pairs
    bytes_ = T * (2 * c.Hq + 2 * c.Hkv) * c.d * 2.0 + 2 * T * c.Hkv * c.d * 2.0
    res["prefill"] = dict(roof(flops, bytes_, ms), kernel_us=dict(time_calls.kernel_us), workload="4 x 8192 tokens, D=64, 32/8 heads, "
                          "d=128, K/V written to pages of 16")
    ku = time_calls.kernel_us.get("attention")
    if ku:  # the attention kernel alone (the library's own events around each launch)
        k = roof(flops, bytes_, ku * 1e-3)
        res["prefill"]["kernel"] = {"name": "attention", "us": ku, "frac": k["frac"], "bound": k["bound"]}
    del q, k, v, out, kp, vp, ws


def other_rows(args, bca, workloads, torch, pk, dev, stream):
    """The block-causal prefill (4 x 8192), the QKV-post of a decode step's
    blocks, the block decode at batch 8 (prefixes 512-4096), the short causal
    extend (batch 64, 9 tokens) and the multicanvas step (batch 16, prompt 1024, 3 canvases of
    256; and 5 canvases under a 1024-token sliding window), each timed over repeated calls with CUDA events and set against
    its roofline: algorithmic flops (every visible (query, key) pair costs 4d
    per query head) and bytes (every input byte once, the output, page
    writes).  Each figure is the median over calls that each start with L2
    flushed."""
    res = {}
    only = set(args.only.split(",")) if args.only else None

    def want(name):
        return only is None or name in only

    def reps(n):
        return args.row_reps if args.row_reps else n

    def with_kernel(row, flops, bytes_, name):
        """Adds the figure of the row's dominant kernel (the library's own
        events around each launch) for the same algorithmic work."""
        ku = time_calls.kernel_us.get(name)
        if ku:
            k = roof(flops, bytes_, ku * 1e-3)
            row["kernel"] = {"name": name, "us": ku, "frac": k["frac"], "bound": k["bound"]}
        return row

    def roof(flops, bytes_, ms):
        t_mem = bytes_ / (pk["hbm_gbs"] * 1e9)
        t_flop = flops / (pk["bf16_tflops"] * 1e12)
        return {"us": ms * 1e3, "tflops": flops / (ms * 1e-3) / 1e12,
                "gbs": bytes_ / (ms * 1e-3) / 1e9,
                "bound": "tensor" if t_flop >= t_mem else "hbm",
                "frac": max(t_mem, t_flop) / (ms * 1e-3),
                "algorithmic_flops": flops, "algorithmic_bytes": bytes_}

    # every timed call starts with a cold, clean L2 (outside the events): a
    # buffer of twice the L2 size is rewritten, then another one is read, so
    # that the L2 holds none of the call's data and no dirty lines whose
    # write-back the call would pay for
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    flush_rd = torch.ones(64 << 20, dtype=torch.int32, device=dev)

    def time_calls(fn, n):
        for _ in range(3):
            fn()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(n)]
        torch.cuda.synchronize()
        bca.profile_start(16 * n + 16)
        for a, b in evs:
            flush.fill_(1)
            flush_rd.sum()
            # keep the device busy while the host marshals the call, so that
            # the events bracket device work and no host time
            torch.cuda._sleep(HOST_LEAD_CYCLES)
            a.record(stream)
            fn()
            b.record(stream)
        torch.cuda.synchronize()
        prof = bca.profile_stop()
        # per kernel kind, the mean device time of its launches (the library's
        # own event pairs around each launch)
        time_calls.kernel_us = {k: 1e3 * ms / cnt for k, (cnt, ms) in prof.items() if cnt}
        return statistics.median(a.elapsed_time(b) for a, b in evs)

    # prefill: 4 sequences of 8192 tokens, D = 64, 32/8 heads, d = 128, pages written
    if want("prefill"):
        prefill_row(args, bca, workloads, torch, dev, roof, time_calls, reps, res)


    def mc(case, window, name, desc):
        dd = bca.dims(case.B, case.canvas_len, case.Hq, case.Hkv, case.d, case.pool.page_size,
                      case.pool.num_pages, case.pool.max_pages_per_seq)
        t = {"q": case.q_live.to(dev), "k": case.k_live.to(dev), "v": case.v_live.to(dev),
             "lp": case.live_pos.to(dev), "lc": case.live_count.to(dev),
             "kp": case.pool.k_pool.to(dev), "vp": case.pool.v_pool.to(dev),
             "pt": case.pool.page_table.to(dev), "kvp": case.kv_pos.to(dev),
             "al": case.arena_len.to(dev)}
        o = torch.empty_like(t["q"])
        w = bca.new_workspace(dd, bca.OP_MULTICANVAS, device=dev)
        max_live = case.q_live.shape[1]
        fn = lambda: bca.bca_multicanvas(dd, t["q"], t["k"], t["v"], t["lp"], t["lc"], max_live,
                                         case.prompt_len, case.n_canvas, t["kp"], t["vp"], t["pt"],
                                         t["kvp"], t["al"], None, None, 0, o, w, window=window)
        ms2 = time_calls(fn, reps(20))
        P0, C = case.prompt_len, case.canvas_len
        pairs2 = 0
        for b in range(case.B):
            n = int(case.live_count[b])
            qp = case.live_pos[b, :n].long()
            lim = P0 + C * ((qp - P0) // C + 1)
            lo = (qp - window + 1).clamp(min=0) if window > 0 else torch.zeros_like(qp)
            pairs2 += int((lim - lo).sum())
        flops2 = 4.0 * case.d * case.Hq * pairs2
        A = int(case.arena_len.sum())
        nl = int(case.live_count.sum())
        bytes2 = (A + nl) * case.Hkv * case.d * 2 * 2.0 + 2 * nl * case.Hq * case.d * 2.0
        res[name] = with_kernel(dict(roof(flops2, bytes2, ms2), workload=desc,
                                     kernel_us=dict(time_calls.kernel_us)), flops2, bytes2, "attention")

    if want("qkv_post"):
        # QKV-post: batch 64 blocks of 64 tokens after the serving prefixes,
        # 32/8 heads, d = 128, norms + RoPE, the key / value rows written to pages
        Pq = workloads.prefix_loguniform_blocks(args.row_batch, 128, 32768, 64, seed=args.seed)
        cq = workloads.make_qkv_post_case(args.row_batch, 64, 32, 8, 128, prefix_len=Pq,
                                              seed=args.seed)
        dq = bca.dims(cq.B, cq.n, cq.Hq, cq.Hkv, cq.d, cq.pool.page_size, cq.pool.num_pages,
                      cq.pool.max_pages_per_seq)
        tq = {k_: v_.to(dev) for k_, v_ in (("qkv", cq.qkv), ("pos", cq.positions),
                                            ("qw", cq.q_norm_w), ("kw", cq.k_norm_w),
                                            ("wp", cq.write_pos), ("kp", cq.pool.k_pool),
                                            ("vp", cq.pool.v_pool), ("pt", cq.pool.page_table))}
        oq = torch.empty((cq.B, cq.n, cq.Hq, cq.d), dtype=torch.bfloat16, device=dev)
        ok_ = torch.empty((cq.B, cq.n, cq.Hkv, cq.d), dtype=torch.bfloat16, device=dev)
        ov = torch.empty_like(ok_)
        wq = bca.new_workspace(dq, bca.OP_COMMIT, device=dev)
        ms_q = time_calls(lambda: bca.bca_qkv_post(dq, tq["qkv"], tq["pos"], oq, ok_, ov, wq,
                                                   q_norm_w=tq["qw"], k_norm_w=tq["kw"], eps=1e-6,
                                                   rope_theta=1e6, write_pos=tq["wp"],
                                                   k_pool=tq["kp"], v_pool=tq["vp"],
                                                   page_table=tq["pt"]), reps(50))
        tokens = cq.B * cq.n
        row = (cq.Hq + 2 * cq.Hkv) * cq.d * 2.0
        bytes_q = tokens * (2 * row + 2 * cq.Hkv * cq.d * 2.0 + 8.0) + 2 * cq.d * 2.0
        res["qkv_post"] = with_kernel(
            dict(roof(0.0, bytes_q, ms_q), kernel_us=dict(time_calls.kernel_us),
                 workload=f"batch {cq.B} x 64 tokens after the serving prefixes, 32/8 heads, "
                          "d=128: per-head RMS norms + RoPE (theta 1e6) of q and k, "
                          "K/V rows written to pages of 16"), 0.0, bytes_q, "qkv_post")
        del tq, oq, ok_, ov, wq, cq

    if want("block_decode"):
        # block decode: batch 8, 64-token blocks after prefixes uniform in
        # {512, 576, ..., 4096}, 32/8 heads, d = 128 (K/V ~ 75 MB: L2-sized,
        # hence the flush before every call)
        cb = workloads.block_decode(seed=args.seed, keep_logical=False)
        db = bca.dims(cb.B, cb.D, cb.Hq, cb.Hkv, cb.d, cb.pool.page_size, cb.pool.num_pages,
                      cb.pool.max_pages_per_seq)
        tb = {"q": cb.q.to(dev), "k": cb.k_blk.to(dev), "v": cb.v_blk.to(dev),
              "kp": cb.pool.k_pool.to(dev), "vp": cb.pool.v_pool.to(dev),
              "pt": cb.pool.page_table.to(dev),
              "pl": torch.tensor(cb.prefix_len, dtype=torch.int32, device=dev)}
        ob = torch.empty_like(tb["q"])
        wb = bca.new_workspace(db, bca.OP_DECODE, device=dev)
        ms_b = time_calls(lambda: bca.bca_decode(db, tb["q"], tb["k"], tb["v"], tb["kp"], tb["vp"],
                                                 tb["pt"], tb["pl"], ob, False, wb), reps(50))
        Pb = cb.prefix_len
        pairs_b = sum((p_ + cb.D) * cb.D for p_ in Pb)
        flops_b = 4.0 * cb.d * cb.Hq * pairs_b
        bytes_b = (sum(Pb) * 2 * cb.Hkv * cb.d * 2.0 + cb.B * cb.D * (2 * cb.Hq + 2 * cb.Hkv) * cb.d * 2.0
                   + cb.B * cb.pool.max_pages_per_seq * 4.0)
        res["block_decode"] = with_kernel(
            dict(roof(flops_b, bytes_b, ms_b), kernel_us=dict(time_calls.kernel_us),
                 workload=f"batch 8, D=64 after prefixes uniform in {{512..4096}} (sum {sum(Pb)}), "
                          "32/8 heads, d=128, page 16"), flops_b, bytes_b, "attention")
        del tb, ob, wb, cb

    if want("extend"):
        # short causal extend: batch 64, 9 new tokens (2N-1, N = 5), prefixes at
        # token granularity, 32/8 heads, d = 128, the new rows committed
        P = workloads.prefix_loguniform_blocks(args.row_batch, 128, 32768, 1, seed=args.seed)
        n = 9
        ce = workloads.make_decode_case(P, D=n, Hq=32, Hkv=8, d=128, seed=args.seed,
                                        keep_logical=False)
        de = bca.dims(ce.B, n, ce.Hq, ce.Hkv, ce.d, ce.pool.page_size, ce.pool.num_pages,
                      ce.pool.max_pages_per_seq)
        te = {"q": ce.q.to(dev), "k": ce.k_blk.to(dev), "v": ce.v_blk.to(dev),
              "kp": ce.pool.k_pool.to(dev), "vp": ce.pool.v_pool.to(dev),
              "pt": ce.pool.page_table.to(dev),
              "pl": torch.tensor(P, dtype=torch.int32, device=dev)}
        oe = torch.empty_like(te["q"])
        we = bca.new_workspace(de, bca.OP_DECODE, device=dev)
        ms_e = time_calls(lambda: bca.bca_extend(de, te["q"], te["k"], te["v"], te["kp"], te["vp"],
                                                 te["pt"], te["pl"], oe, True, we), reps(20))
        pairs_e = sum(p_ * n + n * (n + 1) // 2 for p_ in P)
        flops_e = 4.0 * ce.d * ce.Hq * pairs_e
        kv_row = 2 * ce.Hkv * ce.d * 2.0  # K and V bytes of one token
        bytes_e = (sum(P) * kv_row + ce.B * n * (2 * ce.Hq * ce.d * 2.0 + 2 * kv_row)
                   + ce.B * ce.pool.max_pages_per_seq * 4.0)
        res["extend"] = with_kernel(
            dict(roof(flops_e, bytes_e, ms_e), kernel_us=dict(time_calls.kernel_us),
                 workload=f"batch {ce.B}, 9 new causal tokens after log-uniform prefixes in "
                          f"[128, 32768] (sum {sum(P)}), 32/8 heads, d=128, page 16, "
                          f"new rows committed"), flops_e, bytes_e, "attention")
        del te, oe, we, ce

    if want("multicanvas"):
        mc(workloads.multicanvas_b16(seed=args.seed), 0, "multicanvas",
           "batch 16, prompt 1024, 3 canvases of 256 with 30-100% live rows, 32/8 heads, d=128")
    if want("multicanvas_window"):
        mc(workloads.make_multicanvas_case(16, 1024, 5, 256, 32, 8, 128, seed=args.seed), 1024,
           "multicanvas_window", "as above with 5 canvases under a 1024-token sliding window")
    return res


def run_ours(args):
    import torch
    import torch.distributed as dist
    import block_causal_paged_gb300 as bca
    import workloads

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    bca.load()
    stream = torch.cuda.current_stream()
    pk = peaks()

    def barrier():
        if world > 1:
            dist.barrier()

    if args.only:
        rows = other_rows(args, bca, workloads, torch, pk, dev, stream)
        if rank == 0:
            print(json.dumps({"only": args.only, "other_rows": rows}), flush=True)
        if world > 1:
            dist.destroy_process_group()
        return 0

    def build_case(D, seed):
        # each rank runs its own batch (weak scaling): seed offset by rank
        case = workloads.serving_decode(seed=rank_seed(seed, rank), D=D, B=args.batch,
                                        keep_logical=False)
        S = case.pool.page_size
        dd = bca.dims(case.B, D, case.Hq, case.Hkv, case.d, S, case.pool.num_pages,
                      case.pool.max_pages_per_seq)
        t = dict(q=case.q.to(dev), kb=case.k_blk.to(dev), vb=case.v_blk.to(dev),
                 kp=case.pool.k_pool.to(dev), vp=case.pool.v_pool.to(dev),
                 pt=case.pool.page_table.to(dev),
                 pl=torch.tensor(case.prefix_len, dtype=torch.int32, device=dev))
        t["out"] = torch.empty_like(t["q"])
        t["ws"] = bca.new_workspace(dd, bca.OP_DECODE, device=dev)
        return case, dd, t

    def step_fn(dd, t):
        return lambda: bca.bca_decode(dd, t["q"], t["kb"], t["vb"], t["kp"], t["vp"], t["pt"],
                                      t["pl"], t["out"], True, t["ws"])

    def measure(D, steps, warmup, with_clocks, seed=args.seed):
        case, dd, t = build_case(D, seed)
        step = step_fn(dd, t)
        for _ in range(warmup):
            step()
        torch.cuda.synchronize()
        st = bca.read_device_status(t["ws"])
        if st != 0:
            raise RuntimeError(f"device status after warm-up: {bca.status_string(st)}")
        sampler = ClockSampler(local) if with_clocks else None
        if sampler:
            sampler.start()
            time.sleep(0.3)
        barrier()
        t0 = time.time()
        ms = time_steps(torch, step, steps, stream)
        t1 = time.time()
        barrier()
        clocks = None
        if sampler:
            time.sleep(0.15)
            sampler.stop()
            clocks = sampler.summary(t0, t1)
        # per-kernel device time, CUDA events on the launch stream (separate pass)
        bca.profile_start(steps * 4 + 16)
        for _ in range(steps):
            step()
        torch.cuda.synchronize()
        prof = bca.profile_stop()
        alg = algorithmic(case.prefix_len, D, case.Hq, case.Hkv, case.d, case.pool.page_size)
        return case, dd, t, ms / steps, clocks, prof, alg

    case, dd, t, ms_step, clocks, prof, alg = measure(args.D, args.steps, args.warmup, True)
    ms_max = max_over_ranks(ms_step, dev)
    value = job_throughput_tflops(alg["flops"], world, ms_max)

    traffic, traffic_src = committed_traffic(args.batch, args.D)
    if args.traffic is not None:
        traffic, traffic_src = args.traffic, "--traffic"
    attn_n, attn_ms = prof["attention"]
    attn_avg_ms = attn_ms / max(1, attn_n)
    # the attention kernel's own bytes (the commit runs in the epilogue kernel)
    kern_bytes = alg["attn_bytes"]
    achieved_gbs = kern_bytes / (attn_avg_ms * 1e-3) / 1e9
    achieved_tflops = alg["flops"] / (attn_avg_ms * 1e-3) / 1e12
    t_mem = kern_bytes / (pk["hbm_gbs"] * 1e9)
    t_flop = alg["flops"] / (pk["bf16_tflops"] * 1e12)
    bound = "hbm" if t_mem >= t_flop else "tensor"
    roofline = {
        "kernel": "attention_pair_kernel (bca_decode main kernel: CTA pairs, tcgen05 cta_group::2)",
        "bound": bound,
        "achieved": achieved_gbs if bound == "hbm" else achieved_tflops,
        "peak": pk["hbm_gbs"] if bound == "hbm" else pk["bf16_tflops"],
        "unit": "GB/s" if bound == "hbm" else "TFLOP/s",
        "frac": (achieved_gbs / pk["hbm_gbs"]) if bound == "hbm" else (achieved_tflops / pk["bf16_tflops"]),
        "traffic": traffic,
        "traffic_source": traffic_src,
        "peak_source": f"{pk['source']} (MEASURED_PEAKS.json hbm_gbs / bf16_tflops burst)"
                       if pk["source"] == "measured" else "fallback",
        "kernel_us": attn_avg_ms * 1e3,
        "algorithmic_bytes": kern_bytes,
        "algorithmic_flops": alg["flops"],
        "tensor_frac": achieved_tflops / pk["bf16_tflops"],
        "step_roofline_frac": max(alg["step_bytes"] / (pk["hbm_gbs"] * 1e9),
                                  alg["flops"] / (pk["bf16_tflops"] * 1e12)) / (ms_max * 1e-3),
    }
    launches_per_step = sum(n for n, _ in prof.values()) / max(1, args.steps)

    # end to end through the public API with pinned host buffers: every step
    # copies its inputs (block q/k/v, page table, prefix lengths) in from the
    # host, runs bca_decode (attention + commit) and reads its output back.
    # Serving steps are pipelined over two device staging sets: the copy-in of
    # step i+1 (its own stream) and the read-back of step i-1 (another) run
    # while the kernels of step i do; a staging set is overwritten only after
    # the step that used it has finished with it (events).
    keys = ("q", "kb", "vb", "pt", "pl")
    h = {k: t[k].cpu().pin_memory() for k in keys}
    h_out = [torch.empty(t["out"].shape, dtype=t["out"].dtype).pin_memory() for _ in range(2)]
    h2d = sum(x.numel() * x.element_size() for x in h.values())
    d2h = h_out[0].numel() * h_out[0].element_size()
    stage = [{k: t[k] for k in keys + ("out",)},
             {k: torch.empty_like(t[k]) for k in keys + ("out",)}]
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_dec = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]
    e2e_i = [0]

    def e2e_step():
        s = e2e_i[0] % 2
        e2e_i[0] += 1
        st = stage[s]
        s_in.wait_event(ev_dec[s])          # the step that last read this set is done
        with torch.cuda.stream(s_in):
            for k in keys:
                st[k].copy_(h[k], non_blocking=True)
        ev_in[s].record(s_in)
        stream.wait_event(ev_in[s])
        stream.wait_event(ev_out[s])        # this set's previous output has been read back
        bca.bca_decode(dd, st["q"], st["kb"], st["vb"], t["kp"], t["vp"], st["pt"], st["pl"],
                       st["out"], True, t["ws"], stream=stream)
        ev_dec[s].record(stream)
        s_out.wait_event(ev_dec[s])
        with torch.cuda.stream(s_out):
            h_out[s].copy_(st["out"], non_blocking=True)
        ev_out[s].record(s_out)

    def e2e_serial_step():
        for k in keys:
            t[k].copy_(h[k], non_blocking=True)
        bca.bca_decode(dd, t["q"], t["kb"], t["vb"], t["kp"], t["vp"], t["pt"], t["pl"],
                       t["out"], True, t["ws"])
        h_out[0].copy_(t["out"], non_blocking=True)

    def time_pipelined(n):
        # the copy streams start after the start event and the end event
        # follows the last read-back
        start = torch.cuda.Event(enable_timing=True)
        end = torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        start.record(stream)
        s_in.wait_stream(stream)
        s_out.wait_stream(stream)
        for _ in range(n):
            e2e_step()
        stream.wait_stream(s_out)
        end.record(stream)
        torch.cuda.synchronize()
        return start.elapsed_time(end)

    # (the serial steps reuse staging set 0: never in flight together)
    for _ in range(max(3, args.warmup // 4)):
        e2e_step()
    torch.cuda.synchronize()
    for _ in range(max(3, args.warmup // 4)):
        e2e_serial_step()
    torch.cuda.synchronize()
    e2e_steps = max(10, args.steps // 4)
    barrier()
    e2e_ms = time_pipelined(e2e_steps) / e2e_steps
    e2e_serial_ms = time_steps(torch, e2e_serial_step, e2e_steps, stream) / e2e_steps
    e2e_ms_max = max_over_ranks(e2e_ms, dev)
    e2e_serial_ms_max = max_over_ranks(e2e_serial_ms, dev)
    e2e_value = job_throughput_tflops(alg["flops"], world, e2e_ms_max)
    # the outputs read back by the pipelined (set 1) and serial (set 0) steps
    # against the device output of the last step (same inputs every step)
    e2e_outputs_equal = bool(torch.equal(h_out[0], t["out"].cpu()) and
                             torch.equal(h_out[1], t["out"].cpu()))
    st = bca.read_device_status(t["ws"])
    del t, case

    # confidence of the top prediction at every position of the step's blocks
    # (softmax-plus-argmax over a 262144-token vocabulary, bf16 logits)
    conf_line = None
    if not args.no_sweep:
        rows, vocab = args.batch * args.D, 262144
        lg = workloads.confidence_logits(rows, vocab, seed=args.seed + rank, device=dev)
        c_arg = torch.empty(rows, dtype=torch.int32, device=dev)
        c_conf = torch.empty(rows, dtype=torch.float32, device=dev)
        for _ in range(3):
            bca.bca_confidence(lg, c_arg, c_conf)
        c_steps = max(10, args.steps // 20)
        c_ms = time_steps(torch, lambda: bca.bca_confidence(lg, c_arg, c_conf), c_steps, stream) / c_steps
        c_bytes = rows * vocab * lg.element_size() + rows * 8
        conf_line = {"rows": rows, "vocab": vocab, "dtype": "bf16", "us": c_ms * 1e3,
                     "gbs": c_bytes / (c_ms * 1e-3) / 1e9,
                     "frac": c_bytes / (c_ms * 1e-3) / 1e9 / pk["hbm_gbs"], "bound": "hbm",
                     "algorithmic_bytes": c_bytes}
        del lg
    rows_line = other_rows(args, bca, workloads, torch, pk, dev, stream) if not args.no_sweep else None

    # the headline step on two more seeded batches (prefix lengths differ)
    seeds = [{"seed": args.seed, "us_per_step": ms_max * 1e3, "attn_us": attn_avg_ms * 1e3,
              "attn_hbm_frac": roofline["frac"],
              "step_roofline_frac": roofline["step_roofline_frac"], "sum_prefix": alg["sum_prefix"]}]
    if not args.no_sweep:
        for sd in (args.seed + 1, args.seed + 2):
            c3, _, t3, ms3, _, prof3, alg3 = measure(args.D, max(20, args.steps // 4),
                                                     max(3, args.warmup), False, seed=sd)
            n3, tot3 = prof3["attention"]
            a3 = tot3 / max(1, n3)
            seeds.append({"seed": sd, "us_per_step": ms3 * 1e3, "attn_us": a3 * 1e3,
                          "attn_hbm_frac": alg3["attn_bytes"] / (a3 * 1e-3) / 1e9 / pk["hbm_gbs"],
                          "step_roofline_frac": max(alg3["step_bytes"] / (pk["hbm_gbs"] * 1e9),
                                                    alg3["flops"] / (pk["bf16_tflops"] * 1e12))
                                                / (ms3 * 1e-3),
                          "sum_prefix": alg3["sum_prefix"]})
            del t3, c3

    sweep = []
    if not args.no_sweep:
        for D2 in (32, 64):
            if D2 == args.D:
                sweep.append({"D": D2, "us_per_step": ms_max * 1e3, "tflops": value / world,
                              "attn_us": attn_avg_ms * 1e3, "attn_hbm_frac": roofline["frac"]})
                continue
            c2, _, t2, ms2, _, prof2, alg2 = measure(D2, max(20, args.steps // 2),
                                                     max(3, args.warmup), False)
            n2, tot2 = prof2["attention"]
            a2 = tot2 / max(1, n2)
            sweep.append({"D": D2, "us_per_step": ms2 * 1e3,
                          "tflops": alg2["flops"] / (ms2 * 1e-3) / 1e12, "attn_us": a2 * 1e3,
                          "attn_hbm_frac": alg2["attn_bytes"] / (a2 * 1e-3) / 1e9 / pk["hbm_gbs"],
                          "sum_prefix": alg2["sum_prefix"]})
            del t2, c2

    if rank == 0:
        prefix_len = workloads.prefix_loguniform_blocks(args.batch, 128, 32768, 64, args.seed)
        cpu = None if args.no_cpu_baseline else cpu_baseline(args.seed, prefix_len, args.D, 32, 8,
                                                             128)
        line = {"metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_max,
                "us_per_step": ms_max * 1e3, "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
                "config": workload_config(args, prefix_len),
                "hbm_gbs": alg["step_bytes"] / (ms_max * 1e-3) / 1e9,
                "roofline": roofline, "cpu_baseline": cpu,
                "e2e": {"value": e2e_value, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
                        "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms_max,
                        "pipelining": "copy-in of step i+1 and read-back of step i-1 overlap "
                                      "step i's kernels (two staging sets, two copy streams)",
                        "serial_ms_per_step": e2e_serial_ms_max,
                        "serial_value": job_throughput_tflops(alg["flops"], world, e2e_serial_ms_max),
                        "outputs_equal": e2e_outputs_equal},
                "gpu_launches": int(round(launches_per_step * args.steps)),
                "launches_per_step": launches_per_step,
                "kernel_ms": {k: (v[1] / v[0] if v[0] else None) for k, v in prof.items()},
                "clocks": clocks, "device_status": st, "seeds": seeds, "sweep": sweep,
                "confidence": conf_line,
                "other_rows": rows_line}
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--D", type=int, default=64, choices=[32, 64])
    ap.add_argument("--batch", type=int, default=64,
                    help="sequences per GPU (64 is the benchmarked configuration; smaller "
                         "batches are for profiler captures)")
    ap.add_argument("--no-sweep", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--only", default=None,
                    help="run only these secondary rows (comma list of prefill, qkv_post, block_decode, "
                         "extend, multicanvas, multicanvas_window) and print them; for profiler captures")
    ap.add_argument("--row-reps", type=int, default=0,
                    help="timed calls per secondary row (0: the row's default)")
    ap.add_argument("--row-batch", type=int, default=64,
                    help="sequences of the QKV-post and extend rows (64 is the benchmarked size)")
    ap.add_argument("--traffic", type=float, default=None,
                    help="DRAM bytes per attention launch from an ncu capture (reported as is)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())

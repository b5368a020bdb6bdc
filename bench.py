#!/usr/bin/env python
"""Throughput of the CSA2 decode step on one GB300 (one process per GPU).

Default workload (N=1): Full-layer decode, batch 32, context 65,536 per
sequence, 64 query heads, 64 indexer heads x 128, top-512, 8-bit window.
One step = the whole hot path for that layer on one batch: append the step's
token (RoPE + quantise into the FP4 cache and the window), score every visible
position, select the top 512 and build the 2,048-block candidate pool, attend
over the selected entries plus the window.  Inputs are seeded synthetic data
(N(0,1) KV and queries, U(0,1) head weights) resident in HBM before timing.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

Prints one JSON line (rank 0).  --impl reference times the CPU oracle on a
bounded sample of the same workload on the host cores.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

METRIC = "decode tokens/s and KV HBM GB/s (% of roofline) at 64K-1M context, 1 GB300"
UNIT = "tokens/s"
PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")
FALLBACK_HBM_GBS = 6800.0


# ----------------------------------------------------------------------------- helpers
def peaks():
    try:
        with open(PEAKS_FILE) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def score_traffic(workload):
    """dram read + write bytes per launch of the score kernel from the committed ncu
    summary of the B 32 x 65,536 decode workload, or None for another workload or
    when the kernel source has changed since that capture."""
    if workload != "full_decode_b32_t65536":
        return None
    import hashlib
    here = os.path.dirname(os.path.abspath(__file__))
    prof = os.path.join(here, "profiles", "index_score_tc_full_decode_b32_t65536.md")
    src = os.path.join(here, "fp4_compressed_sparse_gb300", "csrc", "csa2_score_tc.cu")
    try:
        text = open(prof).read()
        sha = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
        rec = dict(line.split(": ", 1) for line in text.splitlines() if line.startswith(("source_sha256:", "traffic_bytes")))
        if rec.get("source_sha256", "").strip() != sha:
            return None
        return int(rec["traffic_bytes_per_launch"])
    except Exception:
        return None


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def replica_seed(seed, rank):
    """Weak scaling: every rank runs its own batch of independent sequences."""
    return seed + 1000 * rank


def aggregate_ranks(total_ms, batch, steps, world, device):
    """Whole-job figures of a replicas-only run: the slowest rank's timed total (max
    over ranks) and the tokens all ranks processed in it.  Returns (total_ms,
    tokens per second)."""
    if world > 1:
        t = torch.tensor([total_ms], dtype=torch.float64, device=device)
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        total_ms = float(t.item())
    return total_ms, batch * world * steps / (total_ms / 1e3)


class ClockSampler:
    """SM clock, power and clock-event reasons sampled through NVML (the driver's
    libnvidia-ml, read-only queries) by a thread polling every ~2 ms, so that
    samples fall inside even a short timed region; mark() brackets that region.
    Falls back to `nvidia-smi -lms 100` when NVML cannot be loaded."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    # nvmlClocksEventReason bits
    BITS = {"sw_power_cap": 0x4, "hw_slowdown": 0x8, "sw_thermal_slowdown": 0x20,
            "hw_thermal_slowdown": 0x40, "hw_power_brake_slowdown": 0x80}

    def __init__(self, device):
        self.device = device
        self.samples = []
        self.region = None
        self.proc = None
        self.thread = None
        self.stop_flag = False

    def _nvml(self):
        import ctypes
        lib = ctypes.CDLL("libnvidia-ml.so.1")
        if lib.nvmlInit_v2() != 0:
            raise RuntimeError("nvmlInit failed")
        h = ctypes.c_void_p()
        uuid = "GPU-" + str(torch.cuda.get_device_properties(self.device).uuid)
        if lib.nvmlDeviceGetHandleByUUID(uuid.encode(), ctypes.byref(h)) != 0:
            raise RuntimeError("no NVML handle for " + uuid)
        reasons_fn = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            lib.nvmlDeviceGetCurrentClocksThrottleReasons
        mx = ctypes.c_uint()
        lib.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx))  # NVML_CLOCK_SM
        return lib, h, reasons_fn, float(mx.value)

    def _poll(self, lib, h, reasons_fn):
        import ctypes
        clk, pw, rs = ctypes.c_uint(), ctypes.c_uint(), ctypes.c_ulonglong()
        while not self.stop_flag:
            if lib.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(clk)) == 0 and \
                    reasons_fn(h, ctypes.byref(rs)) == 0:
                lib.nvmlDeviceGetPowerUsage(h, ctypes.byref(pw))
                self.samples.append((time.perf_counter(), float(clk.value), int(rs.value), pw.value / 1e3))
            time.sleep(0.002)

    def start(self):
        try:
            lib, h, reasons_fn, self.smax = self._nvml()
            self.thread = threading.Thread(target=self._poll, args=(lib, h, reasons_fn), daemon=True)
            self.thread.start()
            self.source = "nvml"
        except Exception:
            self._start_smi()
        self.old_switch = sys.getswitchinterval()
        sys.setswitchinterval(0.0005)  # let the poller run between the replay calls
        time.sleep(0.05)

    def _start_smi(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.device}", f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
            self.source = "nvidia-smi"
        except Exception:
            self.proc = None
            self.source = None

    def mark(self, t0, t1):
        self.region = (t0, t1)

    def stop(self):
        sys.setswitchinterval(self.old_switch)
        if self.thread is not None:
            time.sleep(0.01)
            self.stop_flag = True
            self.thread.join(timeout=2)
            t0, t1 = self.region
            inside = [x for x in self.samples if t0 <= x[0] <= t1]
            if not inside:
                return None
            reasons = sorted(n for n, bit in self.BITS.items() if any(x[2] & bit for x in inside))
            return {"sm_mhz": statistics.median(x[1] for x in inside), "sm_max_mhz": self.smax,
                    "reasons": reasons, "samples": len(inside), "source": "nvml, during the timed region",
                    "power_w_max": max(x[3] for x in inside)}
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax = float(parts[2])
                except ValueError:
                    continue
                for n, v in zip(names, parts[5:9]):
                    if v.lower() == "active":
                        reasons.add(n)
        os.unlink(self.path)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": smax, "reasons": sorted(reasons),
                "samples": len(sm), "source": "nvidia-smi, around the timed region"}


class L2Flush:
    """Evicts the 129 MB L2 between timed steps: a 256 MB buffer is written, then
    read back, so the flush's own dirty lines are written to HBM before the timed
    region starts (otherwise the next step pays for ~129 MB of write-backs)."""

    DESCRIPTION = "flushed between timed steps (256 MB written, then read back; outside the timed region)"

    def __init__(self, dev):
        self.buf = torch.empty(256 << 20, dtype=torch.uint8, device=dev)

    def __call__(self):
        self.buf.zero_()
        self.buf.view(torch.int32).sum()


# ----------------------------------------------------------------------------- workload
def decode_step_bytes(B, T, H, H_I, k, swa_dtype):
    """Algorithmic HBM bytes of one Full-layer decode step (what the method must move)."""
    keys = B * T * 68                                  # indexer keys of every visible position
    qidx = B * (H_I * 128 * 2 + 4 * H_I)               # indexer query (bf16) + head weights
    sel = B * k * (324 + 4)                            # selected entries (288 + 36 sidecar) + index
    swa = B * 128 * (594 if swa_dtype == 1 else 1152)  # window entries
    q = B * H * 576 * 2                                # absorbed query
    out = B * H * 512 * 4 + B * H * 4                  # output + lse
    append = B * ((576 + 128) * 4 + 324 + 68 + (594 if swa_dtype == 1 else 1152))
    return {"keys": keys, "qidx": qidx, "attn": sel + swa + q + out, "append": append,
            "total": keys + qidx + sel + swa + q + out + append}


class FullDecode:
    """Full-layer decode on a batch: caches built through csa2_kv_append."""

    def __init__(self, W, n_steps, device, page_entries=None, entry_format=0):
        from fp4_compressed_sparse_gb300 import csa2
        self.csa2 = csa2
        self.W = W
        B, ctx = W.batch, W.context
        self.cap = ctx + n_steps + 8
        if page_entries:
            # paged: the sequences' pages spread over the pool in a seeded random order
            self.cap = -(-self.cap // page_entries) * page_entries
            max_pages = self.cap // page_entries
            g = torch.Generator().manual_seed(W.seed + 77)
            table = torch.randperm(B * max_pages, generator=g).to(torch.int32).view(B, max_pages)
            self.cache = csa2.Cache(B, self.cap, ratio=1, swa_dtype=W.swa_dtype, page_entries=page_entries,
                                    block_table=table, entry_format=entry_format)
        else:
            self.cache = csa2.Cache(B, self.cap, ratio=1, swa_dtype=W.swa_dtype, entry_format=entry_format)
        self.rope = csa2.rope_table(W.theta, self.cap + 8)
        self.err = torch.zeros(1, dtype=torch.int32, device=device)
        chunk = 8192
        for t0 in range(0, ctx, chunk):
            n = min(chunk, ctx - t0)
            kv = torch.stack([W.kv(b, t0, n, device=device) for b in range(B)])
            ik = torch.stack([W.ik(b, t0, n, device=device) for b in range(B)])
            csa2.kv_append(self.cache, kv, ik, self.rope, err=self.err)
            del kv, ik
        torch.cuda.synchronize()
        # per-step inputs (resident in HBM)
        self.kv_new = [torch.stack([W.kv(b, ctx + s, 1, device=device) for b in range(B)])
                       for s in range(n_steps)]
        self.ik_new = [torch.stack([W.ik(b, ctx + s, 1, device=device) for b in range(B)])
                       for s in range(n_steps)]
        self.q_idx = [W.q_idx(s, 0, device=device) for s in range(n_steps)]
        self.w = [W.w(s, 0, device=device) for s in range(n_steps)]
        self.q = [W.q(s, 0, device=device) for s in range(n_steps)]
        self.q_pos = [torch.full((B,), ctx + s, dtype=torch.int64, device=device) for s in range(n_steps)]
        self.scores = torch.empty((B, self.cap), device=device)
        self.idx = torch.empty((B, W.topk), dtype=torch.int32, device=device)
        self.pool = torch.empty((B, W.pool_blocks), dtype=torch.int32, device=device)
        self.pool_cnt = torch.empty((B,), dtype=torch.int32, device=device)
        self.out = torch.empty((B, W.heads, 512), device=device)
        self.lse = torch.empty((B, W.heads), device=device)
        self.ws_topk = csa2.topk_workspace(B, self.cap, W.topk, W.pool_blocks)
        self.ws_attn = csa2.attn_workspace(B, W.heads, W.topk)
        self.ws_score = csa2.index_score_workspace(B, W.index_heads)
        self.aux = csa2.score_aux(B, self.cap)
        self.side = torch.cuda.Stream(device=device)
        self.launches_per_step = None

    PARTS = ("append", "score", "topk_pool", "attention")

    def part(self, s, name):
        c, W = self.csa2, self.W
        if name == "append":
            c.kv_append(self.cache, self.kv_new[s], self.ik_new[s], self.rope, err=self.err)
        elif name == "score":
            c.index_score(self.cache, self.q_idx[s], self.w[s], self.q_pos[s], self.scores, err=self.err,
                          ws=self.ws_score, aux=self.aux)
        elif name == "topk_pool":
            c.topk(self.scores, 1, self.q_pos[s], W.topk, self.idx, self.ws_topk, pool_out=self.pool,
                   pool_count=self.pool_cnt, err=self.err, aux=self.aux)
        else:
            c.sparse_attn_decode(self.cache, self.q[s], self.q_pos[s], self.idx, self.out, self.lse,
                                 self.ws_attn, W.sm_scale, err=self.err)

    def step(self, s, ev=None):
        """One decode step.  The append runs on a side stream, concurrently with
        the score and the top-k (neither reads the new token: a query at position
        t sees entries < t); the attention waits for it (window slot, n_tokens)."""
        if ev is not None:  # sequential, with an event between parts (diagnostics)
            for k, name in enumerate(self.PARTS):
                ev[k].record()
                self.part(s, name)
            ev[len(self.PARTS)].record()
            return
        main = torch.cuda.current_stream()
        fork, join = torch.cuda.Event(), torch.cuda.Event()
        fork.record(main)
        self.side.wait_event(fork)
        with torch.cuda.stream(self.side):
            self.part(s, "append")
        join.record(self.side)
        self.part(s, "score")
        self.part(s, "topk_pool")
        main.wait_event(join)
        self.part(s, "attention")

    @staticmethod
    def kernel_launches():
        # kv_append ratio 1, one token: 1 (it also advances n_tokens); index_score: query
        # prep (it also clears the sideband histograms) + score; topk: 1 fused selector
        # (top-k and pool); attention: 1 (the splits of a row merge inside)
        return 1 + 2 + 1 + 1


# ----------------------------------------------------------------------------- our arm
def run_ours(args):
    from fp4_compressed_sparse_gb300 import build_lib, csa2
    from fp4_compressed_sparse_gb300 import workloads as wl

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    build_lib.build()
    csa2.load()
    W = getattr(wl, args.workload)(device="cuda")
    # weak scaling: every rank runs its own batch (independent sequences), seeds offset by rank
    W.seed = replica_seed(W.seed, rank)
    n_steps = args.warmup + args.steps + args.e2e_steps
    bench = FullDecode(W, n_steps, dev)
    flush = L2Flush(dev)

    # warm-up steps run eagerly (first calls set kernel attributes)
    for s in range(args.warmup):
        flush()
        bench.step(s)
    torch.cuda.synchronize()
    if bench.err.item() != 0:
        raise RuntimeError(f"device error word {bench.err.item()} during warm-up")
    # every timed step is one CUDA graph (append on a forked branch)
    graphs = None
    if not args.no_graph:
        graphs = []
        for i in range(args.steps):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                bench.step(args.warmup + i)
            graphs.append(g)
        torch.cuda.synchronize()
    ev0 = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ev1 = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    sampler = ClockSampler(local)
    sampler.start()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    t_begin = time.perf_counter()
    for i in range(args.steps):
        flush()  # L2 flushed between timed steps (outside the events)
        ev0[i].record()
        if graphs is not None:
            graphs[i].replay()
        else:
            bench.step(args.warmup + i)
        ev1[i].record()
    torch.cuda.synchronize()
    sampler.mark(t_begin, time.perf_counter())
    if world > 1:
        torch.distributed.barrier()
    clocks = sampler.stop()
    if bench.err.item() != 0:
        raise RuntimeError(f"device error word {bench.err.item()} in the timed steps")
    step_ms = [a.elapsed_time(b) for a, b in zip(ev0, ev1)]
    total_ms, value = aggregate_ranks(sum(step_ms), W.batch, args.steps, world, dev)
    ms_per_step = total_ms / args.steps

    # second timed pass, same steps' inputs: each part as its own graph with
    # events between (score, top-k, attention do not change the cache), for the
    # per-part breakdown and the dominant kernel's launch duration
    part_names = ("score", "topk_pool", "attention")
    parts = {n: [] for n in part_names}
    pgraphs = []
    for i in range(args.steps):
        row = []
        for n in part_names:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                bench.part(args.warmup + i, n)
            row.append(g)
        pgraphs.append(row)
    pev = [[torch.cuda.Event(enable_timing=True) for _ in range(len(part_names) + 1)] for _ in range(args.steps)]
    torch.cuda.synchronize()
    for i in range(args.steps):
        flush()
        for k, g in enumerate(pgraphs[i]):
            pev[i][k].record()
            g.replay()
        pev[i][-1].record()
    torch.cuda.synchronize()
    for i in range(args.steps):
        for k, n in enumerate(part_names):
            parts[n].append(pev[i][k].elapsed_time(pev[i][k + 1]))
    del pgraphs
    score_ms = parts["score"]

    hbm, hbm_kind = peaks()
    T = W.context + args.warmup + args.steps // 2
    nbytes = decode_step_bytes(W.batch, T, W.heads, W.index_heads, W.topk, W.swa_dtype)
    kv_gbs = nbytes["total"] / (ms_per_step / 1e3) / 1e9
    score_avg = statistics.mean(score_ms)
    score_bytes = nbytes["keys"] + nbytes["qidx"]
    achieved = score_bytes / (score_avg / 1e3) / 1e9

    # end to end through the public API: host inputs (pinned) -> device, step, result -> host
    e2e = None
    if args.e2e_steps > 0:
        e2e = run_e2e(bench, W, args, dev, flush)

    line = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "fp4/bf16/fp32",
        "data": "synthetic (seeded N(0,1) KV/queries, U(0,1) head weights)",
        "config": {"workload": W.name, "batch": W.batch, "context": W.context, "heads": W.heads,
                   "index_heads": W.index_heads, "topk": W.topk, "window": 128,
                   "window_dtype": "mxfp8" if W.swa_dtype == 1 else "bf16",
                   "pool_blocks": W.pool_blocks, "l2": L2Flush.DESCRIPTION,
                   "launch": "eager" if args.no_graph else "one CUDA graph per step (append on a forked branch)",
                   "parallelism": f"replicas x{world} (sequences sharded, no collective)"},
        "kv_hbm": {"algorithmic_bytes_per_step": nbytes["total"], "gbs": round(kv_gbs, 1),
                   "frac": round(kv_gbs / hbm, 4), "peak_gbs": hbm, "peak_kind": hbm_kind},
        "roofline": {"kernel": "index_score (Full scan: query prep + tensor-core score + sideband)", "bound": "hbm",
                     "achieved": round(achieved, 1),
                     "peak": hbm, "unit": "GB/s", "frac": round(achieved / hbm, 4), "traffic": score_traffic(W.name),
                     "algorithmic_bytes_per_launch": score_bytes, "avg_launch_ms": round(score_avg, 5),
                     "peak_kind": hbm_kind},
        "step_breakdown_ms": {k: round(statistics.mean(v), 5) for k, v in parts.items()},
        "step_breakdown_note": "score / topk_pool / attention replayed one part per graph over the timed "
                               "steps' inputs; the append overlaps them inside each timed step",
        "gpu_launches": FullDecode.kernel_launches() * args.steps,
        "clocks": clocks,
    }
    if e2e:
        line["e2e"] = e2e
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(W, args)
    if rank == 0 and args.workload == "full_decode" and not args.headline_only:
        # the metric's other context lengths and the prefill indexer, measured in
        # the same run: the 1 M-context decoder group (config of 8 sequences x
        # 1,048,576 tokens) and the chunked prefill, with the FP4 tensor peak
        del bench, graphs
        torch.cuda.empty_cache()
        # the same step on a paged cache (256-entry pages in shuffled order)
        line["paged"] = measure_paged(W, max(10, min(args.steps, 30)), 3, dev, 256)
        torch.cuda.empty_cache()
        # the V4 cache formats at the same configuration
        line["formats"] = measure_formats(W, max(10, min(args.steps, 30)), 3, dev)
        torch.cuda.empty_cache()
        fp4 = measure_fp4_peak(dev)
        line["fp4_peak"] = fp4
        line["stack_1m"] = measure_group(wl.stack_1m(device="cuda"), max(10, min(args.steps, 20)), 3, dev)
        torch.cuda.empty_cache()
        # the 256 K Reindex + 3 Reuse group, then the same group with its Reindex
        # layer in the published reference code's form (every position scored,
        # the rest of the row masked)
        line["reindex_256k"] = measure_group(wl.reindex_decode(device="cuda"), max(10, min(args.steps, 20)), 3, dev,
                                             variant_layers=("reindex_masked", "reuse", "reuse", "reuse"))
        torch.cuda.empty_cache()
        line["prefill"] = measure_prefill(wl.prefill_chunk(device="cuda"), 3, 3, dev, fp4["tflops"])
        torch.cuda.empty_cache()
    if world > 1:
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()
    if rank == 0:
        print(json.dumps(line), flush=True)


def run_e2e(bench, W, args, dev, flush):
    """Same metric through the public calls with host buffers: every step copies its
    inputs (new token, indexer query, head weights, query, positions) from pinned host
    memory and reads the step's result (attention output + lse) back to the host.
    Like the device-timed steps, each step (copies in, the public calls, copies out)
    is launched as one CUDA graph, as a serving loop would; --no-graph launches the
    calls one by one instead."""
    first = args.warmup + args.steps
    names = ("kv_new", "ik_new", "q_idx", "w", "q", "q_pos")
    host_in = [[getattr(bench, n)[first + s].cpu().pin_memory() for n in names]
               for s in range(args.e2e_steps)]
    dev_in = [torch.empty_like(getattr(bench, n)[first]) for n in names]
    out_h = torch.empty(bench.out.shape, dtype=bench.out.dtype).pin_memory()
    lse_h = torch.empty(bench.lse.shape, dtype=bench.lse.dtype).pin_memory()
    h2d = sum(x.numel() * x.element_size() for x in host_in[0])
    d2h = out_h.numel() * out_h.element_size() + lse_h.numel() * lse_h.element_size()
    for n, d in zip(names, dev_in):  # the step reads slot `first` of each input list
        getattr(bench, n)[first] = d
    # the inputs of the score (indexer query, weights, positions) are copied on the
    # main stream; the new token and the attention query on the side branch, where
    # they overlap the score and the top-k (the attention waits for that branch)
    side_names = ("kv_new", "ik_new", "q")

    def one_step(s):
        main = torch.cuda.current_stream()
        fork = torch.cuda.Event()
        fork.record(main)
        bench.side.wait_event(fork)
        for n, d, h in zip(names, dev_in, host_in[s]):
            if n in side_names:
                with torch.cuda.stream(bench.side):
                    d.copy_(h, non_blocking=True)
            else:
                d.copy_(h, non_blocking=True)
        bench.step(first)
        out_h.copy_(bench.out, non_blocking=True)
        lse_h.copy_(bench.lse, non_blocking=True)

    graphs = None
    if not args.no_graph:
        graphs = []
        for s in range(args.e2e_steps):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                one_step(s)
            graphs.append(g)
        torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    total = 0.0
    for s in range(args.e2e_steps):
        flush()
        start.record()
        if graphs is not None:
            graphs[s].replay()
        else:
            one_step(s)
        end.record()
        torch.cuda.synchronize()
        total += start.elapsed_time(end)
    if bench.err.item() != 0:
        raise RuntimeError(f"device error word {bench.err.item()} in the e2e steps")
    value = W.batch * args.e2e_steps / (total / 1e3)
    return {"value": round(value, 2), "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "steps": args.e2e_steps, "ms_per_step": round(total / args.e2e_steps, 4)}


# ----------------------------------------------------------------------------- secondary workloads
# The configurations besides the headline, timed the same way (one CUDA graph per
# step, L2 flushed between steps, CUDA events on the launching stream).  Each prints
# its own JSON line; the headline line above is the Full-layer decode.

def group_step_bytes(W, T):
    """Algorithmic HBM bytes of one decoder-group step with T visible entries (append
    excluded): per layer what the method must move, summed over the group's layers."""
    B, k, H, H_I = W.batch, W.topk, W.heads, W.index_heads
    swa = 128 * (594 if W.swa_dtype == 1 else 1152)
    attn = k * (324 + 4) + swa + H * 576 * 2 + H * 512 * 4      # per sequence and attention layer
    qidx = H_I * 128 * 2 + 4 * H_I
    per_seq = 0
    for role in W.layers:
        if role == "full":
            per_seq += T * 68 + qidx + attn
        elif role == "reindex":
            per_seq += W.pool_blocks * W.pool_block_size * 68 + W.pool_blocks * 4 + qidx + attn
        elif role == "reindex_masked":  # every visible key is read
            per_seq += T * 68 + W.pool_blocks * 4 + qidx + attn
        else:
            per_seq += attn
    return B * per_seq


class GroupDecode:
    """A decoder group at a decode step on one cache: append the step's token, then
    each layer of W.layers in order -- "full": score every visible entry, top-k (and
    the 2,048-block pool when a Reindex layer follows), attention; "reindex": score the
    positions of the pool, top-k, attention; "reuse": attention with the last indexer
    layer's indices.  Every layer has its own queries; the layers share the cache (a
    model's layers have caches of the same shape, and the kernels read them the same
    way).  With W.ratio == 2 the cache is encoder-style: two tokens per entry, the
    step's token goes through the compression buffer."""

    def __init__(self, W, n_steps, device):
        from fp4_compressed_sparse_gb300 import csa2
        from fp4_compressed_sparse_gb300 import workloads as wl
        self.csa2, self.W = csa2, W
        B, ctx, nl = W.batch, W.context, len(W.layers)
        self.cap = (ctx + n_steps) // W.ratio + 8
        self.cache = csa2.Cache(B, self.cap, ratio=W.ratio, swa_dtype=W.swa_dtype)
        self.rope = csa2.rope_table(W.theta, W.ratio * self.cap + 16)
        self.err = torch.zeros(1, dtype=torch.int32, device=device)
        # ratio 1: bound each staging copy to ~512 MB; ratio 2: whole generator chunks
        # (four 704-wide streams; a partial chunk would redraw the whole chunk)
        chunk = max(256, min(wl.CHUNK, (1 << 29) // (B * 576 * 4))) if W.ratio == 1 else wl.CHUNK
        if W.ratio == 2:
            self.ba, self.bb = W.bias(device=device)
        for t0 in range(0, ctx, chunk):
            n = min(chunk, ctx - t0)
            if W.ratio == 1:
                kv = torch.stack([W.kv(b, t0, n, device=device) for b in range(B)])
                ik = torch.stack([W.ik(b, t0, n, device=device) for b in range(B)])
                csa2.kv_append(self.cache, kv, ik, self.rope, err=self.err)
                del kv, ik
            else:
                rows = [torch.stack(x) for x in zip(*[W.cmp_rows(b, t0, n, device=device) for b in range(B)])]
                csa2.kv_append(self.cache, rope_cs=self.rope, cmp=rows + [self.ba, self.bb], err=self.err)
                del rows
        torch.cuda.synchronize()
        if W.ratio == 1:
            self.kv_new = [torch.stack([W.kv(b, ctx + s, 1, device=device) for b in range(B)])
                           for s in range(n_steps)]
            self.ik_new = [torch.stack([W.ik(b, ctx + s, 1, device=device) for b in range(B)])
                           for s in range(n_steps)]
        else:  # (C^a, C^b, Z^a, Z^b) [B, 1, 704] of the step's token
            self.cmp_new = [[torch.stack(x) for x in zip(*[W.cmp_rows(b, ctx + s, 1, device=device)
                                                           for b in range(B)])] for s in range(n_steps)]
        self.q_pos = [torch.full((B,), ctx + s, dtype=torch.int64, device=device) for s in range(n_steps)]
        self.q_idx = [[W.q_idx(s, l, device=device) for l in range(nl)] for s in range(n_steps)]
        self.w = [[W.w(s, l, device=device) for l in range(nl)] for s in range(n_steps)]
        self.q = [[W.q(s, l, device=device) for l in range(nl)] for s in range(n_steps)]
        has_full = "full" in W.layers
        # the Full layer builds the pool only for Reindex layers that follow; a group
        # without a Full layer scores inside the prior pool (uniformly drawn blocks)
        self.build_pool = has_full and "reindex" in W.layers
        self.pool = (torch.empty((B, W.pool_blocks), dtype=torch.int32, device=device) if has_full
                     else W.pool(device=device))
        self.pool_cnt = torch.empty((B,), dtype=torch.int32, device=device)
        pstride = W.pool_blocks * W.pool_block_size
        self.scores = torch.empty((B, self.cap), device=device)
        self.pscores = torch.empty((B, pstride), device=device)
        self.aux = csa2.score_aux(B, self.cap)
        self.paux = csa2.score_aux(B, pstride)
        self.idx = torch.empty((B, W.topk), dtype=torch.int32, device=device)
        self.out = torch.empty((B, W.heads, 512), device=device)
        self.lse = torch.empty((B, W.heads), device=device)
        self.ws_score = csa2.index_score_workspace(B, W.index_heads)
        self.ws_topk = csa2.topk_workspace(B, self.cap, W.topk, W.pool_blocks)
        self.ws_ptopk = csa2.topk_workspace(B, pstride, W.topk)
        self.ws_attn = csa2.attn_workspace(B, W.heads, W.topk)
        self.side = torch.cuda.Stream(device=device)

    def step(self, s, marks=None):
        """One step; with `marks` (a list of events) the parts run in order on one stream
        with an event before each layer's score, its top-k, its attention and at the end
        (a Reuse layer records the first two back to back)."""
        c, W = self.csa2, self.W
        main = torch.cuda.current_stream()
        mark = (lambda: marks.pop(0).record()) if marks is not None else (lambda: None)

        def append():
            if W.ratio == 1:
                c.kv_append(self.cache, self.kv_new[s], self.ik_new[s], self.rope, err=self.err)
            else:
                c.kv_append(self.cache, rope_cs=self.rope, cmp=self.cmp_new[s] + [self.ba, self.bb], err=self.err)

        if marks is not None:
            append()
        else:
            fork, join = torch.cuda.Event(), torch.cuda.Event()
            fork.record(main)
            self.side.wait_event(fork)
            with torch.cuda.stream(self.side):
                append()
            join.record(self.side)
        joined = marks is not None
        for l, role in enumerate(W.layers):
            mark()
            if role == "full":
                c.index_score(self.cache, self.q_idx[s][l], self.w[s][l], self.q_pos[s], self.scores, err=self.err,
                              ws=self.ws_score, aux=self.aux)
                mark()
                c.topk(self.scores, W.ratio, self.q_pos[s], W.topk, self.idx, self.ws_topk,
                       pool_out=self.pool if self.build_pool else None,
                       pool_count=self.pool_cnt if self.build_pool else None, err=self.err, aux=self.aux)
            elif role == "reindex":
                c.index_score(self.cache, self.q_idx[s][l], self.w[s][l], self.q_pos[s], self.pscores,
                              pool=self.pool, err=self.err, ws=self.ws_score, aux=self.paux)
                mark()
                c.topk(self.pscores, W.ratio, self.q_pos[s], W.topk, self.idx, self.ws_ptopk, pool=self.pool,
                       err=self.err, aux=self.paux)
            elif role == "reindex_masked":
                # the published reference code's form: score every visible position,
                # mask the positions outside the pool, top-k of the whole row
                c.index_score(self.cache, self.q_idx[s][l], self.w[s][l], self.q_pos[s], self.scores, err=self.err,
                              ws=self.ws_score)
                mark()
                c.mask_to_pool(self.scores, W.ratio, self.q_pos[s], self.pool, W.pool_block_size)
                c.topk(self.scores, W.ratio, self.q_pos[s], W.topk, self.idx, self.ws_topk, err=self.err)
            else:
                mark()  # Reuse: no indexer
            if not joined:
                main.wait_event(join)  # the attention reads the new token's window slot
                joined = True
            mark()
            c.sparse_attn_decode(self.cache, self.q[s][l], self.q_pos[s], self.idx, self.out, self.lse,
                                 self.ws_attn, W.sm_scale, err=self.err)
        mark()


class PrefillBench:
    """Encoder-style chunked prefill (ratio 2): one step = csa2_prefill_chunk of the
    chunk's tokens against the prior entries.  The cache's token count, window ring
    and compression buffer are put back before every step (outside the timed region),
    so that every step appends the same chunk at the same positions."""

    def __init__(self, W, device):
        from fp4_compressed_sparse_gb300 import csa2
        from fp4_compressed_sparse_gb300 import workloads as wl
        self.csa2, self.W = csa2, W
        self.cap = (W.prior + W.chunk) // 2 + 8
        c = self.cache = csa2.Cache(1, self.cap, ratio=2, swa_dtype=W.swa_dtype)
        self.rope = csa2.rope_table(W.theta, 2 * self.cap + 16)
        self.err = torch.zeros(1, dtype=torch.int32, device=device)
        self.ba, self.bb = W.bias(device=device)
        for t0 in range(0, W.prior, wl.CHUNK):
            rows = W.cmp_rows(t0, wl.CHUNK, device=device)
            csa2.kv_append(c, rope_cs=self.rope, cmp=[r[None] for r in rows] + [self.ba, self.bb], err=self.err)
        torch.cuda.synchronize()
        self.saved = [t.clone() for t in (c.n_tokens, c.swa_codes, c.swa_scales, c.cmp_buf)]
        self.rows = list(W.cmp_rows(W.prior, W.chunk, device=device))
        self.q_idx, self.w, self.q = W.q_idx(device=device), W.w(device=device), W.q(device=device)
        Q, k = W.chunk, W.topk
        self.idx = torch.empty((Q, k), dtype=torch.int32, device=device)
        self.out = torch.empty((Q, W.heads, 512), device=device)
        self.lse = torch.empty((Q, W.heads), device=device)
        self.ws = csa2.prefill_workspace(Q, self.cap, W.index_heads, W.heads, k)

    def restore(self):
        c = self.cache
        for dst, src in zip((c.n_tokens, c.swa_codes, c.swa_scales, c.cmp_buf), self.saved):
            dst.copy_(src)

    def step(self, s):
        W = self.W
        self.csa2.prefill_chunk(self.cache, 0, self.rows + [self.ba, self.bb], self.rope, self.q_idx, self.w, self.q,
                                W.topk, W.sm_scale, self.idx, self.out, self.lse, self.ws, err=self.err)


def _time_steps(bench, steps, warmup, dev, step_fn=None):
    """Mean ms of `steps` CUDA-graph steps of a bench object (warm-up eager, L2
    flushed before every timed step, events around each)."""
    step_fn = step_fn or bench.step
    flush = L2Flush(dev)
    for s in range(warmup):
        flush()
        step_fn(s)
    torch.cuda.synchronize()
    graphs = []
    for i in range(steps):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            step_fn(warmup + i)
        graphs.append(g)
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for i in range(steps):
        flush()
        ev[i][0].record()
        graphs[i].replay()
        ev[i][1].record()
    torch.cuda.synchronize()
    if bench.err.item() != 0:
        raise RuntimeError(f"device error word {bench.err.item()} in the timed steps")
    return statistics.mean(a.elapsed_time(b) for a, b in ev)


class HcaDecode:
    """A heavily compressed attention layer in the V4 format, for the comparison of
    cache formats ([P5] §2.3.2: one entry per m' = 128 tokens, no overlap, attention
    over every compressed entry, no indexer): a cache of context/128 V4-format
    entries (seeded N(0,1) rows standing for the compressed entries), and each step
    attends over all of them plus the 128-token window through the sparse-attention
    call with every entry selected."""

    def __init__(self, W, n_steps, device, m=128):
        from fp4_compressed_sparse_gb300 import csa2
        self.csa2, self.W = csa2, W
        B, n = W.batch, W.context // m
        self.n = n
        self.cache = csa2.Cache(B, n + 8, ratio=1, swa_dtype=W.swa_dtype, entry_format=csa2.ENTRY_FP8)
        rope = csa2.rope_table(W.theta, n + 16)
        self.err = torch.zeros(1, dtype=torch.int32, device=device)
        kv = torch.stack([W.kv(b, 0, n, device=device) for b in range(B)])
        ik = torch.stack([W.ik(b, 0, n, device=device) for b in range(B)])
        csa2.kv_append(self.cache, kv, ik, rope, err=self.err)
        del kv, ik
        self.idx = torch.arange(n, dtype=torch.int32, device=device).repeat(B, 1).contiguous()
        self.q = [W.q(s, 7, device=device) for s in range(n_steps)]
        self.q_pos = torch.full((B,), n, dtype=torch.int64, device=device)
        self.out = torch.empty((B, W.heads, 512), device=device)
        self.lse = torch.empty((B, W.heads), device=device)
        self.ws = csa2.attn_workspace(B, W.heads, n)

    def step(self, s):
        self.csa2.sparse_attn_decode(self.cache, self.q[s], self.q_pos, self.idx, self.out, self.lse, self.ws,
                                     self.W.sm_scale, err=self.err)


def measure_formats(W, steps, warmup, dev):
    """The cache formats compared at the headline configuration ([P5] §2.3.2,
    §2.3.4; [P3] per-token global KV by generation): the Full-layer decode step
    with V4.1 FP4 entries and with V4 FP8 + bf16-RoPE entries (same indexer keys,
    scan and selection), and an HCA-style layer (m' = 128, dense over its entries)."""
    from fp4_compressed_sparse_gb300 import csa2
    out = {}
    for name, fmt in (("v41_fp4", csa2.ENTRY_FP4), ("v4_fp8", csa2.ENTRY_FP8)):
        bench = FullDecode(W, warmup + steps, dev, entry_format=fmt)
        ms = _time_steps(bench, steps, warmup, dev)
        out[name] = {"ms_per_step": round(ms, 4), "tokens_per_s": round(W.batch / (ms / 1e3), 2),
                     "entry_bytes": bench.cache.entry_bytes(),
                     "selected_entry_bytes": bench.cache.entry_bytes() - 68}
        del bench
        torch.cuda.empty_cache()
    hca = HcaDecode(W, warmup + steps, dev)
    ms = _time_steps(hca, steps, warmup, dev)
    out["hca_m128_fp8"] = {"ms_per_step": round(ms, 4), "entries_per_sequence": hca.n,
                           "entry_bytes": hca.cache.entry_bytes() - 68,
                           "note": "attention over every compressed entry + the window; no indexer"}
    del hca
    out["config"] = f"{W.name}: batch {W.batch}, context {W.context}, {W.heads} heads, top-{W.topk}"
    return out


def measure_paged(W, steps, warmup, dev, page_entries):
    """The headline decode step on a paged cache (pages of page_entries entries in
    a shuffled order over the pool): `steps` CUDA-graph steps, L2 flushed between."""
    bench = FullDecode(W, warmup + steps, dev, page_entries=page_entries)
    flush = L2Flush(dev)
    for s in range(warmup):
        flush()
        bench.step(s)
    torch.cuda.synchronize()
    graphs = []
    for i in range(steps):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            bench.step(warmup + i)
        graphs.append(g)
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for i in range(steps):
        flush()
        ev[i][0].record()
        graphs[i].replay()
        ev[i][1].record()
    torch.cuda.synchronize()
    if bench.err.item() != 0:
        raise RuntimeError(f"device error word {bench.err.item()} in the paged steps")
    ms = statistics.mean(a.elapsed_time(b) for a, b in ev)
    del graphs
    # the parts one after another with events between (a few eager steps)
    parts = {n: [] for n in FullDecode.PARTS}
    for i in range(min(steps, 5)):
        pev = [torch.cuda.Event(enable_timing=True) for _ in range(len(FullDecode.PARTS) + 1)]
        flush()
        bench.step(warmup + i, ev=pev)
        torch.cuda.synchronize()
        for k, n in enumerate(FullDecode.PARTS):
            parts[n].append(pev[k].elapsed_time(pev[k + 1]))
    del bench
    return {"workload": W.name, "page_entries": page_entries, "page_order": "seeded random permutation of the pool",
            "steps": steps, "ms_per_step": round(ms, 4), "value": round(W.batch / (ms / 1e3), 2), "unit": UNIT,
            "part_ms_eager": {k: round(statistics.median(v), 4) for k, v in parts.items()}}


def measure_group(W, steps, warmup, dev, variant_layers=None):
    """One decoder-group workload (Full / Reindex / Reuse layers over one cache):
    `steps` timed steps, one CUDA graph each, L2 flushed between them; then one
    more step run layer by layer with events between, for the per-layer split.
    With variant_layers, the same cache and inputs are timed again with those
    layer roles (a comparison of two forms of the same group)."""
    # inputs (and cache room) for every step: warm-up, timed, the breakdown step,
    # and the variant's timed and breakdown steps after them
    n_steps = warmup + steps + 1 + ((steps + 1) if variant_layers else 0)
    bench = GroupDecode(W, n_steps, dev)
    out = _time_group(bench, W, steps, warmup, dev, first=0)
    if variant_layers:
        import dataclasses
        Wv = dataclasses.replace(W, layers=tuple(variant_layers))
        bench.W = Wv
        out["variant"] = _time_group(bench, Wv, steps, 0, dev, first=warmup + steps + 1)
    del bench
    return out


def _time_group(bench, W, steps, warmup, dev, first=0):
    """Time `steps` steps of a GroupDecode whose step inputs start at index
    `first` (warm-up steps first, then the timed ones, then one breakdown step)."""
    flush = L2Flush(dev)
    for s in range(warmup):
        flush()
        bench.step(first + s)
    torch.cuda.synchronize()
    if bench.err.item() != 0:
        raise RuntimeError(f"device error word {bench.err.item()} during warm-up")
    graphs = []
    for i in range(steps):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            bench.step(first + warmup + i)
        graphs.append(g)
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    sampler = ClockSampler(dev.index or 0)
    sampler.start()
    t_begin = time.perf_counter()
    for i in range(steps):
        flush()
        ev[i][0].record()
        graphs[i].replay()
        ev[i][1].record()
    torch.cuda.synchronize()
    sampler.mark(t_begin, time.perf_counter())
    clocks = sampler.stop()
    if bench.err.item() != 0:
        raise RuntimeError(f"device error word {bench.err.item()} in the timed steps")
    step_ms = [a.elapsed_time(b) for a, b in ev]
    ms = statistics.mean(step_ms)
    del graphs
    # per-layer breakdown: one more step, parts in order with events between
    marks = [torch.cuda.Event(enable_timing=True) for _ in range(3 * len(W.layers) + 1)]
    flush()
    bench.step(first + warmup + steps, marks=list(marks))
    torch.cuda.synchronize()
    parts = []
    for l, role in enumerate(W.layers):
        a, m, b, c2 = marks[3 * l], marks[3 * l + 1], marks[3 * l + 2], marks[3 * l + 3]
        parts.append({"layer": l, "role": role, "indexer_ms": round(a.elapsed_time(b), 4),
                      "score_ms": round(a.elapsed_time(m), 4), "topk_ms": round(m.elapsed_time(b), 4),
                      "attention_ms": round(b.elapsed_time(c2), 4)})
    hbm, hbm_kind = peaks()
    T = (W.context + first + warmup + steps // 2) // W.ratio  # visible entries at the middle step
    nbytes = group_step_bytes(W, T)
    gbs = nbytes / (ms / 1e3) / 1e9
    return {"metric": "decoder-group tokens/s and algorithmic HBM GB/s (% of roofline)",
            "workload": W.name, "value": round(W.batch / (ms / 1e3), 2), "unit": "tokens/s",
            "higher_is_better": True, "steps": steps, "warmup": warmup, "ms_per_step": round(ms, 4),
            "ms_per_step_min_max": [round(min(step_ms), 4), round(max(step_ms), 4)],
            "layers": list(W.layers), "batch": W.batch, "context": W.context,
            "kv_hbm": {"algorithmic_bytes_per_step": nbytes, "gbs": round(gbs, 1), "frac": round(gbs / hbm, 4),
                       "peak_gbs": hbm, "peak_kind": hbm_kind},
            "layer_breakdown": parts, "clocks": clocks, "l2": "flushed between timed steps",
            "launch": "one CUDA graph per step"}


def prefill_flop(W):
    """FP4 indexer scoring FLOP of one chunk: 2 * H_I * 128 per (query, visible
    entry); query i sees prior/2 + i//2 entries."""
    return sum(2 * W.index_heads * 128 * (W.prior // 2 + i // 2) for i in range(W.chunk))


def measure_prefill(W, steps, warmup, dev, fp4_peak=None):
    """Chunked prefill: `steps` timed chunks (one CUDA graph each, the cache's token
    count, window ring and compression buffer restored and the L2 flushed before
    each, outside the events), then one chunk with the library's phase events for
    the append / score / select / attention split."""
    from fp4_compressed_sparse_gb300 import csa2
    bench = PrefillBench(W, dev)
    flush = L2Flush(dev)
    for s in range(warmup):
        bench.restore()
        flush()
        bench.step(s)
    torch.cuda.synchronize()
    if bench.err.item() != 0:
        raise RuntimeError(f"device error word {bench.err.item()} during warm-up")
    graphs = []
    for i in range(steps):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            bench.step(0)
        graphs.append(g)
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    sampler = ClockSampler(dev.index or 0)
    sampler.start()
    t_begin = time.perf_counter()
    for i in range(steps):
        bench.restore()
        flush()
        ev[i][0].record()
        graphs[i].replay()
        ev[i][1].record()
    torch.cuda.synchronize()
    sampler.mark(t_begin, time.perf_counter())
    clocks = sampler.stop()
    if bench.err.item() != 0:
        raise RuntimeError(f"device error word {bench.err.item()} in the timed steps")
    ms = statistics.median([a.elapsed_time(b) for a, b in ev])
    del graphs
    # phase split: events recorded by the library at its phase boundaries
    pev = [torch.cuda.Event(enable_timing=True) for _ in range(256)]
    for e in pev:
        e.record()
    torch.cuda.synchronize()
    bench.restore()
    flush()
    csa2.set_phase_events(pev)
    bench.step(0)
    n = csa2.phase_events_recorded()
    csa2.set_phase_events(None)
    torch.cuda.synchronize()
    phases = {"append": pev[0].elapsed_time(pev[1]), "score": 0.0, "select": 0.0, "attention": 0.0}
    for b in range(2, n - 2, 3):
        phases["score"] += pev[b - 1].elapsed_time(pev[b])
        phases["select"] += pev[b].elapsed_time(pev[b + 1])
        phases["attention"] += pev[b + 1].elapsed_time(pev[b + 2])
    flop = prefill_flop(W)
    score_rate = flop / (phases["score"] / 1e3) / 1e12
    chunk_rate = flop / (ms / 1e3) / 1e12
    out = {"metric": "prefill chunk: query tokens/s, and FP4 scoring TFLOP/s",
           "workload": W.name, "value": round(W.chunk / (ms / 1e3), 2), "unit": "tokens/s",
           "higher_is_better": True, "steps": steps, "warmup": warmup, "ms_per_chunk": round(ms, 4),
           "chunk": W.chunk, "prior_tokens": W.prior, "scoring_tflop": round(flop / 1e12, 3),
           "phase_ms": {k: round(v, 4) for k, v in phases.items()},
           "phase_note": "one extra chunk with the library's phase events (score blocks of queries, "
                         "each scored, selected and attended in turn)",
           "tensor": {"scoring_tflops_in_score_phase": round(score_rate, 1),
                      "scoring_tflops_over_chunk": round(chunk_rate, 1)},
           "clocks": clocks, "l2": "flushed between timed chunks", "launch": "one CUDA graph per chunk"}
    if fp4_peak:
        out["tensor"].update({"fp4_peak_tflops": fp4_peak, "frac_in_score_phase": round(score_rate / fp4_peak, 4),
                              "peak_kind": "measured (tcgen05 kind::mxf4 M128 N128 K64 back to back)"})
    del bench
    return out


def measure_fp4_peak(dev, reps=5):
    """Dense rate of the index score's block-scaled FP4 MMA (tcgen05 kind::mxf4,
    M 128 x N 128 x K 64), operands resident in shared memory, one CTA per SM:
    best of `reps` launches of ~2-4 ms, timed with CUDA events."""
    from fp4_compressed_sparse_gb300 import csa2
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    iters = 1 << 15
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    sink = torch.zeros(sms, dtype=torch.int32, device=dev)
    csa2.mxf4_peak_launch(sms, 64, sink, err)  # warm-up
    best = 0.0
    times = []
    for _ in range(reps):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        csa2.mxf4_peak_launch(sms, iters, sink, err)
        b.record()
        torch.cuda.synchronize()
        ms = a.elapsed_time(b)
        times.append(ms)
        best = max(best, sms * iters * 2.0 * 128 * 128 * 64 / (ms / 1e3) / 1e12)
    if int(err.item()) != 0:
        raise RuntimeError(f"device error word {int(err.item())} in the FP4 peak kernel")
    return {"tflops": round(best, 1), "ctas": sms, "mma_per_cta": iters, "launch_ms": [round(t, 3) for t in times],
            "instruction": "tcgen05.mma.cta_group::1.kind::mxf4.block_scale.scale_vec::2X M128 N128 K64"}


def run_secondary(args):
    from fp4_compressed_sparse_gb300 import build_lib, csa2
    from fp4_compressed_sparse_gb300 import workloads as wl
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    build_lib.build()
    csa2.load()
    W = getattr(wl, args.workload)(device="cuda")
    if args.workload.startswith("prefill_chunk"):
        line = measure_prefill(W, args.steps, args.warmup, dev, measure_fp4_peak(dev)["tflops"])
    else:
        line = measure_group(W, args.steps, args.warmup, dev)
    line.update({"data": "synthetic (seeded)", "impl": "ours"})
    print(json.dumps(line), flush=True)

# ----------------------------------------------------------------------------- oracle arm
def cpu_baseline(W, args, sample_steps=None, min_seconds=10.0, max_steps=1024, single_thread_steps=3):
    """The CPU oracle (as it stands) on a bounded sample of the workload: sequence 0,
    decode steps (append the token, Full-layer score over every visible position,
    top-k, pool, attention) on the host cores, `sample_steps` of them, or when that is
    None as many as fill `min_seconds` of oracle time (at most `max_steps`)."""
    import numpy as np
    from oracle import oracle as orc

    dev = "cuda" if torch.cuda.is_available() else "cpu"
    orc.build()
    cap = sample_steps if sample_steps is not None else max_steps
    cache = orc.Cache(W.context + cap + 8, swa_dtype=W.swa_dtype)
    chunk = 8192
    for t0 in range(0, W.context, chunk):
        n = min(chunk, W.context - t0)
        orc.append_r1(cache, W.kv(0, t0, n, device=dev).cpu().numpy(),
                      W.ik(0, t0, n, device=dev).cpu().numpy(), W.theta)
    u16 = lambda t: t.cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
    t_total = 0.0
    done = 0
    for s in range(cap):
        if sample_steps is None and t_total >= min_seconds:
            break
        kv = W.kv(0, W.context + s, 1, device=dev).cpu().numpy()
        ik = W.ik(0, W.context + s, 1, device=dev).cpu().numpy()
        q_idx = u16(W.q_idx(s, 0, device=dev)[0])
        w = W.w(s, 0, device=dev)[0].cpu().numpy()
        q = u16(W.q(s, 0, device=dev)[0])
        t0 = time.perf_counter()
        orc.append_r1(cache, kv, ik, W.theta)
        orc.full_layer(cache, q_idx, w, q, W.context + s, W.topk, W.sm_scale)
        t_total += time.perf_counter() - t0
        done += 1
    out = {"value": round(done / t_total, 4), "unit": UNIT, "cores": orc.num_threads(),
           "kind": "oracle", "seconds": round(t_total, 3), "steps": done,
           "sample": f"sequence 0 x {done} decode step(s) of {W.name}: append + Full-layer "
                     f"score over {W.context} positions x {W.index_heads} heads + top-{W.topk} + "
                     f"pool + attention ({W.heads} heads)"}
    if single_thread_steps > 0:
        # the same steps again on one host thread
        threads = orc.num_threads()
        orc.set_num_threads(1)
        t1 = 0.0
        n1 = min(single_thread_steps, done)
        for s in range(n1):
            q_idx = u16(W.q_idx(s, 0, device=dev)[0])
            w = W.w(s, 0, device=dev)[0].cpu().numpy()
            q = u16(W.q(s, 0, device=dev)[0])
            t0 = time.perf_counter()
            orc.full_layer(cache, q_idx, w, q, W.context + s, W.topk, W.sm_scale)
            t1 += time.perf_counter() - t0
        orc.set_num_threads(threads)
        out["single_thread"] = {"value": round(n1 / t1, 4), "unit": UNIT, "cores": 1, "seconds": round(t1, 3),
                                "steps": n1, "note": "Full-layer score + top-k + pool + attention of the first "
                                                     "steps again (the cache already holds their tokens)"}
    return out


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    from fp4_compressed_sparse_gb300 import workloads as wl
    W = getattr(wl, args.workload)(device="cuda" if torch.cuda.is_available() else "cpu")
    steps = max(1, args.steps)
    cb = cpu_baseline(W, args, sample_steps=steps, single_thread_steps=0)
    line = {"impl": "reference", "metric": METRIC, "value": cb["value"], "unit": UNIT, "n_gpus": world,
            "steps": steps, "warmup": args.warmup, "ms_per_step": round(1e3 * cb["seconds"] / steps, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64/f32",
            "data": "synthetic (seeded)", "config": {"workload": W.name, "batch": W.batch,
                                                      "context": W.context, "heads": W.heads,
                                                      "index_heads": W.index_heads, "topk": W.topk},
            "cpu_baseline": cb,
            "e2e": {"value": cb["value"], "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def spawn_ranks(n):
    """Run this command as n local ranks (torch.distributed.run on 127.0.0.1) and
    return its exit status; rank 0 prints the line."""
    import socket
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        port = sk.getsockname()[1]
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={n}",
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.abspath(__file__)] + sys.argv[1:]
    return subprocess.call(cmd)


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="full_decode",
                    choices=["full_decode", "full_decode_small", "tiny_decode", "reindex_decode", "reindex_masked_decode",
                             "stack_1m", "encoder_decode", "prefill_chunk", "prefill_chunk_small"],
                    help="full_decode is the headline; reindex_decode, stack_1m, encoder_decode and prefill_chunk "
                         "print their own "
                         "measurement line")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--e2e-steps", type=int, default=5)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-graph", action="store_true", help="launch every kernel eagerly instead of one "
                    "CUDA graph per step")
    ap.add_argument("--headline-only", action="store_true", help="skip the 1 M-context group, the prefill chunk "
                    "and the FP4 peak that the default run adds to its line")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.gpus < 1:
        ap.error("--gpus must be >= 1")
    if "WORLD_SIZE" in os.environ:
        if int(os.environ["WORLD_SIZE"]) != args.gpus:
            ap.error(f"--gpus {args.gpus} but WORLD_SIZE={os.environ['WORLD_SIZE']}")
    elif args.gpus > 1:
        # one process per GPU: start the ranks here, as the launcher would
        sys.exit(spawn_ranks(args.gpus))
    if args.impl == "reference":
        run_reference(args)
    elif args.workload in ("reindex_decode", "reindex_masked_decode", "stack_1m", "encoder_decode", "prefill_chunk",
                           "prefill_chunk_small"):
        run_secondary(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()

"""Benchmark of the gated-attention hot path on GB300.

One step = one pass of the whole path on synthetic inputs already resident in
HBM: a causal prefill of the Qwen3.5-0.8B-shaped full-attention layer (B1 S4096
H8 G2 d256, rotary 64, elementwise gate) followed by one decode step of 64
sequences with 16k-32k cached tokens each (H8 G2 d256).  L2 is flushed (a 256 MiB
write) before every timed call; each call is timed with CUDA events on the stream
it runs on.

  value        prefill TFLOP/s (algorithmic causal FLOPs / time of the prefill call)
  decode       decode GB/s (K/V cache + q/gate/out bytes / time of the decode call)
  roofline     the dominant kernel (tcgen05 prefill) against measured bf16 peak,
               plus the decode split kernel against measured HBM copy bandwidth
  e2e          prefill through the public API with pinned host buffers, H2D and
               D2H copies inside the timed region (steps pipelined: two device
               slots, copy streams beside the compute stream)
  cpu_baseline the fp64 oracle on a bounded sample of the prefill workload

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
Under torchrun (N > 1) every rank runs the same workload on its own GPU (replicas:
the path has no exchange step); times are maxed over ranks.
"""
import argparse
import dataclasses
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "gated-attn causal prefill TFLOP/s (% bf16 peak); decode KV GB/s (% HBM)"
PREFILL = "qwen35_08b_prefill"
DECODE = "qwen35_08b_decode"
# The projection after the path: Qwen3.5-0.8B's W_O maps the concatenated heads (8 x 256
# = 2048) back to its residual width 1024 ("Multi-head attention and GQA" chapter,
# glossary entry d_model).
OPROJ_PREFILL, OPROJ_HIDDEN = PREFILL, 1024
L2_FLUSH_BYTES = 256 << 20


def reduce_max(values, device=None):
    """Element-wise max of a list of floats over all ranks (the slowest rank sets
    every timing); identity when torch.distributed is not initialised."""
    import torch
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return list(values)
    t = torch.tensor(list(values), dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--prefill", default=PREFILL, help="prefill workload name (parity/tuning runs)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--only", choices=["prefill", "decode", "oproj"], default=None,
                    help="run one half of the path only (profiling runs; not a bench line)")
    ap.add_argument("--decode-batch", type=int, default=None,
                    help="override the decode batch (smaller profiling case; not a bench line)")
    ap.add_argument("--cpu-budget-s", type=float, default=8.0)
    ap.add_argument("--next-rows", action="store_true",
                    help="time the scope table's next rows (append / paged decode, packed sequences, gate "
                         "variants) and print their own JSON line")
    return ap.parse_args()


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return p["hbm_gbs"], p["bf16_tflops"], "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, 1900.0, "fallback"


def kernel_source_hash(files):
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, "gated_softmax_attention_gqa_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def profiled_traffic(summary_name, src_files):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on the
    kernel source as it is now (else None)."""
    path = os.path.join(ROOT, "profiles", summary_name)
    try:
        kv = {}
        with open(path) as f:
            for line in f:
                if ":" in line and line.strip().startswith("- "):
                    k, v = line.strip()[2:].split(":", 1)
                    kv[k.strip()] = v.strip().strip("`")
        if kv.get("kernel_source_sha256") != kernel_source_hash(src_files):
            return None
        return int(float(kv["dram_bytes_per_launch_full_workload"]))
    except (OSError, KeyError, ValueError):
        return None


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 20 ms."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "20", "-i",
                 str(gpu_index)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        self.t0 = self.t1 = None

    def mark_start(self):
        self.t0 = time.time()

    def mark_end(self):
        self.t1 = time.time()

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        time.sleep(0.05)
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        rows = [[c.strip() for c in ln.split(",")] for ln in out.strip().splitlines() if ln.count(",") >= 8]
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        sm = []
        smax = None
        for r in rows:
            try:
                sm.append(float(r[1]))
                smax = float(r[2])
            except ValueError:
                continue
            for n, v in zip(names, r[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        loaded = [s for s in sm if smax and s > 0.5 * smax] or sm
        return {"sm_mhz": statistics.median(loaded) if loaded else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(rows)}


def cpu_baseline(w, inputs, budget_s):
    """The fp64 oracle, as it stands, on a bounded sample of the prefill workload:
    all heads of a seeded set of query rows (the whole workload when that fits the
    budget); TFLOP/s over the causal FLOPs of the rows computed."""
    import numpy as np

    import oracle
    from gated_softmax_attention_gqa_gb300.workloads import prefill_flops

    rng = np.random.default_rng(1234)
    n = 16
    while True:
        full = n >= w.B * w.S
        if full:
            rb = np.repeat(np.arange(w.B, dtype=np.int32), w.S)
            rt = np.tile(np.arange(w.S, dtype=np.int32), w.B)
        else:
            flat = np.sort(rng.choice(w.B * w.S, size=n, replace=False))
            rb, rt = (flat // w.S).astype(np.int32), (flat % w.S).astype(np.int32)
        t0 = time.perf_counter()
        oracle.prefill_rows(inputs["q"], inputs["k"], inputs["v"], inputs["gate"], inputs["qnorm_w"],
                            inputs["knorm_w"], None, w.rotary_dim, w.rope_base, w.eps, w.gate_mode, rb, rt)
        dt = time.perf_counter() - t0
        flops = prefill_flops(w.B, w.S, w.H, w.d) if full else sum(4 * w.H * w.d * (int(t) + 1) for t in rt)
        if dt >= budget_s * 0.5 or full:
            what = "every query row" if full else f"{n} seeded query rows"
            return {"value": flops / dt / 1e12, "unit": "TFLOP/s", "cores": oracle.threads_used(), "kind": "oracle",
                    "sample": f"{what} x all {w.H} heads of {w.name} (B{w.B} S{w.S} H{w.H} G{w.G} d{w.d}); "
                              f"fp64 C loops, OpenMP; {dt:.1f} s",
                    "seconds": dt}
        n = min(w.B * w.S, int(n * max(2.0, budget_s / max(dt, 1e-3))))


def run_reference(args):
    """Reference arm: the fp64 oracle timed on the host cores (rank 0 only), on the
    same step as the GPU arm -- the headline prefill then the decode step -- each a
    bounded sample of its workload.  value = prefill TFLOP/s of the sample;
    ms_per_step = the oracle's time for one whole step at the sampled rates."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    from gated_softmax_attention_gqa_gb300.workloads import (WORKLOADS, decode_io_bytes, make_decode_inputs,
                                                             make_prefill_inputs, prefill_flops)

    w = WORKLOADS[args.prefill]
    wd = WORKLOADS[DECODE]
    inputs = make_prefill_inputs(w)
    per_step = max(2.0, 60.0 / max(1, args.steps + args.warmup))
    for _ in range(args.warmup):
        cpu_baseline(w, inputs, min(per_step, 2.0))
    vals, dvals = [], []
    last = dlast = None
    for _ in range(args.steps):
        last = cpu_baseline(w, inputs, per_step * 0.75)
        dlast = cpu_decode_baseline(wd, per_step * 0.25)
        vals.append(last["value"])
        dvals.append(dlast["value"])
    v, dv = statistics.median(vals), statistics.median(dvals)
    # the full step at these rates: the whole prefill's FLOPs and the whole decode step's bytes
    seqlens = torch_free_seqlens(wd)
    step_ms = 1e3 * (prefill_flops(w.B, w.S, w.H, w.d) / (v * 1e12) +
                     decode_io_bytes(seqlens, wd.H, wd.G, wd.d, wd.gate_mode) / (dv * 1e9))
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "TFLOP/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": step_ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": step_config(w, wd, args.gpus, seqlens),
            "decode": {"value": dv, "unit": "GB/s", "sample": dlast["sample"]},
            "cpu_baseline": {"value": v, "unit": "TFLOP/s", "cores": last["cores"], "kind": "oracle",
                             "sample": last["sample"] + "; decode: " + dlast["sample"] +
                             "; ms_per_step extrapolates both samples' rates to the whole step"},
            "e2e": {"value": v, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def torch_free_seqlens(wd):
    """The decode workload's sequence lengths (the same seeded draw as its inputs,
    without generating the cache)."""
    import torch

    g = torch.Generator("cpu").manual_seed(wd.seed)
    lo, hi = wd.seqlen_range
    return torch.randint(lo, hi + 1, (wd.B,), generator=g, dtype=torch.int64).tolist()


def run_next_rows(args):
    """The scope table's next rows, each timed like the headline calls (CUDA events
    around the call on its stream, L2 flushed before each, median of --steps after
    --warmup) on the headline shapes: decode with the new token appended and decode
    through a paged cache (GB/s of the algorithmic K/V + q/gate/out bytes, against
    the measured HBM copy), packed-sequence prefill and two gate variants (TFLOP/s
    against the measured bf16 peak).  One JSON line; one GPU."""
    import torch

    import gated_softmax_attention_gqa_gb300 as ga
    from gated_softmax_attention_gqa_gb300.workloads import (WORKLOADS, decode_io_bytes, make_decode_inputs,
                                                             make_prefill_inputs, prefill_flops)

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev)
    hbm_peak, bf16_peak, peak_kind = peaks()
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)

    def timed(fn):
        for _ in range(max(3, args.warmup)):
            flush.zero_()
            fn()
        torch.cuda.synchronize()
        evs = []
        for _ in range(args.steps):
            flush.zero_()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn()
            b.record(stream)
            evs.append((a, b))
        torch.cuda.synchronize()
        if ga.gattn_get_device_status() != 0:
            raise RuntimeError("device status set")
        return statistics.median(a.elapsed_time(b) for a, b in evs)

    rows = {}
    gen = torch.Generator().manual_seed(7)

    # ---- decode (the 64-sequence bf16-cache step): contiguous, with append, paged
    wd = WORKLOADS[DECODE]
    din = make_decode_inputs(wd)
    d = {k: v.to(dev) for k, v in din.items()}
    seqlens = din["seqlens"].tolist()
    dbytes = decode_io_bytes(seqlens, wd.H, wd.G, wd.d, wd.gate_mode)
    d_out = torch.empty((wd.B, wd.H * wd.d), dtype=torch.bfloat16, device=dev)
    d_ws = torch.empty(ga.gattn_decode_workspace_size(wd.B, wd.H, wd.G, wd.d, wd.Lmax), dtype=torch.uint8,
                       device=dev)
    dkw = dict(rotary_dim=wd.rotary_dim, rope_base=wd.rope_base, eps=wd.eps, gate_mode=wd.gate_mode, out=d_out,
               workspace=d_ws)

    def hbm_row(ms):
        gbs = dbytes / (ms * 1e-3) / 1e9
        return {"ms": ms, "value": gbs, "unit": "GB/s", "frac": gbs / hbm_peak}

    rows["decode_contiguous"] = hbm_row(timed(lambda: ga.gattn_decode(d["q_new"], d["kv_cache"], d["seqlens"],
                                                                       d["gate"], d["qnorm_w"], **dkw)))
    k_new = torch.randn(wd.B, wd.G, wd.d, generator=gen).to(torch.bfloat16).to(dev)
    v_new = torch.randn(wd.B, wd.G, wd.d, generator=gen).to(torch.bfloat16).to(dev)
    knorm_w = (1.0 + 0.1 * torch.randn(wd.d, generator=gen)).to(torch.bfloat16).to(dev)
    rows["decode_append"] = hbm_row(timed(lambda: ga.gattn_decode_append(
        d["q_new"], k_new, v_new, d["kv_cache"], d["seqlens"], d["gate"], d["qnorm_w"], knorm_w, **dkw)))
    # the same cache in a page pool: 256-token pages, each sequence's pages scattered
    # over the pool by a seeded permutation
    ps = 256
    n_pages = [(L + ps - 1) // ps for L in seqlens]
    perm = torch.randperm(sum(n_pages), generator=gen)
    pool = torch.empty((2, sum(n_pages), wd.G, ps, wd.d), dtype=torch.bfloat16, device=dev)
    table = torch.zeros((wd.B, max(n_pages)), dtype=torch.int32)
    at = 0
    for b, n in enumerate(n_pages):
        ids = perm[at:at + n]
        at += n
        table[b, :n] = ids.to(torch.int32)
        src = d["kv_cache"][:, b, :, :n * ps].reshape(2, wd.G, n, ps, wd.d).permute(0, 2, 1, 3, 4)
        pool[:, ids.to(dev)] = src
    table = table.to(dev)
    rows["decode_paged_256"] = hbm_row(timed(lambda: ga.gattn_decode_paged(
        d["q_new"], pool, table, d["seqlens"], d["gate"], d["qnorm_w"], **dkw)))
    del pool, d

    # ---- prefill on the Qwen3.5-0.8B-shaped layer's 4096 tokens
    wp = WORKLOADS[PREFILL]
    pin = make_prefill_inputs(wp)
    p = {k: v.to(dev) for k, v in pin.items()}
    p_out = torch.empty((wp.B, wp.S, wp.H * wp.d), dtype=torch.bfloat16, device=dev)
    p_ws = torch.empty(ga.gattn_prefill_workspace_size(wp.B, wp.S, wp.H, wp.G, wp.d), dtype=torch.uint8, device=dev)
    pkw = dict(rotary_dim=wp.rotary_dim, rope_base=wp.rope_base, eps=wp.eps)

    def tensor_row(ms, flops):
        tf = flops / (ms * 1e-3) / 1e12
        return {"ms": ms, "value": tf, "unit": "TFLOP/s", "frac": tf / bf16_peak}

    full = prefill_flops(wp.B, wp.S, wp.H, wp.d)
    rows["prefill_default_gate"] = tensor_row(timed(lambda: ga.gattn_prefill(
        p["q"], p["k"], p["v"], p["gate"], p["qnorm_w"], p["knorm_w"], gate_mode=wp.gate_mode, out=p_out,
        workspace=p_ws, **pkw)), full)
    rows["prefill_silu_additive_gate"] = tensor_row(timed(lambda: ga.gattn_prefill(
        p["q"], p["k"], p["v"], p["gate"], p["qnorm_w"], p["knorm_w"], gate_mode="elementwise", gate_act="silu",
        gate_additive=True, out=p_out, workspace=p_ws, **pkw)), full)
    z_shared = torch.randn(wp.B, wp.S, wp.d, generator=gen).to(torch.bfloat16).to(dev)
    rows["prefill_head_shared_gate"] = tensor_row(timed(lambda: ga.gattn_prefill(
        p["q"], p["k"], p["v"], z_shared, p["qnorm_w"], p["knorm_w"], gate_mode="head_shared", out=p_out,
        workspace=p_ws, **pkw)), full)
    # the same tokens as packed sequences of mixed lengths
    lens = [2048, 1024, 512, 256, 128, 128]
    assert sum(lens) == wp.S
    cu = [0]
    for n in lens:
        cu.append(cu[-1] + n)
    vflops = sum(prefill_flops(1, n, wp.H, wp.d) for n in lens)
    v_ws = torch.empty(ga.gattn_prefill_varlen_workspace_size(wp.S, len(lens), wp.H, wp.G, wp.d),
                       dtype=torch.uint8, device=dev)
    rows["prefill_packed_6_sequences"] = tensor_row(timed(lambda: ga.gattn_prefill_varlen(
        p["q"][0], p["k"][0], p["v"][0], p["gate"][0], p["qnorm_w"], p["knorm_w"], cu, gate_mode=wp.gate_mode,
        out=p_out[0], workspace=v_ws, **pkw)), vflops)

    line = {"next_rows": rows, "peaks": {"hbm_gbs": hbm_peak, "bf16_tflops": bf16_peak, "kind": peak_kind},
            "steps": args.steps, "warmup": args.warmup, "l2": "flushed (256 MiB write) before every timed call",
            "config": {"decode": f"{DECODE} (B{wd.B} H{wd.H} G{wd.G} d{wd.d}, lengths U[16384,32768]); paged: "
                                 f"{ps}-token pages in a shuffled pool",
                       "prefill": f"{PREFILL} (B1 S4096 H8 G2 d256); packed: lengths {lens}"}}
    print(json.dumps(line), flush=True)


# prefill workloads of the default run: the headline (Qwen3.5-0.8B-shaped layer) first, then the
# Qwen3-0.6B-shaped and the paper-MoE-shaped layers, each timed and reported on its own
PREFILLS = [PREFILL, "qwen3_06b_prefill", "paper_moe_prefill"]


def prefill_kernel(w):
    """(name, source files, committed ncu summary) of the attention kernel a bf16
    prefill workload runs on."""
    common = ["common.cuh", "internal.h"]
    if w.d == 256 and (w.H // w.G) % 2 == 0:
        return "prefill_pair_kernel<256, false>", ["prefill_pair.cu"] + common, "prefill_pair_qwen35_08b.md"
    summary = {"qwen3_06b_prefill": "prefill_tc_qwen3_06b.md", "paper_moe_prefill": "prefill_tc_paper_moe.md"}
    return f"prefill_tc_kernel<{w.d}, false>", ["prefill_tc.cu"] + common, summary.get(w.name, "")


def step_config(wp, wd, world, seqlens):
    """The workload description shared by both arms' JSON lines."""
    return {"workload": f"{wp.name} + {wd.name}",
            "prefill": {"B": wp.B, "S": wp.S, "H": wp.H, "G": wp.G, "d": wp.d, "rotary_dim": wp.rotary_dim,
                        "rope_base": wp.rope_base, "gate": wp.gate_mode},
            "decode": {"B": wd.B, "H": wd.H, "G": wd.G, "d": wd.d, "Lmax": wd.Lmax,
                       "seqlens": f"U[{wd.seqlen_range[0]},{wd.seqlen_range[1]}] seed {wd.seed}",
                       "sum_seqlens": sum(seqlens)},
            "l2": "flushed (256 MiB write) before every timed call", "parallelism": f"replicas x{world}"}


def cpu_decode_baseline(w, budget_s):
    """The fp64 oracle on a bounded sample of the decode workload: whole sequences of
    its shape and length distribution (a two-sequence cache is generated for it);
    GB/s of the algorithmic K/V + q/gate/out bytes of the sequences computed."""
    import oracle
    from gated_softmax_attention_gqa_gb300.workloads import decode_io_bytes, make_decode_inputs

    inp = make_decode_inputs(w, B=2)
    sl = inp["seqlens"].tolist()
    n, dt = 0, 0.0
    t0 = time.perf_counter()
    while dt < budget_s * 0.5 or n == 0:
        oracle.decode(inp["q_new"], inp["kv_cache"][0], inp["kv_cache"][1], inp["seqlens"], inp["gate"],
                      inp["qnorm_w"], w.rotary_dim, w.rope_base, w.eps, w.gate_mode)
        n += 1
        dt = time.perf_counter() - t0
    nbytes = n * decode_io_bytes(sl, w.H, w.G, w.d, w.gate_mode)
    return {"value": nbytes / dt / 1e9, "unit": "GB/s", "cores": oracle.threads_used(), "kind": "oracle",
            "sample": f"{n} x 2 sequences of {w.name} (lengths {sl}, H{w.H} G{w.G} d{w.d}); fp64 C loops, OpenMP; "
                      f"{dt:.1f} s", "seconds": dt}


def host_link_rates(dev, nbytes):
    """Plain pinned-memory copy rates between this process's host buffers and the GPU
    (one cudaMemcpyAsync of nbytes each way, median of 5), with the NUMA node the
    GPU reports and the CPUs this process may run on."""
    import torch

    h = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
    dbuf = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    out = {"bytes": nbytes}
    for name, fn in (("h2d_gbs", lambda: dbuf.copy_(h, non_blocking=True)),
                     ("d2h_gbs", lambda: h.copy_(dbuf, non_blocking=True))):
        ts = []
        for _ in range(6):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            fn()
            b.record()
            torch.cuda.synchronize()
            ts.append(a.elapsed_time(b))
        out[name] = nbytes / (statistics.median(ts[1:]) * 1e-3) / 1e9
    try:
        bus = torch.cuda.get_device_properties(dev).pci_bus_id if hasattr(
            torch.cuda.get_device_properties(dev), "pci_bus_id") else None
        out["cpus_allowed"] = len(os.sched_getaffinity(0))
        if bus:
            with open(f"/sys/bus/pci/devices/{bus.lower()}/numa_node") as f:
                out["gpu_numa_node"] = int(f.read().strip())
    except (OSError, ValueError, AttributeError):
        pass
    return out


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
        return
    if args.next_rows:
        run_next_rows(args)
        return

    import torch
    import torch.distributed as dist

    import gated_softmax_attention_gqa_gb300 as ga
    from gated_softmax_attention_gqa_gb300.workloads import (WORKLOADS, decode_io_bytes, make_decode_inputs,
                                                             make_prefill_inputs, prefill_flops)

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream(dev)
    hbm_peak, bf16_peak, peak_kind = peaks()

    profiling = bool(args.only or args.decode_batch)
    do_p, do_d = args.only in (None, "prefill"), args.only in (None, "decode")
    do_o = args.only in (None, "oproj") and not args.decode_batch
    # the headline prefill (a profiling run may pick another); the other two are
    # timed after the headline step in the default run
    head = args.prefill
    others = [n for n in PREFILLS if n != head] if not profiling else []
    wd = WORKLOADS[DECODE]
    if args.decode_batch:
        wd = dataclasses.replace(wd, B=args.decode_batch)

    P = {}  # per prefill workload: workload, host inputs, device inputs, out, workspace
    for name in ([head] if do_p else []) + others:
        w = WORKLOADS[name]
        pin = make_prefill_inputs(w)
        P[name] = {"w": w, "pin": pin, "dev": {k: v.to(dev) for k, v in pin.items()},
                   "out": torch.empty((w.B, w.S, w.H * w.d), dtype=torch.bfloat16, device=dev),
                   "ws": torch.empty(ga.gattn_prefill_workspace_size(w.B, w.S, w.H, w.G, w.d), dtype=torch.uint8,
                                     device=dev)}
    din = make_decode_inputs(wd) if do_d else None
    d_dev = {k: v.to(dev) for k, v in din.items()} if do_d else {}
    seqlens = din["seqlens"].tolist() if do_d else [1]
    d_out = torch.empty((wd.B, wd.H * wd.d), dtype=torch.bfloat16, device=dev)
    d_ws = torch.empty(ga.gattn_decode_workspace_size(wd.B, wd.H, wd.G, wd.d, wd.Lmax), dtype=torch.uint8,
                       device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)

    def prefill(name):
        e = P[name]
        w, x = e["w"], e["dev"]
        ga.gattn_prefill(x["q"], x["k"], x["v"], x["gate"], x["qnorm_w"], x["knorm_w"], rotary_dim=w.rotary_dim,
                         rope_base=w.rope_base, eps=w.eps, gate_mode=w.gate_mode, out=e["out"], workspace=e["ws"])

    def decode():
        if not do_d:
            return
        ga.gattn_decode(d_dev["q_new"], d_dev["kv_cache"], d_dev["seqlens"], d_dev["gate"], d_dev["qnorm_w"],
                        rotary_dim=wd.rotary_dim, rope_base=wd.rope_base, eps=wd.eps, gate_mode=wd.gate_mode,
                        out=d_out, workspace=d_ws)

    def ev():
        return torch.cuda.Event(enable_timing=True)

    for _ in range(max(3, args.warmup)):
        for name in P:
            flush.zero_()
            prefill(name)
        flush.zero_()
        decode()
    torch.cuda.synchronize()
    if ga.gattn_get_device_status() != 0:
        raise RuntimeError("device status set during warm-up")

    K = args.steps
    keys = ["d", "dk"] + [f"{n}:call" for n in P] + [f"{n}:kernel" for n in P]
    evs = {k: [(ev(), ev()) for _ in range(K)] for k in keys}
    for pairs in evs.values():  # create every event before the timed region
        for a, b in pairs:
            a.record(stream)
            b.record(stream)
    sampler = ClockSampler(dev.index)
    time.sleep(0.1)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    sampler.mark_start()
    # Timed region 1: the headline step exactly as a user makes its calls: the prefill,
    # then the decode step.
    for i in range(K):
        if do_p:
            flush.zero_()
            evs[f"{head}:call"][i][0].record(stream)
            prefill(head)
            evs[f"{head}:call"][i][1].record(stream)
        flush.zero_()
        evs["d"][i][0].record(stream)
        decode()
        evs["d"][i][1].record(stream)
    # Timed region 2: the same calls with the library recording events around its main
    # attention kernel (the roofline numbers).  Kept separate because an event between
    # the K pre-pass and the attention kernel stops them from overlapping.
    for i in range(K):
        if do_p:
            flush.zero_()
            ga.gattn_set_profile_events(*evs[f"{head}:kernel"][i])
            prefill(head)
        flush.zero_()
        ga.gattn_set_profile_events(*evs["dk"][i])
        decode()
    ga.gattn_set_profile_events(None, None)
    # Timed region 3: the other prefill workloads, whole calls then kernel alone.
    for name in others:
        for i in range(K):
            flush.zero_()
            evs[f"{name}:call"][i][0].record(stream)
            prefill(name)
            evs[f"{name}:call"][i][1].record(stream)
        for i in range(K):
            flush.zero_()
            ga.gattn_set_profile_events(*evs[f"{name}:kernel"][i])
            prefill(name)
        ga.gattn_set_profile_events(None, None)
    torch.cuda.synchronize()
    sampler.mark_end()
    if world > 1:
        dist.barrier()
    clocks = sampler.stop()

    def ms(key):
        return statistics.mean(a.elapsed_time(b) for a, b in evs[key])

    t = {k: ms(k) if (k[0] != "d" or do_d) else float("nan") for k in keys}
    t = dict(zip(keys, reduce_max([t[k] for k in keys], dev)))
    status = ga.gattn_get_device_status()

    dbytes = decode_io_bytes(seqlens, wd.H, wd.G, wd.d, wd.gate_mode)
    dec_gbs = world * dbytes / (t["d"] * 1e-3) / 1e9 if do_d else float("nan")
    dec_kern_gbs = dbytes / (t["dk"] * 1e-3) / 1e9 if do_d else float("nan")

    def prefill_entry(name):
        w = P[name]["w"]
        flops = prefill_flops(w.B, w.S, w.H, w.d)
        call, kern = t[f"{name}:call"], t[f"{name}:kernel"]
        kname, src, summary = prefill_kernel(w)
        kt = flops / (kern * 1e-3) / 1e12
        return {"workload": name, "shape": {"B": w.B, "S": w.S, "H": w.H, "G": w.G, "d": w.d,
                                            "rotary_dim": w.rotary_dim, "gate": w.gate_mode},
                "flops": flops, "ms": call, "kernel_ms": kern, "value": world * flops / (call * 1e-3) / 1e12,
                "unit": "TFLOP/s",
                "roofline": {"bound": "tensor", "achieved": kt, "peak": bf16_peak, "unit": "TFLOP/s",
                             "frac": kt / bf16_peak, "peak_kind": f"{peak_kind} bf16 dense (burst)", "kernel": kname,
                             "traffic": profiled_traffic(summary, src) if summary else None}}

    configs = {name: prefill_entry(name) for name in P}
    value = configs[head]["value"] if do_p else float("nan")

    # ---- Timed region 4: the output projection that follows the path (y = x W_O^T, the
    # library's tcgen05 GEMM), on the Qwen3.5-0.8B shape: x = the headline prefill's
    # output [B*S, H*d] = [4096, 2048], W_O [hidden 1024, 2048] (synthetic N(0, 1/K)).
    oproj = None
    if do_o:
        ow = WORKLOADS[OPROJ_PREFILL]
        T_o, K_o, N_o = ow.B * ow.S, ow.H * ow.d, OPROJ_HIDDEN
        x_o = (P[OPROJ_PREFILL]["out"] if OPROJ_PREFILL in P else
               torch.randn(T_o, K_o, generator=torch.Generator().manual_seed(7)).to(torch.bfloat16).to(dev))
        x_o = x_o.view(T_o, K_o)
        w_o = (torch.randn(N_o, K_o, generator=torch.Generator().manual_seed(8)) / K_o ** 0.5).to(torch.bfloat16)
        w_o = w_o.to(dev)
        y_o = torch.empty(T_o, N_o, dtype=torch.bfloat16, device=dev)
        for _ in range(max(3, args.warmup)):
            flush.zero_()
            ga.gattn_o_proj(x_o, w_o, out=y_o)
        pairs = [(ev(), ev()) for _ in range(K)]
        torch.cuda.synchronize()
        for i in range(K):
            flush.zero_()
            pairs[i][0].record(stream)
            ga.gattn_o_proj(x_o, w_o, out=y_o)
            pairs[i][1].record(stream)
        torch.cuda.synchronize()
        o_ms = reduce_max([statistics.median(a.elapsed_time(b) for a, b in pairs)], dev)[0]
        o_flops = 2 * T_o * K_o * N_o
        o_tf = o_flops / (o_ms * 1e-3) / 1e12
        oproj = {"workload": f"{OPROJ_PREFILL} o_proj", "shape": {"T": T_o, "K": K_o, "N": N_o}, "flops": o_flops,
                 "ms": o_ms, "value": world * o_tf, "unit": "TFLOP/s",
                 "roofline": {"bound": "tensor", "achieved": o_tf, "peak": bf16_peak, "unit": "TFLOP/s",
                              "frac": o_tf / bf16_peak, "peak_kind": f"{peak_kind} bf16 dense (burst)",
                              "kernel": "oproj_kernel<256>",
                              "traffic": profiled_traffic("oproj_qwen35_08b.md", ["oproj.cu", "common.cuh",
                                                                                 "internal.h"])}}

    # ---- end to end through the public API: pinned host -> device, prefill, device -> host.
    # Steps are pipelined the way a serving loop runs them: two device slots; step i's
    # inputs go in on a copy stream while step i-1 computes, and its result comes back
    # on another copy stream while step i+1 computes.  Every step's copies are inside
    # the timed region (it ends when the last result has reached the host).
    e2e_val, e2e_ms, h2d, d2h, link = float("nan"), float("nan"), 0, 0, {}
    if do_p:
        wp, pin, p_out, p_ws = P[head]["w"], P[head]["pin"], P[head]["out"], P[head]["ws"]
        host_in = {k: v.pin_memory() for k, v in pin.items()}
        host_out = torch.empty(p_out.shape, dtype=p_out.dtype).pin_memory()
        h2d = sum(v.numel() * v.element_size() for v in host_in.values())
        d2h = host_out.numel() * host_out.element_size()
        NSLOT = 2
        e2e_in = [{k: torch.empty_like(v, device=dev) for k, v in pin.items()} for _ in range(NSLOT)]
        e2e_out = [torch.empty_like(p_out) for _ in range(NSLOT)]
        s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        ev_in = [torch.cuda.Event() for _ in range(NSLOT)]    # the slot's inputs have landed
        ev_done = [torch.cuda.Event() for _ in range(NSLOT)]  # the slot's prefill is done (inputs free, result ready)
        ev_out = [torch.cuda.Event() for _ in range(NSLOT)]   # the slot's result has been copied out

        def e2e_step(i):
            sl = i % NSLOT
            s_in.wait_event(ev_done[sl])  # step i-2 no longer reads the slot's inputs
            with torch.cuda.stream(s_in):
                for k, v in host_in.items():
                    e2e_in[sl][k].copy_(v, non_blocking=True)
            ev_in[sl].record(s_in)
            stream.wait_event(ev_in[sl])
            stream.wait_event(ev_out[sl])  # step i-2's result has left the slot
            b = e2e_in[sl]
            ga.gattn_prefill(b["q"], b["k"], b["v"], b["gate"], b["qnorm_w"], b["knorm_w"],
                             rotary_dim=wp.rotary_dim, rope_base=wp.rope_base, eps=wp.eps, gate_mode=wp.gate_mode,
                             out=e2e_out[sl], workspace=p_ws, stream=stream)
            ev_done[sl].record(stream)
            s_out.wait_event(ev_done[sl])
            with torch.cuda.stream(s_out):
                host_out.copy_(e2e_out[sl], non_blocking=True)
            ev_out[sl].record(s_out)

        for i in range(3):
            e2e_step(i)
        torch.cuda.synchronize()
        e0, e1 = ev(), ev()
        e0.record(stream)
        s_in.wait_event(e0)
        s_out.wait_event(e0)
        for i in range(K):
            e2e_step(i)
        for sl in range(NSLOT):
            stream.wait_event(ev_out[sl])  # the last results are on the host
        e1.record(stream)
        torch.cuda.synchronize()
        e2e_ms = reduce_max([e0.elapsed_time(e1) / K], dev)[0]
        e2e_val = world * configs[head]["flops"] / (e2e_ms * 1e-3) / 1e12
        link = host_link_rates(dev, h2d)

    if rank == 0:
        dec_src = ["decode.cu", "common.cuh", "internal.h"]
        hc = configs.get(head, {})
        # launches of this library's kernels inside the timed regions: a prefill call is
        # the K pre-pass + the attention kernel, a decode call the split + combine kernels
        launches = {"headline_step": 2 * K * (2 * do_p + 2 * do_d), "other_prefills": 4 * K * len(others),
                    "o_proj": K * do_o, "e2e": 2 * K * do_p}
        wp = P[head]["w"] if do_p else WORKLOADS[head]
        line = {
            "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": K,
            "warmup": args.warmup, "ms_per_step": (hc.get("ms", 0.0) if do_p else 0.0) + (t["d"] if do_d else 0.0),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": step_config(wp, wd, world, seqlens),
            "prefill_ms": hc.get("ms"), "prefill_kernel_ms": hc.get("kernel_ms"),
            "roofline": hc.get("roofline"),
            "decode": {"value": dec_gbs, "unit": "GB/s", "ms": t["d"], "kernel_ms": t["dk"],
                       "bytes_per_step": dbytes,
                       "roofline": {"bound": "hbm", "achieved": dec_kern_gbs, "peak": hbm_peak, "unit": "GB/s",
                                    "frac": dec_kern_gbs / hbm_peak, "frac_of_8TBs": dec_kern_gbs / 8000.0,
                                    "peak_kind": f"{peak_kind} HBM copy", "kernel": "decode_split_kernel<256>",
                                    "traffic": profiled_traffic("decode_split_qwen35_08b.md", dec_src)}},
            "prefill_configs": configs,
            "o_proj": oproj,
            "e2e": {"value": e2e_val, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "ms_per_step": e2e_ms, "host_link": link},
            "gpu_launches": sum(launches.values()), "gpu_launches_by_region": launches,
            "clocks": clocks,
            "device_status": status,
        }
        if profiling:
            line = {"profiling_run": True, "only": args.only, "decode_batch": wd.B, "prefill": head,
                    "prefill_ms": hc.get("ms"), "prefill_kernel_ms": hc.get("kernel_ms"),
                    "decode_ms": t["d"], "decode_kernel_ms": t["dk"],
                    "prefill_kernel_tflops": hc.get("roofline", {}).get("achieved"),
                    "decode_kernel_gbs": dec_kern_gbs, "o_proj": oproj, "clocks": clocks}
        elif not args.no_cpu_baseline:
            for name in P:
                cb = cpu_baseline(P[name]["w"], P[name]["pin"], args.cpu_budget_s)
                cb.pop("seconds", None)
                configs[name]["cpu_baseline"] = cb
            line["cpu_baseline"] = configs[head]["cpu_baseline"]
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
